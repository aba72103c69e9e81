"""The allocation-free attention entry point against the workspace one.

Some callers cannot allocate device memory -- a plugin inside a framework that
owns all device memory and hands out no allocator, or a serving loop that
forbids cudaMalloc/cudaFree after start-up because they synchronise the device
-- so they cannot pass the workspace pkv_paged_decode_attention needs.
pkv_paged_decode_attention_static keeps that scratch in a static device array
instead. Here, through the C ABI, two calls in a row must match the workspace
entry point's output within the parity tests' tolerance, and a geometry whose
scratch is over the array's size must be refused.
"""
import ctypes

import pytest

torch = pytest.importorskip("torch")

import paged_kv_cache_101_gb300 as pkv  # noqa: E402
import workloads as W  # noqa: E402
from gpu_helpers import DeviceStep, compare, to_f64  # noqa: E402
from paged_kv_cache_101_gb300 import _build  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.lib()


def static_call(lib, d, out):
    w = d.w
    return lib.pkv_paged_decode_attention_static(
        d.q.data_ptr(), d.k_cache.data_ptr(), d.v_cache.data_ptr(), w.num_blocks,
        d.tables.data_ptr(), w.max_blocks_per_seq, d.lens.data_ptr(), w.num_seqs,
        w.n_query_per_seq, w.num_q_heads, w.num_kv_heads, w.head_dim, float(w.scale),
        out.data_ptr(), pkv.PKV_BF16, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("name", ["tiny", "llama3_8b_decode", "spec_verify"])
def test_static_scratch_matches_workspace_entry_point(lib, name):
    pkv.set_option(pkv.PKV_OPT_NUM_CTAS, 0)
    w = W.make_workload(name)
    d = DeviceStep(w, torch)
    d.append()
    ref = d.attend().clone()          # workspace entry point, torch-allocated workspace
    torch.cuda.synchronize()
    for call in range(2):             # the second call reuses the first call's scratch
        out = torch.full_like(d.out, float("nan"))
        st = static_call(lib, d, out)
        assert st == pkv.PKV_OK, pkv.status_string(st)
        torch.cuda.synchronize()
        compare(to_f64(out), to_f64(ref), what=f"{name}, static call {call + 1}")


def test_static_scratch_refuses_oversized_geometry(lib):
    # 32 query rows per kv head and 1000 CTAs: ~130 MiB of split-K scratch
    w = W.make_custom(4, 4, 64, 8, 128, [40, 50, 60, 70], seed=7)
    d = DeviceStep(w, torch)
    prev = pkv.set_option(pkv.PKV_OPT_NUM_CTAS, 1000)    # scratch grows with the grid
    try:
        out = torch.zeros_like(d.out)
        assert static_call(lib, d, out) == 6             # PKV_ERR_WORKSPACE
    finally:
        pkv.set_option(pkv.PKV_OPT_NUM_CTAS, prev)
