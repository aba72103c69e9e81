"""The allocation-free attention entry point against the oracle and the workspace one.

Some callers cannot allocate device memory -- a plugin inside a framework that
owns all device memory and hands out no allocator, or a serving loop that
forbids cudaMalloc/cudaFree after start-up because they synchronise the device
-- so they cannot pass the workspace pkv_paged_decode_attention needs.
pkv_paged_decode_attention_static keeps that scratch in a static device array
instead. Here, through the C ABI:

* two calls in a row match the fp64 oracle within the parity tests' tolerance,
  and match the workspace entry point's output;
* invalid arguments return the same status as the workspace entry point;
* a geometry whose scratch is over the array's size is refused;
* device-side errors reach the caller through pkv_static_error_word.

This file is collected last on purpose: a failure here leaves every other test
already run.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import paged_kv_cache_101_gb300 as pkv  # noqa: E402
import workloads as W  # noqa: E402
from gpu_helpers import DeviceStep, compare, to_f64  # noqa: E402
from paged_kv_cache_101_gb300 import _build  # noqa: E402

pytestmark = pytest.mark.gpu

OK, NULL, SHAPE, DTYPE, ALIGN, RANGE, WORKSPACE, CUDA, UNSUP = range(9)
OPTIONS = (pkv.PKV_OPT_NUM_CTAS, pkv.PKV_OPT_STAGES, pkv.PKV_OPT_HEADS_PER_CTA,
           pkv.PKV_OPT_TMA_BOX, pkv.PKV_OPT_TAIL, pkv.PKV_OPT_PACE, pkv.PKV_OPT_MATH,
           pkv.PKV_OPT_UMMA, pkv.PKV_OPT_PREFETCH)


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.lib()


@pytest.fixture(autouse=True)
def default_options(lib):
    for opt in OPTIONS:
        pkv.set_option(opt, 0)
    yield
    for opt in OPTIONS:
        pkv.set_option(opt, 0)


def _stream(s=None):
    s = s if s is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def call_args(d, out, **over):
    """The argument list shared by the two entry points (workspace left out)."""
    w = d.w
    a = dict(q=d.q.data_ptr(), k=d.k_cache.data_ptr(), v=d.v_cache.data_ptr(), nb=w.num_blocks,
             tables=d.tables.data_ptr(), mb=w.max_blocks_per_seq, lens=d.lens.data_ptr(),
             S=w.num_seqs, nq=w.n_query_per_seq, Hq=w.num_q_heads, Hkv=w.num_kv_heads,
             D=w.head_dim, scale=float(w.scale), out_ptr=out.data_ptr(),
             dtype=pkv.PKV_FP32 if out.dtype == torch.float32 else pkv.PKV_BF16)
    a.update(over)
    return [a[k] for k in ("q", "k", "v", "nb", "tables", "mb", "lens", "S", "nq", "Hq", "Hkv",
                           "D", "scale", "out_ptr", "dtype")]


def static_call(lib, d, out, stream=None, **over):
    return lib.pkv_paged_decode_attention_static(*call_args(d, out, **over), _stream(stream))


def workspace_call(lib, d, out, ws, **over):
    return lib.pkv_paged_decode_attention(*call_args(d, out, **over), ws.data_ptr(), ws.numel(),
                                          _stream())


@pytest.mark.parametrize("name", ["tiny", "llama3_8b_decode", "spec_verify"])
def test_static_scratch_matches_oracle_and_workspace_entry_point(lib, name):
    w = W.make_workload(name)
    d = DeviceStep(w, torch)
    d.append()
    ref_ws = d.attend().clone()       # workspace entry point, torch-allocated workspace
    torch.cuda.synchronize()
    ref, _, _ = oracle.Oracle().step(w)
    for call in range(2):             # the second call reuses the first call's scratch
        out = torch.full_like(d.out, float("nan"))
        st = static_call(lib, d, out)
        assert st == OK, pkv.status_string(st)
        torch.cuda.synchronize()
        got = to_f64(out)
        max_abs, max_rel = compare(got, ref, what=f"{name}, static call {call + 1} vs oracle")
        compare(got, to_f64(ref_ws), what=f"{name}, static call {call + 1} vs workspace call")
        print(f"{name} static call {call + 1}: max_abs={max_abs:.2e} max_rel={max_rel:.2e}")
    assert pkv.static_error_word() == 0


def test_static_scratch_fp32_output_on_a_second_stream(lib):
    """fp32 output (strict 2e-3 absolute bound), first on the current stream, then
    on another stream once the first call has finished."""
    w = W.make_custom(6, 2, 16, 2, 128, [900, 33, 4000, 2, 260, 17], seed=71)
    d = DeviceStep(w, torch, out_dtype=torch.float32)
    d.append()
    torch.cuda.synchronize()
    ref, _, _ = oracle.Oracle().step(w)
    out = torch.full_like(d.out, float("nan"))
    assert static_call(lib, d, out) == OK
    torch.cuda.synchronize()
    compare(to_f64(out), ref, atol=2e-3, rtol=0.0, what="static fp32, current stream")
    side = torch.cuda.Stream()
    out2 = torch.full_like(d.out, float("nan"))
    with torch.cuda.stream(side):
        assert static_call(lib, d, out2, stream=side) == OK
    side.synchronize()
    compare(to_f64(out2), ref, atol=2e-3, rtol=0.0, what="static fp32, second stream")


def test_static_scratch_refuses_oversized_geometry(lib):
    # 64 query rows per kv head and 1000 CTAs: over 60 MiB of split-K scratch
    w = W.make_custom(4, 4, 128, 8, 128, [40, 50, 60, 70], seed=7)
    d = DeviceStep(w, torch)
    pkv.set_option(pkv.PKV_OPT_NUM_CTAS, 1000)    # scratch grows with the grid
    out = torch.zeros_like(d.out)
    assert static_call(lib, d, out) == WORKSPACE


# invalid arguments: (what, overrides) -- the status must equal the workspace call's
INVALID = [
    ("five queries per sequence", dict(nq=5)),
    ("no query", dict(nq=0)),
    ("head_dim 96", dict(D=96)),
    ("q heads not a multiple of kv heads", dict(Hq=15)),
    ("unknown output dtype", dict(dtype=7)),
    ("no pool blocks", dict(nb=0)),
    ("no table columns", dict(mb=0)),
    ("q not 16-byte aligned", "q+2"),
    ("null output", dict(out_ptr=0)),
    ("null tables", dict(tables=0)),
    ("negative sequence count", dict(S=-1)),
]


@pytest.mark.parametrize("what,over", INVALID, ids=[x[0] for x in INVALID])
def test_static_status_matches_workspace_call(lib, what, over):
    w = W.make_custom(3, 1, 16, 4, 128, [40, 77, 2], seed=72)
    d = DeviceStep(w, torch)
    if over == "q+2":
        over = dict(q=d.q.data_ptr() + 2)
    ws = torch.zeros(max(pkv.workspace_size(3, 1, 16, 4, 128), 1 << 20), dtype=torch.uint8,
                     device="cuda")
    out = torch.zeros_like(d.out)
    expect = workspace_call(lib, d, out, ws, **over)
    assert expect != OK, what
    assert static_call(lib, d, out, **over) == expect, what
    torch.cuda.synchronize()


def test_static_error_word_reports_out_of_pool_block(lib):
    """A table entry past the pool reads zeros and sets bit 8 of the static error
    word; the next valid call clears it."""
    w = W.make_custom(2, 1, 8, 2, 64, [40, 20], seed=89)
    d = DeviceStep(w, torch)
    d.append()
    good_tables = d.tables
    tables = w.block_tables.copy()
    tables[0, 1] = w.num_blocks + 3
    d.tables = torch.from_numpy(tables).cuda()
    out = torch.zeros_like(d.out)
    assert static_call(lib, d, out) == OK
    assert pkv.static_error_word() == 8
    assert np.isfinite(to_f64(out)).all()
    d.tables = good_tables
    assert static_call(lib, d, out) == OK
    assert pkv.static_error_word() == 0
