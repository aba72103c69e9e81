"""GPU parity of the CUDA-core consumers (PKV_OPT_MATH = 1), the reference point
against which the tensor-core consumers were chosen: same pipeline, same cells
and merge, the scores and P.V as fp32 FMA with shuffle reductions.

Against the fp64 oracle on the same seeded inputs, element by element within
2e-3 + 1e-2*|ref| (bf16 out) and max-abs 2e-3 (fp32 out): 1 to 32 query rows
per kv head (4- and 8-row warps, one to four warps per kv head), every length
mod 16, causal speculative queries, rows that see no token, split-K at several
grid sizes, and the full-size 8B-layer and speculative-verify workloads on
sampled (sequence, kv head) pairs. The option leaves the other entry points on
the tensor cores (checked bit for bit on an E4M3 pool).
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_101_gb300 as pkv
import workloads as W
from gpu_helpers import ATOL, DeviceStep, bf16_dev, compare, full_reference, report, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


@pytest.fixture(autouse=True)
def _fma():
    pkv.set_option(pkv.PKV_OPT_NUM_CTAS, 0)
    pkv.set_option(pkv.PKV_OPT_MATH, 1)
    yield
    pkv.set_option(pkv.PKV_OPT_MATH, 0)
    pkv.set_option(pkv.PKV_OPT_NUM_CTAS, 0)


def run(o, w, out_dtype=None):
    d = DeviceStep(w, torch, out_dtype=out_dtype)
    ref, _, _ = o.step(w)
    d.step()
    torch.cuda.synchronize()
    got = to_f64(d.out)
    stats = compare(got, ref, what=w.name)
    assert pkv.workspace_error(pkv.workspace(d.q.device, 0)) == 0
    return got, ref, stats


@pytest.mark.parametrize("G,nq", [(1, 1), (2, 1), (3, 1), (4, 1), (8, 1), (5, 1), (4, 2),
                                  (2, 4), (3, 3), (8, 2), (4, 4), (8, 4), (16, 2), (32, 1)])
def test_rows_per_kv_head(o, G, nq):
    Hkv = 2
    T = [nq, nq + 1, 15, 16, 17, 31, 32, 33, 100, 257, 1000]
    w = W.make_custom(len(T), nq, G * Hkv, Hkv, 128, T, seed=300 + 7 * G + nq)
    run(o, w)


def test_every_length_mod_16(o):
    T = list(range(1, 49)) + [63, 64, 65, 127, 128, 129, 511, 512, 513]
    w = W.make_custom(len(T), 1, 16, 4, 128, T, seed=301)
    run(o, w)


def test_fp32_output_strict(o):
    w = W.make_custom(6, 4, 64, 8, 128, [4, 33, 190, 600, 17, 1000], seed=302)
    _, _, (max_abs, max_rel) = run(o, w, out_dtype=torch.float32)
    assert max_abs <= ATOL


@pytest.mark.parametrize("ctas", [1, 7, 152, 400])
def test_split_grid_invariance(o, ctas):
    pkv.set_option(pkv.PKV_OPT_NUM_CTAS, ctas)
    T = [3000, 20, 4, 777, 4096, 129]
    w = W.make_custom(len(T), 4, 64, 8, 128, T, seed=303)
    run(o, w)


def test_rows_that_see_no_token(o):
    w = W.make_custom(3, 4, 16, 2, 128, [4, 9, 40], seed=304)
    d = DeviceStep(w, torch)
    d.append()
    lens = w.context_lens.copy()
    lens[0] = 2   # queries 0 and 1 of sequence 0 see nothing
    d.lens = torch.from_numpy(lens).cuda()
    d.attend()
    torch.cuda.synchronize()
    k, v = o.kv_append(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache)
    ref = o.paged_attention(w.q, k, v, w.block_tables, lens, 4, w.scale)
    got = to_f64(d.out)
    compare(got, ref, what="rows without tokens")
    assert np.all(got[0:2] == 0)


@pytest.mark.parametrize("name", ["llama3_8b_decode", "spec_verify"])
def test_full_size(o, name):
    w = W.make_workload(name)
    d = DeviceStep(w, torch)
    d.step()
    torch.cuda.synchronize()
    ref = full_reference(o, w, name)
    got = to_f64(d.out)
    max_abs, max_rel = compare(got, ref, what=f"{name}, CUDA-core consumers")
    report(f"{name}, CUDA-core consumers", max_abs, max_rel, got.size)
    assert pkv.workspace_error(pkv.workspace(d.q.device, 0)) == 0


def test_other_entry_points_stay_on_tensor_cores():
    w = W.make_custom(4, 1, 32, 8, 128, [100, 600, 17, 2000], seed=305)
    k8, v8, ks, vs = W.fp8_pools(w)
    kc, vc = torch.from_numpy(k8).cuda(), torch.from_numpy(v8).cuda()
    ksd, vsd = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    q = bf16_dev(w.q, torch)
    pkv.kv_append_fp8(bf16_dev(w.k_new, torch), bf16_dev(w.v_new, torch),
                      torch.from_numpy(w.slot_mapping).cuda(), kc, vc, ksd, vsd)
    tables = torch.from_numpy(w.block_tables).cuda()
    lens = torch.from_numpy(w.context_lens).cuda()
    outs = []
    for math in (1, 0):
        pkv.set_option(pkv.PKV_OPT_MATH, math)
        out = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
        pkv.paged_decode_attention_fp8(q, kc, vc, ksd, vsd, tables, lens, 1, w.scale, out)
        torch.cuda.synchronize()
        outs.append(out.view(torch.int16))
    assert torch.equal(outs[0], outs[1])
