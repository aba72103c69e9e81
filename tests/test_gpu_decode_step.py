"""GPU checks of pkv_decode_step (append + attention in one call).

- bf16 and E4M3 pools: the pool and the output are bit-identical to
  pkv_kv_append / pkv_kv_append_fp8 followed by the attention call, and the output
  is within 2e-3 + 1e-2*|ref| of the fp64 oracle; decode (1 query, 8-row
  consumers), speculative verification (4 queries, 32 rows per kv head) and
  head_dim 64; several steps in a row on one stream.
- Errors: one scale alone, a misaligned or too small workspace and an unsupported
  geometry return their status with nothing enqueued (the pool is unchanged).
"""
import ctypes

import numpy as np
import pytest

import oracle
import paged_kv_cache_101_gb300 as pkv
import workloads as W
from gpu_helpers import DeviceStep, bf16_dev, bf16_host, compare, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


CASES = [  # (S, nq, Hq, Hkv, D, lengths)
    (5, 1, 32, 8, 128, [40, 777, 16, 2048, 130]),
    (4, 4, 64, 8, 128, [300, 1025, 64, 2000]),
    (3, 2, 16, 4, 64, [17, 500, 129]),
]


@pytest.mark.parametrize("S,nq,Hq,Hkv,D,T", CASES)
def test_bf16_step_matches_two_calls_and_oracle(o, S, nq, Hq, Hkv, D, T):
    w = W.make_custom(S, nq, Hq, Hkv, D, T, seed=900 + nq + D)
    a, b = DeviceStep(w, torch), DeviceStep(w, torch)
    a.step()                                               # the two calls
    pkv.decode_step(b.q, b.k_new, b.v_new, b.slots, b.k_cache, b.v_cache, b.tables, b.lens,
                    nq, w.scale, b.out)                    # one call
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host(a.k_cache), bf16_host(b.k_cache))
    assert np.array_equal(bf16_host(a.v_cache), bf16_host(b.v_cache))
    assert np.array_equal(bf16_host(a.out), bf16_host(b.out))
    ref, k_ref, v_ref = o.step(w)
    assert np.array_equal(bf16_host(b.k_cache), k_ref)
    compare(to_f64(b.out), ref, what="decode_step")


def test_steps_in_a_row(o):
    """Several one-call steps on one stream, each appending its rows: the pool and
    the outputs match the same sequence of two-call steps."""
    w = W.make_custom(4, 1, 32, 8, 128, [100, 2000, 33, 700], seed=910)
    a, b = DeviceStep(w, torch), DeviceStep(w, torch)
    rng = np.random.default_rng(910)
    for _ in range(4):
        kn = W.f32_to_bf16_bits(rng.standard_normal(w.k_new.shape).astype(np.float32))
        vn = W.f32_to_bf16_bits(rng.standard_normal(w.v_new.shape).astype(np.float32))
        for d in (a, b):
            d.k_new.copy_(bf16_dev(kn, torch))
            d.v_new.copy_(bf16_dev(vn, torch))
        a.step()
        pkv.decode_step(b.q, b.k_new, b.v_new, b.slots, b.k_cache, b.v_cache, b.tables,
                        b.lens, 1, w.scale, b.out)
        torch.cuda.synchronize()
        assert np.array_equal(bf16_host(a.k_cache), bf16_host(b.k_cache))
        assert np.array_equal(bf16_host(a.out), bf16_host(b.out))


@pytest.mark.parametrize("nq,G", [(1, 4), (4, 8)])
def test_fp8_step_matches_two_calls_and_oracle(o, nq, G):
    w = W.make_custom(4, nq, 8 * G, 8, 128, [60, 1500, 17, 800], seed=920 + nq)
    k8, v8, ks, vs = W.fp8_pools(w, seed=7)

    def u8(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()

    ksd = torch.from_numpy(ks).cuda()
    vsd = torch.from_numpy(vs).cuda()
    q, kn, vn = bf16_dev(w.q, torch), bf16_dev(w.k_new, torch), bf16_dev(w.v_new, torch)
    slots = torch.from_numpy(w.slot_mapping).cuda()
    tables = torch.from_numpy(w.block_tables).cuda()
    lens = torch.from_numpy(w.context_lens).cuda()
    ka, va, kb, vb = u8(k8), u8(v8), u8(k8), u8(v8)
    oa = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ob = torch.empty_like(oa)
    pkv.kv_append_fp8(kn, vn, slots, ka, va, ksd, vsd)
    pkv.paged_decode_attention_fp8(q, ka, va, ksd, vsd, tables, lens, nq, w.scale, oa)
    pkv.decode_step(q, kn, vn, slots, kb, vb, tables, lens, nq, w.scale, ob,
                    k_scale=ksd, v_scale=vsd)
    torch.cuda.synchronize()
    assert torch.equal(ka, kb) and torch.equal(va, vb)
    assert torch.equal(oa, ob)
    kr, vr = o.kv_append_fp8(w.k_new, w.v_new, w.slot_mapping, k8, v8, ks, vs)
    assert np.array_equal(kb.cpu().numpy(), kr)
    ref = o.paged_attention_fp8(w.q, kr, vr, w.block_tables, w.context_lens, nq, w.scale, ks, vs)
    compare(ob.cpu().numpy().astype(np.float64), ref, what="decode_step E4M3")


def _raw_call(d, w, nq, ws_ptr, ws_bytes, k_scale=None, v_scale=None, hq=None):
    S = w.num_seqs
    Hq = hq if hq is not None else w.num_q_heads
    return pkv.lib().pkv_decode_step(
        d.q.data_ptr(), d.k_new.data_ptr(), d.v_new.data_ptr(), d.slots.data_ptr(),
        d.k_cache.data_ptr(), d.v_cache.data_ptr(), w.num_blocks, d.tables.data_ptr(),
        d.tables.shape[1], d.lens.data_ptr(), S, nq, Hq, w.num_kv_heads, w.head_dim,
        float(w.scale), d.out.data_ptr(), pkv.PKV_BF16, ws_ptr, ws_bytes, k_scale, v_scale,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_errors_enqueue_nothing():
    w = W.make_custom(3, 1, 16, 4, 128, [40, 300, 17], seed=930)
    d = DeviceStep(w, torch)
    k0 = bf16_host(d.k_cache).copy()
    need = pkv.workspace_size(3, 1, 16, 4, 128)
    ws = torch.zeros(need + 512, dtype=torch.uint8, device="cuda")
    scale = torch.ones(4, dtype=torch.float32, device="cuda")
    cases = [
        (dict(ws_ptr=ws.data_ptr(), ws_bytes=need, k_scale=scale.data_ptr()), pkv.PKV_ERR_NULL),
        (dict(ws_ptr=ws.data_ptr() + 16, ws_bytes=need), pkv.PKV_ERR_ALIGN),
        (dict(ws_ptr=ws.data_ptr(), ws_bytes=need - 256), pkv.PKV_ERR_WORKSPACE),
        (dict(ws_ptr=None, ws_bytes=0), pkv.PKV_ERR_WORKSPACE),
        (dict(ws_ptr=ws.data_ptr(), ws_bytes=need, hq=15), None),   # Hq % Hkv != 0
    ]
    for kw, want in cases:
        st = _raw_call(d, w, 1, **kw)
        torch.cuda.synchronize()
        assert st != pkv.PKV_OK, kw
        if want is not None:
            assert st == want, (kw, st)
        assert np.array_equal(bf16_host(d.k_cache), k0), f"pool written by a refused call {kw}"
    assert _raw_call(d, w, 1, ws.data_ptr(), need) == pkv.PKV_OK
    torch.cuda.synchronize()
    assert not np.array_equal(bf16_host(d.k_cache), k0)      # the append ran
