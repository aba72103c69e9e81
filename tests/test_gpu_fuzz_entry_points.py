"""Seeded random cases for the other attention entry points, against the oracle.

- E4M3 pools: random geometry (head_dim 128), lengths, grid size and pipeline
  depth; the pool bit for bit, the output within 2e-3 + 1e-2*|ref|.
- Variable query counts: random counts 0..max per sequence, with or without
  random tree masks (each node sees itself and one random ancestor chain).
- Cascade: a random number of sharers moved to the front as one group, random
  prefix length, random grid size.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_101_gb300 as pkv
import workloads as W
from gpu_helpers import DeviceStep, bf16_dev, compare, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


@pytest.fixture(autouse=True)
def _defaults():
    for opt in (pkv.PKV_OPT_NUM_CTAS, pkv.PKV_OPT_STAGES):
        pkv.set_option(opt, 0)
    yield
    for opt in (pkv.PKV_OPT_NUM_CTAS, pkv.PKV_OPT_STAGES):
        pkv.set_option(opt, 0)


def geometry(rng, max_rows=32):
    Hkv = int(rng.choice([1, 2, 4, 8]))
    while True:
        G = int(rng.choice([1, 2, 4, 8]))
        nq = int(rng.integers(1, 5))
        if G * nq <= max_rows:
            return Hkv, G, nq


@pytest.mark.parametrize("seed", range(12))
def test_fp8_random(o, seed):
    rng = np.random.default_rng(7000 + seed)
    Hkv, G, nq = geometry(rng)
    S = int(rng.integers(1, 10))
    T = rng.integers(nq, 2500, S).astype(np.int64)
    pkv.set_option(pkv.PKV_OPT_NUM_CTAS, int(rng.choice([0, 3, 152, 400])))
    pkv.set_option(pkv.PKV_OPT_STAGES, int(rng.choice([0, 2, 4])))
    w = W.make_custom(S, nq, G * Hkv, Hkv, 128, T, seed=7100 + seed)
    k8, v8, ks, vs = W.fp8_pools(w, seed=seed)
    kc, vc = torch.from_numpy(k8).cuda(), torch.from_numpy(v8).cuda()
    ksd, vsd = torch.from_numpy(ks).cuda(), torch.from_numpy(vs).cuda()
    q = bf16_dev(w.q, torch)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    pkv.kv_append_fp8(bf16_dev(w.k_new, torch), bf16_dev(w.v_new, torch),
                      torch.from_numpy(w.slot_mapping).cuda(), kc, vc, ksd, vsd)
    pkv.paged_decode_attention_fp8(q, kc, vc, ksd, vsd, torch.from_numpy(w.block_tables).cuda(),
                                   torch.from_numpy(w.context_lens).cuda(), nq, w.scale, out)
    torch.cuda.synchronize()
    k_ref, v_ref = o.kv_append_fp8(w.k_new, w.v_new, w.slot_mapping, k8, v8, ks, vs)
    assert np.array_equal(kc.cpu().numpy(), k_ref) and np.array_equal(vc.cpu().numpy(), v_ref)
    ref = o.paged_attention_fp8(w.q, k_ref, v_ref, w.block_tables, w.context_lens, nq, w.scale,
                                ks, vs)
    compare(to_f64(out), ref, what=f"fp8 case {seed}")
    assert pkv.workspace_error(pkv.workspace(q.device, 0)) == 0


def random_tree(rng, n):
    if n == 0:
        return []
    masks = [1]
    for i in range(1, n):
        masks.append(masks[int(rng.integers(0, i))] | (1 << i))
    return masks


def i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


@pytest.mark.parametrize("seed", range(12))
def test_varlen_random(o, seed):
    rng = np.random.default_rng(8000 + seed)
    Hkv, G, _ = geometry(rng)
    max_q = min(4, 32 // G)
    S = int(rng.integers(1, 10))
    use_tree = bool(rng.random() < 0.5)
    qlen = rng.integers(0, max_q + 1, S)
    ctx = rng.integers(0, 1500, S)
    T = np.maximum(ctx + qlen, 1).astype(np.int32)
    D = int(rng.choice([64, 128]))
    pkv.set_option(pkv.PKV_OPT_NUM_CTAS, int(rng.choice([0, 7, 152])))
    w = W.make_custom(S, 1, G * Hkv, Hkv, D, T, seed=8100 + seed, keep_full=True)
    qs = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    q = W.f32_to_bf16_bits(rng.standard_normal((max(int(qs[-1]), 1), G * Hkv, D))
                           .astype(np.float32))[: int(qs[-1])]
    kw = {}
    masks = tl = None
    if use_tree:
        masks = np.concatenate([random_tree(rng, int(n)) for n in qlen] or [[]]).astype(np.uint32)
        tl = qlen.astype(np.int32)
        kw = dict(tree_mask=i32(masks.view(np.int32)), tree_len=i32(tl))
    ref = o.paged_attention_varlen(q, w.k_full, w.v_full, w.block_tables, T, qs, w.scale,
                                   tree_mask=masks, tree_len=tl)
    kd, vd = bf16_dev(w.k_full, torch), bf16_dev(w.v_full, torch)
    out = torch.full((int(qs[-1]), G * Hkv, D), float("nan"), dtype=torch.float32, device="cuda")
    if qs[-1] > 0:
        pkv.paged_decode_attention_varlen(bf16_dev(q, torch), kd, vd, i32(w.block_tables), i32(T),
                                          i32(qs), max_q, w.scale, out, **kw)
        torch.cuda.synchronize()
        compare(to_f64(out), ref, what=f"varlen case {seed}")
    assert pkv.workspace_error(pkv.workspace(kd.device, 0)) == 0


@pytest.mark.parametrize("seed", range(10))
def test_cascade_random(o, seed):
    rng = np.random.default_rng(9000 + seed)
    Hkv, G, nq = geometry(rng)
    S = int(rng.integers(3, 20))
    M = int(rng.integers(2, S + 1))
    prefix = int(rng.choice([16, 64, 256, 512]))
    T = np.concatenate([prefix + rng.integers(nq, 700, M), rng.integers(nq, 900, S - M)])
    pkv.set_option(pkv.PKV_OPT_NUM_CTAS, int(rng.choice([0, 5, 152])))
    w = W.make_custom(S, nq, G * Hkv, Hkv, 128, T.astype(np.int64), seed=9100 + seed,
                      shared=np.arange(S) < M, prefix_tokens=prefix)
    d = DeviceStep(w, torch)
    d.append()
    ws = pkv.workspace("cuda", int(pkv.lib().pkv_workspace_size_cascade(S, nq, G * Hkv, Hkv, 128)))
    groups = torch.from_numpy(np.array([[0, M, prefix // 16]], np.int32)).cuda()
    pkv.paged_decode_attention_cascade(d.q, d.k_cache, d.v_cache, d.tables, d.lens, nq, w.scale,
                                       d.out, groups, M, ws=ws)
    torch.cuda.synchronize()
    ref, _, _ = o.step(w)
    compare(to_f64(d.out), ref, what=f"cascade case {seed}")
    assert pkv.workspace_error(ws) == 0
