"""GPU parity of variable query counts, tree masks and chunked prefill through
pkv_paged_decode_attention_varlen, against the oracle's unsplit definition.

- causal query counts 0..4 per sequence (every length mod 16), for 1, 4 and 8
  query heads per kv head, and up to 16 (4 heads) or 8 (8 heads) queries: 64 score
  rows per kv head; bf16 and fp32 outputs;
- tree masks: the 15-node binary tree of "Chapter 18" section 18.1.2 with 8
  query heads per kv head (120 score rows, split into runs of 4 queries that
  share the sequence's table row), and random trees;
- chunked prefill: a 200-token prompt appended and attended in chunks of 64,
  100 and 36 (each chunk split into runs) equals the one-pass prefill;
- a sequence whose query rows break the rules gets no output and sets the
  error bit, and the others stay exact.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_101_gb300 as pkv
import workloads as W
from gpu_helpers import bf16_dev, compare, to_f64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


@pytest.fixture(autouse=True)
def _defaults():
    pkv.set_option(pkv.PKV_OPT_NUM_CTAS, 0)
    yield
    pkv.set_option(pkv.PKV_OPT_NUM_CTAS, 0)


def i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def masks_i32(m):
    return torch.from_numpy(np.ascontiguousarray(m, dtype=np.uint32).view(np.int32)).cuda()


def run_varlen(w_full_k, w_full_v, tables, cl, qs, q, scale, max_q, tree_mask=None,
               tree_len=None, table_row=None, out_dtype=None):
    kd, vd = bf16_dev(w_full_k, torch), bf16_dev(w_full_v, torch)
    qd = bf16_dev(q, torch)
    out = torch.full(qd.shape, float("nan"), dtype=out_dtype or torch.bfloat16, device="cuda")
    pkv.paged_decode_attention_varlen(
        qd, kd, vd, i32(tables), i32(cl), i32(qs), max_q, scale, out,
        tree_mask=masks_i32(tree_mask) if tree_mask is not None else None,
        tree_len=i32(tree_len) if tree_len is not None else None,
        table_row=i32(table_row) if table_row is not None else None)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("hq,hkv,mq", [(8, 8, 4), (16, 4, 4), (32, 4, 4), (16, 4, 16),
                                       (16, 2, 8)])
@pytest.mark.parametrize("out32", [False, True])
def test_varlen_causal(o, hq, hkv, mq, out32):
    rng = np.random.default_rng(hq + out32 + mq)
    G = hq // hkv
    max_q = min(mq, 64 // G)
    S = 48
    qlen = rng.integers(0, max_q + 1, size=S)
    T = np.array([int(n) + i for i, n in enumerate(qlen)], np.int32)    # every length mod 16
    T = np.maximum(T, 1)
    w = W.make_custom(S, 1, hq, hkv, 128, T, seed=50 + hq, keep_full=True)
    qs = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    q = W.f32_to_bf16_bits(rng.standard_normal((int(qs[-1]), hq, 128)).astype(np.float32))
    ref = o.paged_attention_varlen(q, w.k_full, w.v_full, w.block_tables, T, qs, w.scale)
    out = run_varlen(w.k_full, w.v_full, w.block_tables, T, qs, q, w.scale, max_q,
                     out_dtype=torch.float32 if out32 else None)
    got = to_f64(out)
    compare(got, ref, what=f"varlen G={G}")
    if out32:
        assert np.abs(got - ref).max() <= 2e-3
    assert pkv.workspace_error(pkv.workspace(out.device, 0)) == 0


def binary_tree(levels):
    masks = []
    for node in range(2 ** levels - 1):
        m, a = 0, node
        while True:
            m |= 1 << a
            if a == 0:
                break
            a = (a - 1) // 2
        masks.append(m)
    return masks


def random_tree(rng, n):
    masks = [1]
    for i in range(1, n):
        masks.append(masks[int(rng.integers(0, i))] | (1 << i))
    return masks


@pytest.mark.parametrize("kind,hq,run", [("binary15", 64, 4), ("random", 64, 4),
                                         ("binary15", 32, 16), ("random", 32, 16)])
def test_tree_masks_split_into_runs(o, kind, hq, run):
    """8 query heads per kv head in runs of 4 queries (32 rows), and 4 heads in runs
    of 16 (64 rows: a 15-node tree in one run)."""
    rng = np.random.default_rng(7 if kind == "random" else 8)
    hkv = 8
    if kind == "binary15":
        trees = [binary_tree(4)] * 6
    else:
        trees = [random_tree(rng, int(n)) for n in rng.integers(1, 33, size=10)]
    nodes = [len(t) for t in trees]
    ctx = rng.integers(0, 700, size=len(trees))
    T = (ctx + nodes).astype(np.int32)
    w = W.make_custom(len(trees), 1, hq, hkv, 128, T, seed=60, keep_full=True)
    qs = np.concatenate([[0], np.cumsum(nodes)]).astype(np.int32)
    q = W.f32_to_bf16_bits(rng.standard_normal((int(qs[-1]), hq, 128)).astype(np.float32))
    masks = np.concatenate(trees).astype(np.uint32)
    tl = np.array(nodes, np.int32)
    ref = o.paged_attention_varlen(q, w.k_full, w.v_full, w.block_tables, T, qs, w.scale,
                                   tree_mask=masks, tree_len=tl)
    r = pkv.split_queries(qs, T, run, tree_len=tl)
    out = run_varlen(w.k_full, w.v_full, w.block_tables, r["context_lens"], r["q_start"], q,
                     w.scale, run, tree_mask=masks, tree_len=r["tree_len"],
                     table_row=r["table_row"])
    compare(to_f64(out), ref, what=f"{kind}, runs of {run}")
    assert pkv.workspace_error(pkv.workspace(out.device, 0)) == 0


def test_chunked_prefill_equals_single_prefill(o):
    rng = np.random.default_rng(9)
    hq, hkv, D, T = 32, 8, 128, 200
    w = W.make_custom(1, 1, hq, hkv, D, [T], seed=70, keep_full=True, keep_dense=True)
    q = W.f32_to_bf16_bits(rng.standard_normal((T, hq, D)).astype(np.float32))
    single = o.paged_attention_varlen(q, w.k_full, w.v_full, w.block_tables, [T],
                                      np.array([0, T], np.int32), w.scale)
    # the pool starts empty (NaN everywhere) and each chunk appends its tokens
    k_pool = bf16_dev(np.full_like(w.k_full, W.SENTINEL_BF16), torch)
    v_pool = bf16_dev(np.full_like(w.v_full, W.SENTINEL_BF16), torch)
    dense_k, dense_v = w.dense_k[0], w.dense_v[0]
    tbl = w.block_tables[0]
    got = np.zeros_like(single)
    start = 0
    for n in (64, 100, 36):
        end = start + n
        pos = np.arange(start, end)
        slots = (tbl[pos // 16].astype(np.int64) * 16 + pos % 16)
        pkv.kv_append(bf16_dev(dense_k[start:end], torch), bf16_dev(dense_v[start:end], torch),
                      torch.from_numpy(slots).cuda(), k_pool, v_pool)
        r = pkv.split_queries([0, n], [end], 4)
        qd = bf16_dev(q[start:end], torch)
        out = torch.empty(qd.shape, dtype=torch.float32, device="cuda")
        pkv.paged_decode_attention_varlen(qd, k_pool, v_pool, i32(w.block_tables),
                                          i32(r["context_lens"]), i32(r["q_start"]), 4, w.scale,
                                          out, table_row=i32(r["table_row"]))
        torch.cuda.synchronize()
        got[start:end] = to_f64(out)
        start = end
    compare(got, single, what="chunked prefill")
    assert np.abs(got - single).max() <= 2e-3


def test_invalid_rows_flagged_others_exact(o):
    rng = np.random.default_rng(11)
    T = np.array([30, 50, 70], np.int32)
    w = W.make_custom(3, 1, 16, 4, 128, T, seed=80, keep_full=True)
    qs = np.array([0, 2, 9, 12], np.int32)            # sequence 1 claims 7 rows (> 4)
    q = W.f32_to_bf16_bits(rng.standard_normal((12, 16, 128)).astype(np.float32))
    ws = pkv.workspace("cuda", pkv.workspace_size(3, 4, 16, 4, 128))
    ws.zero_()
    kd, vd = bf16_dev(w.k_full, torch), bf16_dev(w.v_full, torch)
    out = torch.zeros((12, 16, 128), dtype=torch.float32, device="cuda")
    pkv.paged_decode_attention_varlen(bf16_dev(q, torch), kd, vd, i32(w.block_tables), i32(T),
                                      i32(qs), 4, w.scale, out, ws=ws)
    torch.cuda.synchronize()
    assert pkv.workspace_error(ws) & 16
    got = to_f64(out)
    assert np.all(got[2:9] == 0)                       # untouched
    for s in (0, 2):
        one = o.paged_attention_varlen(q, w.k_full, w.v_full, w.block_tables[s:s + 1], T[s:s + 1],
                                       np.array([qs[s], qs[s + 1]], np.int32), w.scale)
        compare(got[qs[s]:qs[s + 1]], one[qs[s]:qs[s + 1]], what=f"seq {s}")
    ws.zero_()
