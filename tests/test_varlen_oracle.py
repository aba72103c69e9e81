"""Pins of the oracle's variable-query-count attention (causal and tree masks)
against what the pages and the definitions fix, and planted mistakes in copies
of the oracle, each caught.

- with equal query counts and no masks it is the pinned fixed-nq oracle, bit
  for bit; with varying counts, each sequence equals the fixed-nq oracle run on
  that sequence alone;
- a lower-triangular tree mask is the causal mask;
- a Medusa-style tree ("Chapter 18" section 18.1.2: 15 nodes, branching 2,
  4 levels, each node seeing its ancestors) matches library attention (torch
  SDPA in float64 with a boolean mask) on the generator's dense K/V;
- chunked prefill equals single prefill ("07 -- Inference" section 2.4): a
  prompt attended in chunks 20 + 30 + 14 gives the one-pass result bit for bit,
  and both match causal library attention;
- a node that sees only itself, with no earlier context, returns its own V.
"""
import numpy as np
import pytest

import oracle
import workloads as W

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


def binary_tree_masks(levels: int):
    """Ancestor-or-self bitmasks of a complete binary tree, nodes in level order."""
    n = 2 ** levels - 1
    masks = []
    for node in range(n):
        m, a = 0, node
        while True:
            m |= 1 << a
            if a == 0:
                break
            a = (a - 1) // 2
        masks.append(m)
    return np.array(masks, dtype=np.uint32)


def dense_sdpa(q_rows, k, v, visible, scale, G):
    """q_rows [R, Hq, D] f64, k/v [T, Hkv, D] f64, visible [R, T] bool -> [R, Hq, D]."""
    R, Hq, D = q_rows.shape
    kk = torch.from_numpy(np.repeat(k, G, axis=1)).permute(1, 0, 2)      # [Hq, T, D]
    vv = torch.from_numpy(np.repeat(v, G, axis=1)).permute(1, 0, 2)
    qq = torch.from_numpy(q_rows).permute(1, 0, 2)                       # [Hq, R, D]
    mask = torch.from_numpy(visible)[None].expand(Hq, R, -1)
    out = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask,
                                                           scale=float(scale))
    return out.permute(1, 0, 2).numpy()


def f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


# ------------------------------------------------------------------ pins
def pin_equal_counts_is_fixed_nq(o):
    for nq in (1, 3):
        lens = [nq, 17, 33, 100, 64 + nq]
        w = W.make_custom(len(lens), nq, 16, 4, 64, lens, seed=20 + nq)
        k, v = o.kv_append(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache)
        ref = o.paged_attention(w.q, k, v, w.block_tables, w.context_lens, nq, w.scale)
        qs = np.arange(len(lens) + 1, dtype=np.int32) * nq
        got = o.paged_attention_varlen(w.q, k, v, w.block_tables, w.context_lens, qs, w.scale)
        assert np.array_equal(got, ref)


def pin_varying_counts_are_per_sequence(o):
    qlen = [1, 4, 2, 3, 1]
    lens = [9, 40, 18, 100, 1]
    w = W.make_custom(len(lens), 1, 8, 2, 64, lens, seed=31, keep_full=True)
    rng = np.random.default_rng(3)
    qs = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    q = W.f32_to_bf16_bits(rng.standard_normal((int(qs[-1]), 8, 64)).astype(np.float32))
    got = o.paged_attention_varlen(q, w.k_full, w.v_full, w.block_tables, w.context_lens, qs,
                                   w.scale)
    assert np.isfinite(got).all()
    for s, n in enumerate(qlen):
        one = o.paged_attention(q[qs[s]:qs[s + 1]], w.k_full, w.v_full, w.block_tables[s:s + 1],
                                w.context_lens[s:s + 1], n, w.scale)
        assert np.array_equal(got[qs[s]:qs[s + 1]], one)


def pin_triangular_tree_is_causal(o):
    qlen = [4, 2, 3]
    lens = [30, 2, 50]
    w = W.make_custom(len(lens), 1, 8, 2, 64, lens, seed=32, keep_full=True)
    rng = np.random.default_rng(4)
    qs = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    q = W.f32_to_bf16_bits(rng.standard_normal((int(qs[-1]), 8, 64)).astype(np.float32))
    masks = np.concatenate([[(1 << (j + 1)) - 1 for j in range(n)] for n in qlen]).astype(np.uint32)
    causal = o.paged_attention_varlen(q, w.k_full, w.v_full, w.block_tables, w.context_lens, qs,
                                      w.scale)
    assert np.isfinite(causal).all()
    tree = o.paged_attention_varlen(q, w.k_full, w.v_full, w.block_tables, w.context_lens, qs,
                                    w.scale, tree_mask=masks, tree_len=np.array(qlen, np.int32))
    assert np.array_equal(causal, tree)


def pin_medusa_tree_matches_library(o):
    masks = binary_tree_masks(4)                 # 15 nodes
    n = masks.size
    T = 40 + n                                   # 40 cached tokens, then the 15 tree nodes
    w = W.make_custom(1, 1, 16, 2, 64, [T], seed=33, keep_dense=True, keep_full=True)
    rng = np.random.default_rng(5)
    q = W.f32_to_bf16_bits(rng.standard_normal((n, 16, 64)).astype(np.float32))
    qs = np.array([0, n], np.int32)
    got = o.paged_attention_varlen(q, w.k_full, w.v_full, w.block_tables, w.context_lens, qs,
                                   w.scale, tree_mask=masks, tree_len=np.array([n], np.int32))
    visible = np.zeros((n, T), dtype=bool)
    visible[:, :T - n] = True
    for j in range(n):
        for i in range(n):
            visible[j, T - n + i] = bool((int(masks[j]) >> i) & 1)
    ref = dense_sdpa(f64(q), f64(w.dense_k[0]), f64(w.dense_v[0]), visible, w.scale, 8)
    assert np.abs(got - ref).max() < 1e-12


def pin_chunked_equals_single_prefill(o):
    T = 64
    w = W.make_custom(1, 1, 8, 2, 64, [T], seed=34, keep_dense=True, keep_full=True)
    rng = np.random.default_rng(6)
    q = W.f32_to_bf16_bits(rng.standard_normal((T, 8, 64)).astype(np.float32))
    single = o.paged_attention_varlen(q, w.k_full, w.v_full, w.block_tables, w.context_lens,
                                      np.array([0, T], np.int32), w.scale)
    ends = np.cumsum([20, 30, 14])
    starts = ends - [20, 30, 14]
    qs = np.concatenate([[0], ends]).astype(np.int32)
    chunked = o.paged_attention_varlen(q, w.k_full, w.v_full, np.repeat(w.block_tables, 3, axis=0),
                                       ends.astype(np.int32), qs, w.scale)
    assert np.array_equal(single, chunked)
    visible = np.tril(np.ones((T, T), dtype=bool))
    ref = dense_sdpa(f64(q), f64(w.dense_k[0]), f64(w.dense_v[0]), visible, w.scale, 4)
    assert np.abs(single - ref).max() < 1e-12
    del starts


def pin_self_only_node_returns_its_value(o):
    n = 5
    w = W.make_custom(1, 1, 4, 1, 64, [n], seed=35, keep_dense=True, keep_full=True)
    rng = np.random.default_rng(7)
    q = W.f32_to_bf16_bits(rng.standard_normal((n, 4, 64)).astype(np.float32))
    masks = np.array([1 << i for i in range(n)], np.uint32)
    got = o.paged_attention_varlen(q, w.k_full, w.v_full, w.block_tables, w.context_lens,
                                   np.array([0, n], np.int32), w.scale, tree_mask=masks,
                                   tree_len=np.array([n], np.int32))
    vd = f64(w.dense_v[0])                       # [T, 1, D]
    for j in range(n):
        assert np.array_equal(got[j], np.repeat(vd[j], 4, axis=0))


VARLEN_PINS = [pin_equal_counts_is_fixed_nq, pin_varying_counts_are_per_sequence,
               pin_triangular_tree_is_causal, pin_medusa_tree_matches_library,
               pin_chunked_equals_single_prefill, pin_self_only_node_returns_its_value]


@pytest.mark.parametrize("pin", VARLEN_PINS, ids=lambda f: f.__name__)
def test_varlen_pin(o, pin):
    pin(o)


# every planted mistake keeps all reads and writes inside the caller's arrays
MUTANTS = {
    "window_start": ("const int32_t w0 = T - tree_len[s];", "const int32_t w0 = T - tree_len[s] + 1;"),
    "causal_strict": ("vis[t] = (uint8_t)(t <= T - ql + j);", "vis[t] = (uint8_t)(t < T - ql + j);"),
    "mask_bit_shift": ("((tree_mask[qr] >> (t - w0)) & 1u)", "((tree_mask[qr] >> (t - w0 + 1)) & 1u)"),
    "query_rows_reversed": ("const int64_t qr = (int64_t)q_start[s] + j;",
                            "const int64_t qr = (int64_t)q_start[s] + (ql - 1 - j);"),
    "no_causality_among_new": ("vis[t] = (uint8_t)(t <= T - ql + j);", "vis[t] = (uint8_t)(t < T);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_varlen_mutant_is_caught(name, tmp_path):
    src = open(oracle.SOURCE).read()
    before, after = MUTANTS[name]
    assert src.count(before) == 1, f"mutation site for {name} not found once"
    path = tmp_path / "mut.c"
    path.write_text(src.replace(before, after, 1))
    lib = tmp_path / "mut.so"
    oracle.build(str(path), str(lib), force=True)
    m = oracle.Oracle(oracle.load(str(lib)))
    caught = []
    for pin in VARLEN_PINS:
        try:
            pin(m)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"
