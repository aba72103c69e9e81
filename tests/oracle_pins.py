"""Checks that pin the fp64 oracle to facts other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises ``AssertionError``
(or ``ValueError``) when the oracle disagrees with:

* dense attention computed by a library routine (``torch`` scaled-dot-product
  attention in float64) on the generator's dense, never-paged K/V;
* invariance of the output under a random relabelling of physical block ids;
* softmax weights that sum to one, lie in [0, 1] and vanish past the causal limit;
* equality of a physically shared prefix with privately copied prefix blocks;
* closed forms (one token, zero query, constant V, one dominant key, scale 0);
* the block-table diagram of "07 -- Inference" section 2.2 (A -> [0, 3, 5]);
* the split/merge algebra of "07 -- Inference" section 5.3;
* the generator's independently built post-append pool (for the append).

They are functions, not tests, so ``test_oracle_mutants.py`` can run them against
oracle builds with planted mistakes and show that every mistake trips one.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _small_cases():
    """Small workloads covering GQA groups 1/4/8, nq 1..4, D 64/128, ragged tails."""
    cases = [W.make_workload("tiny", keep_dense=True, keep_full=True)]
    cases.append(W.make_custom(5, 4, 16, 2, 128, [4, 16, 17, 31, 50], seed=11,
                               keep_dense=True, keep_full=True))
    cases.append(W.make_custom(3, 2, 4, 4, 64, [2, 19, 40], seed=12,
                               keep_dense=True, keep_full=True))
    sh = np.array([True, False, True, True, False, False])
    cases.append(W.make_custom(6, 1, 8, 2, 64, [40, 33, 64, 36, 5, 90], seed=13, shared=sh,
                               prefix_tokens=32, keep_dense=True, keep_full=True))
    return cases


def _torch_dense(w):
    """Dense reference: torch SDPA in float64 over each sequence's dense K/V."""
    import torch
    import torch.nn.functional as F

    S, nq, Hq, Hkv, D = w.num_seqs, w.n_query_per_seq, w.num_q_heads, w.num_kv_heads, w.head_dim
    G = Hq // Hkv
    q = torch.from_numpy(W.bf16_bits_to_f32(w.q).astype(np.float64)).reshape(S, nq, Hq, D)
    out = np.zeros((S * nq, Hq, D))
    for s in range(S):
        T = int(w.context_lens[s])
        K = torch.from_numpy(W.bf16_bits_to_f32(w.dense_k[s]).astype(np.float64))  # [T,Hkv,D]
        V = torch.from_numpy(W.bf16_bits_to_f32(w.dense_v[s]).astype(np.float64))
        t = torch.arange(T)[None, :]
        j = torch.arange(nq)[:, None]
        mask = t <= (T - nq + j)                                               # [nq, T]
        for h in range(Hkv):
            Q = q[s, :, h * G:(h + 1) * G, :].permute(1, 0, 2)                   # [G, nq, D]
            Kh = K[:, h, :].unsqueeze(0).expand(G, T, D)
            Vh = V[:, h, :].unsqueeze(0).expand(G, T, D)
            o = F.scaled_dot_product_attention(Q, Kh, Vh, attn_mask=mask, scale=float(w.scale))
            out[s * nq:(s + 1) * nq, h * G:(h + 1) * G, :] = o.permute(1, 0, 2).numpy()
    return out


def pin_dense_library(o, cases=None):
    for w in cases or _small_cases():
        ref = _torch_dense(w)
        got = o.paged_attention(w.q, w.k_full, w.v_full, w.block_tables, w.context_lens,
                                w.n_query_per_seq, w.scale)
        err = np.max(np.abs(got - ref))
        assert err <= 1e-12, f"{w.name}: oracle vs dense library attention max-abs {err}"


def pin_append_matches_generator(o, cases=None):
    for w in cases or _small_cases():
        k, v = o.kv_append(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache)
        assert np.array_equal(k, w.k_full) and np.array_equal(v, w.v_full), w.name
    # a padding slot (-1) writes nothing
    w = cases[0] if cases else W.make_workload("tiny", keep_full=True)
    slots = w.slot_mapping.copy()
    slots[1] = -1
    k, v = o.kv_append(w.k_new, w.v_new, slots, w.k_cache, w.v_cache)
    blk, off = divmod(int(w.slot_mapping[1]), 16)
    assert np.all(k[blk, off] == W.SENTINEL_BF16) and np.all(v[blk, off] == W.SENTINEL_BF16)
    mask = np.ones(w.k_cache.shape[:2], dtype=bool)
    mask[blk, off] = False
    assert np.array_equal(k[mask], w.k_full[mask]) and np.array_equal(v[mask], w.v_full[mask])


def pin_permutation_invariance(o):
    sh = np.array([True, True, False, True])
    w = W.make_custom(4, 2, 8, 2, 64, [50, 41, 77, 34], seed=21, shared=sh, prefix_tokens=32,
                      keep_full=True)
    for seed in (1, 2):
        p = W.permute_pool(w, seed=seed)
        a = o.paged_attention(w.q, w.k_full, w.v_full, w.block_tables, w.context_lens, 2, w.scale)
        b = o.paged_attention(p.q, p.k_full, p.v_full, p.block_tables, p.context_lens, 2, p.scale)
        assert not np.array_equal(w.block_tables, p.block_tables)
        assert np.array_equal(a, b), "output changed under a relabelling of physical blocks"


def pin_weight_sums(o):
    w = W.make_custom(3, 4, 8, 2, 64, [5, 23, 48], seed=31, keep_full=True)
    for s in range(3):
        T = int(w.context_lens[s])
        for j in range(4):
            for qh in (0, 3, 5):
                wt = o.attention_weights(w.q, w.k_full, w.v_full, w.block_tables,
                                         w.context_lens, 4, w.scale, s, j, qh)
                lim = T - 4 + j
                assert wt.shape == (T,)
                assert abs(wt.sum() - 1.0) <= 1e-12
                assert np.all(wt >= 0) and np.all(wt <= 1)
                assert np.all(wt[lim + 1:] == 0.0), "weight past the causal limit"
                assert np.all(wt[: lim + 1] > 0.0)


def pin_shared_equals_copied(o):
    sh = np.array([True, False, True, True, False, True])
    w = W.make_custom(6, 1, 8, 2, 64, [40, 33, 64, 49, 5, 90], seed=41, shared=sh,
                      prefix_tokens=32, keep_full=True)
    w.k_cache, w.v_cache = w.k_full, w.v_full
    u = W.unshare_prefix(w)
    assert u.num_blocks > w.num_blocks
    a = o.paged_attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, 1, w.scale)
    b = o.paged_attention(u.q, u.k_cache, u.v_cache, u.block_tables, u.context_lens, 1, u.scale)
    assert np.array_equal(a, b), "shared prefix differs from copied prefix"


def _bf(x):
    return W.f32_to_bf16_bits(np.asarray(x, dtype=np.float32).copy())


def pin_closed_forms(o):
    rng = np.random.default_rng(51)
    # (a) one token: the output is V[0] exactly
    w = W.make_custom(3, 1, 8, 2, 64, [1, 1, 1], seed=52, keep_full=True, keep_dense=True)
    got = o.paged_attention(w.q, w.k_full, w.v_full, w.block_tables, w.context_lens, 1, w.scale)
    for s in range(3):
        for qh in range(8):
            v0 = W.bf16_bits_to_f32(w.dense_v[s][0, qh // 4]).astype(np.float64)
            assert np.array_equal(got[s, qh], v0)
    # (b) zero query, and (e) scale 0: the mean of the visible V rows
    w = W.make_custom(3, 3, 8, 4, 64, [3, 20, 33], seed=53, keep_full=True, keep_dense=True)
    zq = np.zeros_like(w.q)
    for q_in, sc in ((zq, w.scale), (w.q, 0.0)):
        got = o.paged_attention(q_in, w.k_full, w.v_full, w.block_tables, w.context_lens, 3, sc)
        for s in range(3):
            T = int(w.context_lens[s])
            V = W.bf16_bits_to_f32(w.dense_v[s]).astype(np.float64)
            for j in range(3):
                lim = T - 3 + j
                for qh in range(8):
                    mean = V[: lim + 1, qh // 2].mean(axis=0)
                    assert np.max(np.abs(got[s * 3 + j, qh] - mean)) <= 1e-13
    # (c) constant V rows: the output is that constant
    c = _bf(rng.standard_normal((2, 64)))

    def vconst(kind, s, shape, r):
        x = W._normal_bf16(r, shape)
        if kind in ("v", "pv"):
            x[...] = c[None, :, :]
        return x
    w = W.make_custom(2, 2, 4, 2, 64, [7, 45], seed=54, keep_full=True, value_fn=vconst)
    got = o.paged_attention(w.q, w.k_full, w.v_full, w.block_tables, w.context_lens, 2, w.scale)
    cf = W.bf16_bits_to_f32(c).astype(np.float64)
    for r in range(4):
        for qh in range(4):
            assert np.max(np.abs(got[r, qh] - cf[qh // 2])) <= 1e-13
    # (d) one dominant key: the output is that token's V
    T = [37, 20]
    star = {0: 29, 1: 3}

    def kdom(kind, s, shape, r):
        x = W._normal_bf16(r, shape)
        if kind == "k":
            x[...] = _bf(-16.0)
            x[star[s]] = _bf(16.0)
        if kind == "q":
            x[...] = _bf(16.0)
        return x
    w = W.make_custom(2, 1, 4, 2, 64, T, seed=55, keep_full=True, keep_dense=True, value_fn=kdom)
    got = o.paged_attention(w.q, w.k_full, w.v_full, w.block_tables, w.context_lens, 1, w.scale)
    for s in range(2):
        for qh in range(4):
            vt = W.bf16_bits_to_f32(w.dense_v[s][star[s], qh // 2]).astype(np.float64)
            assert np.array_equal(got[s, qh], vt)


def pin_block_table_diagram(o):
    """Sequence A of the diagram: 38 tokens in physical blocks 0, 3 and 5."""
    g = json.load(open(os.path.join(GOLDEN, "block_table_diagram.json")))
    bs, table, T = g["block_size"], g["block_table"], g["context_len"]
    NB, Hkv, D = 6, 1, 64
    # V[b][r] holds the value 16*b + r in every element; K = 0 unless a test sets it.
    v = np.empty((NB, bs, Hkv, D), dtype=np.uint16)
    for b in range(NB):
        for r in range(bs):
            v[b, r] = _bf(16.0 * b + r)
    k = np.zeros_like(v)
    bt = np.array([table], dtype=np.int32)
    cl = np.array([T], dtype=np.int32)
    q = np.zeros((1, 1, D), dtype=np.uint16)
    expected = []
    for seg in g["logical_to_physical"]:
        for r in range(seg["rows"][0], seg["rows"][1] + 1):
            expected.append(16.0 * seg["physical_block"] + r)
    assert len(expected) == T
    got = o.paged_attention(q, k, v, bt, cl, 1, 0.125)
    assert abs(got[0, 0, 0] - np.mean(expected)) <= 1e-12
    # a dominant key at logical token t picks out exactly its physical slot
    qd = np.full((1, 1, D), _bf(16.0), dtype=np.uint16)
    for t in (0, 15, 16, 31, 32, 37):
        kk = np.full_like(v, _bf(-16.0))
        blk, r = table[t // bs], t % bs
        kk[blk, r] = _bf(16.0)
        got = o.paged_attention(qd, kk, v, bt, cl, 1, 0.125)
        assert got[0, 0, 0] == expected[t]


def pin_merge_algebra(o):
    w = W.make_custom(2, 2, 8, 2, 64, [70, 129], seed=61, keep_full=True)
    full = o.paged_attention(w.q, w.k_full, w.v_full, w.block_tables, w.context_lens, 2, w.scale)
    rng = np.random.default_rng(62)
    for s in range(2):
        T = int(w.context_lens[s])
        for j in range(2):
            for qh in (1, 6):
                for nparts in (1, 2, 5):
                    cuts = np.sort(rng.choice(np.arange(1, T), size=nparts - 1, replace=False))
                    edges = [0, *cuts.tolist(), T]
                    ms, ls, accs = [], [], []
                    for a, b in zip(edges[:-1], edges[1:]):
                        m, l, acc = o.partial_state(w.q, w.k_full, w.v_full, w.block_tables,
                                                    w.context_lens, 2, w.scale, s, j, qh, a, b)
                        ms.append(m)
                        ls.append(l)
                        accs.append(acc)
                    merged = o.merge_states(ms, ls, np.array(accs))
                    err = np.max(np.abs(merged - full[s * 2 + j, qh]))
                    assert err <= 1e-12, f"merge of {nparts} partials differs by {err}"


ALL_PINS = [pin_dense_library, pin_append_matches_generator, pin_permutation_invariance,
            pin_weight_sums, pin_shared_equals_copied, pin_closed_forms,
            pin_block_table_diagram, pin_merge_algebra]
