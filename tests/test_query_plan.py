"""The host planners: pkv_split_queries and the host checks of the
variable-query-count attention call, and pkv_cascade_pays (cascade or plain call).

The split must keep every query row's visibility: attention over the virtual
sequences, computed by the oracle, equals attention over the original ones bit
for bit, for causal runs (prefill chunks) and for tree masks.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_101_gb300 as pkv
import workloads as W
from paged_kv_cache_101_gb300 import _build

SHAPE, RANGE, NULL, ALIGN = 2, 5, 1, 4


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.lib()


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


def test_split_invariants(lib):
    rng = np.random.default_rng(0)
    qlen = rng.integers(0, 40, size=30)
    qs = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    T = (qlen + rng.integers(0, 300, size=30)).astype(np.int32)
    for m in (1, 3, 4, 32):
        r = pkv.split_queries(qs, T, m)
        vq, vc, vr = r["q_start"], r["context_lens"], r["table_row"]
        assert vq[0] == 0 and vq[-1] == qs[-1] and np.all(np.diff(vq) >= 1) and np.all(np.diff(vq) <= m)
        assert vr.size == sum(-(-int(n) // m) for n in qlen)
        for k in range(vr.size):
            s = vr[k]
            assert qs[s] <= vq[k] < vq[k + 1] <= qs[s + 1]
            for row in range(vq[k], vq[k + 1]):
                # causal limit of the row, before and after the split
                before = T[s] - qlen[s] + (row - qs[s])
                after = vc[k] - (vq[k + 1] - vq[k]) + (row - vq[k])
                assert before == after


def test_split_errors(lib):
    import ctypes
    nv = ctypes.c_int32(0)
    qs = np.array([0, 9], np.int32)
    T = np.array([20], np.int32)
    st = lib.pkv_split_queries(qs.ctypes.data, T.ctypes.data, None, 1, 4, None, None, None, None,
                               2, ctypes.byref(nv))
    assert st == RANGE and nv.value == 3                  # needs 3 runs, room for 2
    assert lib.pkv_split_queries(qs.ctypes.data, T.ctypes.data, None, 1, 0, None, None, None,
                                 None, 0, ctypes.byref(nv)) == SHAPE
    bad = np.array([0, -1], np.int32)
    assert lib.pkv_split_queries(bad.ctypes.data, T.ctypes.data, None, 1, 4, None, None, None,
                                 None, 0, ctypes.byref(nv)) == SHAPE
    tl = np.array([33], np.int32)
    assert lib.pkv_split_queries(qs.ctypes.data, T.ctypes.data, tl.ctypes.data, 1, 4, None, None,
                                 None, None, 0, ctypes.byref(nv)) == RANGE
    assert lib.pkv_split_queries(qs.ctypes.data, T.ctypes.data, None, 1, 4, None, None, None,
                                 None, 0, None) == NULL


def _random_tree(rng, n):
    """Ancestor-or-self masks of a random tree on n nodes (parents come first)."""
    masks = [1]
    for i in range(1, n):
        masks.append(masks[int(rng.integers(0, i))] | (1 << i))
    return masks


@pytest.mark.parametrize("tree", [False, True])
def test_split_keeps_the_oracle_result(lib, o, tree):
    rng = np.random.default_rng(1 + tree)
    qlen = [15, 1, 7, 0, 30] if tree else [64, 1, 9, 0, 33]
    ctx = [40, 3, 7, 5, 30] if tree else [0, 5, 20, 5, 2]
    T = [c + n for c, n in zip(ctx, qlen)]
    w = W.make_custom(len(T), 1, 8, 2, 64, [max(t, 1) for t in T], seed=40 + tree, keep_full=True)
    qs = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    q = W.f32_to_bf16_bits(rng.standard_normal((int(qs[-1]), 8, 64)).astype(np.float32))
    cl = np.array(T, np.int32)
    kw = {}
    if tree:
        masks = np.concatenate([_random_tree(rng, n) if n else [] for n in qlen]).astype(np.uint32)
        kw = dict(tree_mask=masks, tree_len=np.array(qlen, np.int32))
    ref = o.paged_attention_varlen(q, w.k_full, w.v_full, w.block_tables, cl, qs, w.scale, **kw)
    r = pkv.split_queries(qs, cl, 4, tree_len=kw.get("tree_len"))
    tables = w.block_tables[r["table_row"]]
    kv = dict(tree_mask=kw["tree_mask"], tree_len=r["tree_len"]) if tree else {}
    got = o.paged_attention_varlen(q, w.k_full, w.v_full, tables, r["context_lens"], r["q_start"],
                                   w.scale, **kv)
    assert np.array_equal(got, ref)


A = 0x10000


def varlen(lib, q=A, nb=64, bt=A, mb=8, ntr=4, tr=None, cl=A, qs=A, tm=None, tl=None, S=4,
           mq=2, tq=8, hq=8, hkv=2, d=64, out=A, ws=A):
    return lib.pkv_paged_decode_attention_varlen(q, A, A, nb, bt, mb, ntr, tr, cl, qs, tm, tl, S,
                                                 mq, tq, hq, hkv, d, 0.125, out, 0, ws, 1 << 30,
                                                 None)


def test_varlen_host_validation(lib):
    assert varlen(lib, S=0, qs=None) == 0
    assert varlen(lib, qs=None) == NULL
    assert varlen(lib, tm=A) == NULL                     # mask without its windows
    assert varlen(lib, tl=A) == NULL
    assert varlen(lib, ntr=2) == SHAPE                   # fewer table rows than sequences
    assert varlen(lib, tq=-1) == SHAPE
    assert varlen(lib, qs=A + 2) == ALIGN
    assert varlen(lib, mq=17) == 8                       # 4 x 17 = 68 score rows per kv head
    assert varlen(lib, hq=32, hkv=2, mq=5) == 8          # 80 rows per kv head
    # the geometry check (before any device query): 16 queries x 4 heads = 64 rows
    assert lib.pkv_workspace_size(0, 16, 8, 2, 64) == 256
    assert lib.pkv_workspace_size(0, 17, 8, 2, 64) == 0


def cascade(lib, groups=A, ng=2, mg=8, S=4, nq=1, hq=8, hkv=2, d=64, ws=A):
    return lib.pkv_paged_decode_attention_cascade(A, A, A, 64, A, 8, A, S, nq, hq, hkv, d, 0.125,
                                                  groups, ng, mg, A, 0, ws, 1 << 30, None)


def test_cascade_host_validation(lib):
    assert cascade(lib, S=0) == 0
    assert cascade(lib, groups=None) == NULL
    assert cascade(lib, groups=A + 2) == ALIGN
    assert cascade(lib, ng=-1) == SHAPE
    assert cascade(lib, ng=5) == RANGE                   # more groups than sequences
    assert cascade(lib, mg=9) == RANGE
    assert cascade(lib, nq=5, mg=4) == 8
    # the cascade's workspace adds the prefix partials to the plain one
    assert lib.pkv_workspace_size_cascade(4, 1, 8, 2, 64) == 0 or \
        lib.pkv_workspace_size_cascade(4, 1, 8, 2, 64) > lib.pkv_workspace_size(4, 1, 8, 2, 64)


# ------------------------------------------------------------------ cascade rule
def shared_prompt_lengths(S=256, prefix=4096, suffix_max=512, seed=1234 + 23):
    """A shared-prompt batch like the benchmark's: a system prompt of `prefix`
    tokens and private suffixes of 16 .. suffix_max - 1 tokens."""
    rng = np.random.default_rng(seed)
    return (prefix + rng.integers(16, suffix_max, size=S)).astype(np.int32)


# (prompt tokens, largest suffix, faster path measured on GB300 at 8 kv heads x 128
# dims); a tie (under 1 %) is listed under the rule's answer
MEASURED = [(4096, 512, True), (2048, 512, True), (4096, 4096, True), (1024, 512, False),
            (512, 512, False), (512, 4096, False), (1024, 2048, False), (2048, 4096, True)]


@pytest.mark.parametrize("prefix,suffix,cascade", MEASURED)
def test_cascade_rule_matches_the_measured_faster_path(lib, prefix, suffix, cascade):
    lens = shared_prompt_lengths(prefix=prefix, suffix_max=suffix)
    assert pkv.cascade_pays(lens, [[0, lens.size, prefix // 16]], 8, 128) == cascade


def test_cascade_rule_picks_the_plain_call_for_the_70b_mix(lib):
    T, shared, prefix = W.workload_lengths("llama3_70b_mix")
    lens = np.concatenate([T[shared], T[~shared]]).astype(np.int32)   # sharers first
    assert not pkv.cascade_pays(lens, [[0, int(shared.sum()), prefix // 16]], 8, 128)


def test_cascade_rule_edges(lib):
    lens = np.full(8, 600, np.int32)
    assert not pkv.cascade_pays(lens, np.zeros((0, 3), np.int32), 8, 128)    # no group
    assert not pkv.cascade_pays(lens, [[0, 1, 32]], 8, 128)                 # a lone member
    # members whose context is the prefix alone fall back, so they repeat nothing
    assert not pkv.cascade_pays(np.full(8, 512, np.int32), [[0, 8, 32]], 8, 128)
    # repeated >= unique, but 7 copies of 512 tokens are far below the fixed price
    assert not pkv.cascade_pays(lens, [[0, 8, 32]], 8, 128)
    # 4,000 sequences of a 4,096-token prompt: far above it
    big = np.full(4000, 4096 + 8, np.int32)
    assert pkv.cascade_pays(big, [[0, 4000, 256]], 8, 128)
    with pytest.raises(ValueError):
        pkv.cascade_pays(lens, [[4, 8, 32]], 8, 128)                        # past the batch
