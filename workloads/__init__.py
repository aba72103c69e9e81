"""Seeded synthetic inputs for paged decode attention and the KV-cache append.

This module only *makes inputs*: pools of 16-token physical blocks, per-sequence
block tables, context lengths, queries and the new tokens of one decode step. It
holds none of the attention arithmetic and none of the append's logic, so that
the fp64 oracle (``oracle/``) and the CUDA library can both be fed from it
without sharing any of the method's code.

Layouts follow the paged KV cache described in "LLM Inference Serving"
(systeminternals.dev, KV-cache shape section): K and V are each stored as
``[num_blocks, block_size, num_kv_heads, head_dim]``; a per-sequence block table
maps logical block ``i`` (tokens ``16i .. 16i+15``) to a physical block id
("ML Interview Prep, Lesson 13", section 3.5 "Paged attention").

Values are i.i.d. N(0, 1) samples rounded to bfloat16 (round to nearest even)
and carried as their 16-bit patterns (``uint16``). Unused slots of the pool hold
a NaN bit pattern, so a kernel that reads outside a sequence's context (or the
last block's free slots) without masking shows up as NaN in its output.

Seeding: every stream (lengths, pool permutation, prefix choice, queries, and
the K/V values of each sequence) draws from its own ``numpy`` PCG64 generator
spawned from ``SeedSequence(seed)``; the K/V values of sequence ``s`` come in 4096-token
chunks from the keys ``(seed, 7, s, chunk)`` so a workload is identical whatever
the number of worker threads.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

BLOCK_SIZE = 16
# A bf16 quiet-NaN pattern that marks pool slots holding no token.
SENTINEL_BF16 = np.uint16(0x7FC1)

# Tokens per generator chunk of a sequence's K/V values (a multiple of 16).
CHUNK_TOKENS = 4096

# Stream ids inside one workload's SeedSequence.
_S_LENS, _S_PERM, _S_SHARE, _S_Q, _S_KV = 1, 2, 3, 4, 7
_S_FP8 = 11
E4M3_NAN = np.uint8(0x7F)  # the E4M3 code S.1111.111 is NaN


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 samples to bfloat16 (nearest, ties to even); return bit patterns.

    Destroys ``x`` (works in place on its bits). Inputs are finite samples.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    t = np.right_shift(u, 16)
    np.bitwise_and(t, 1, out=t)
    t += np.uint32(0x7FFF)
    u += t
    # little endian: the upper 16 bits of each word are the odd uint16 lanes
    return np.ascontiguousarray(u.view(np.uint16)[..., 1::2]).reshape(u.shape)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


@dataclass
class Workload:
    """One decode step's inputs (all host arrays; bf16 carried as uint16 bits)."""

    name: str
    seed: int
    num_seqs: int
    n_query_per_seq: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    scale: np.float32
    num_blocks: int
    max_blocks_per_seq: int
    context_lens: np.ndarray          # int32 [S], tokens INCLUDING this step's nq new ones
    block_tables: np.ndarray          # int32 [S, MB], -1 past ceil(T_s/16)
    q: np.ndarray                     # uint16 [S*nq, Hq, D]
    k_cache: np.ndarray               # uint16 [NB, 16, Hkv, D] before this step's append
    v_cache: np.ndarray
    k_new: np.ndarray                 # uint16 [S*nq, Hkv, D]: K of the step's new tokens
    v_new: np.ndarray
    slot_mapping: np.ndarray          # int64 [S*nq]: physical_block*16 + offset
    shared: np.ndarray                # bool [S]: sequence reads the shared prefix blocks
    prefix_blocks: np.ndarray         # int32 [n_prefix]: physical ids of the shared prefix
    k_full: Optional[np.ndarray] = None   # pool after the append (built independently)
    v_full: Optional[np.ndarray] = None
    dense_k: Optional[List[np.ndarray]] = None  # per sequence [T_s, Hkv, D] in logical order
    dense_v: Optional[List[np.ndarray]] = None
    meta: dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def nblocks(self) -> np.ndarray:
        return (self.context_lens.astype(np.int64) + BLOCK_SIZE - 1) // BLOCK_SIZE

    def unique_blocks(self) -> int:
        """Physical blocks the step reads, shared prefix blocks counted once."""
        used = set()
        for s in range(self.num_seqs):
            used.update(self.block_tables[s, : int(self.nblocks()[s])].tolist())
        return len(used)


# ----------------------------------------------------------------------------
# The five workloads (shapes, length laws and pool structure as stated for the
# synthetic benchmark); seed = 1234 + workload index.
# ----------------------------------------------------------------------------
WORKLOADS = {
    "tiny": dict(index=0, S=4, nq=1, Hq=8, Hkv=2, D=64),
    "llama3_8b_decode": dict(index=1, S=64, nq=1, Hq=32, Hkv=8, D=128),
    "llama3_70b_mix": dict(index=2, S=256, nq=1, Hq=64, Hkv=8, D=128),
    "long_splitk": dict(index=3, S=8, nq=1, Hq=32, Hkv=8, D=128),
    "spec_verify": dict(index=4, S=128, nq=4, Hq=64, Hkv=8, D=128),
}
WORKLOAD_ORDER = ["tiny", "llama3_8b_decode", "llama3_70b_mix", "long_splitk", "spec_verify"]


def workload_lengths(name: str, seed: Optional[int] = None):
    """Context lengths (after the append) and prefix sharing of a named workload.

    Returns ``(context_lens int64 [S], shared bool [S], prefix_tokens int)``.
    """
    cfg = WORKLOADS[name]
    if seed is None:
        seed = 1234 + cfg["index"]
    S = cfg["S"]
    shared = np.zeros(S, dtype=bool)
    prefix_tokens = 0
    r = _rng(seed, _S_LENS)
    if name == "tiny":
        T = np.array([17, 33, 64, 100], dtype=np.int64)
    elif name == "llama3_8b_decode":
        T = r.integers(512, 4096, size=S, endpoint=True)
    elif name == "llama3_70b_mix":
        T = np.rint(np.exp(r.normal(math.log(1024.0), 1.0, size=S)))
        T = np.clip(T, 16, 8192).astype(np.int64)
        # half of the batch shares one 512-token system prompt (32 blocks); a
        # sharer holds at least one private token past it, so this step's new
        # token never lands in a shared block.
        prefix_tokens = 512
        idx = _rng(seed, _S_SHARE).choice(S, size=S // 2, replace=False)
        shared[idx] = True
        T[shared] = np.maximum(T[shared], prefix_tokens + 1)
    elif name == "long_splitk":
        T = r.integers(32768, 131072, size=S, endpoint=True)
    elif name == "spec_verify":
        T = r.integers(1024, 4096, size=S, endpoint=True) + cfg["nq"]
    else:  # pragma: no cover
        raise KeyError(name)
    return T.astype(np.int64), shared, prefix_tokens


def make_workload(name: str, seed: Optional[int] = None, keep_full: bool = False,
                  keep_dense: bool = False, threads: Optional[int] = None) -> Workload:
    """Build one of the five named workloads."""
    cfg = WORKLOADS[name]
    if seed is None:
        seed = 1234 + cfg["index"]
    T, shared, prefix_tokens = workload_lengths(name, seed)
    num_blocks = 64 if name == "tiny" else None
    scale = np.float32(1.0 / math.sqrt(cfg["D"]))
    return make_custom(cfg["S"], cfg["nq"], cfg["Hq"], cfg["Hkv"], cfg["D"], T,
                       seed=seed, name=name, shared=shared, prefix_tokens=prefix_tokens,
                       num_blocks=num_blocks, scale=scale, keep_full=keep_full,
                       keep_dense=keep_dense, threads=threads)


def make_custom(S: int, nq: int, Hq: int, Hkv: int, D: int, context_lens: Sequence[int],
                seed: int = 99, name: str = "custom", shared=None, prefix_tokens: int = 0,
                num_blocks: Optional[int] = None, pool_factor: float = 1.25,
                scale: Optional[float] = None, keep_full: bool = False,
                keep_dense: bool = False, threads: Optional[int] = None,
                value_fn=None) -> Workload:
    """Build a workload of any shape.

    ``context_lens`` counts every token of a sequence including this step's
    ``nq`` new ones. Sequences flagged in ``shared`` start with the same
    ``prefix_tokens`` tokens (a multiple of 16), stored once in the pool and
    referenced by all of their block tables. The pool holds
    ``ceil(pool_factor * blocks_needed)`` blocks (or ``num_blocks``), assigned by
    a seeded permutation of the physical ids. ``value_fn(kind, s, shape, rng)``
    may replace the N(0,1) bf16 values (``kind`` in {"k", "v", "q", "pk", "pv"}).
    """
    T = np.asarray(context_lens, dtype=np.int64).reshape(-1)
    assert T.shape[0] == S and S >= 0
    assert Hq % Hkv == 0 and D % 8 == 0 and nq >= 1
    assert S == 0 or T.min() >= nq, "every sequence holds at least its nq new tokens"
    if shared is None:
        shared = np.zeros(S, dtype=bool)
    shared = np.asarray(shared, dtype=bool)
    assert prefix_tokens % BLOCK_SIZE == 0
    if prefix_tokens == 0:
        shared = np.zeros(S, dtype=bool)
    assert np.all(T[shared] > prefix_tokens), "a sharer must own tokens past the prefix"
    n_prefix = prefix_tokens // BLOCK_SIZE
    nb = (T + BLOCK_SIZE - 1) // BLOCK_SIZE
    private = nb - np.where(shared, n_prefix, 0)
    need = int(private.sum()) + (n_prefix if shared.any() else 0)
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(pool_factor * need)))
    assert num_blocks >= need, "pool too small"
    MB = int(max(1, nb.max() if S else 1))
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    scale = np.float32(scale)

    # physical ids: a seeded permutation of the pool, handed out in order
    perm = _rng(seed, _S_PERM).permutation(num_blocks).astype(np.int32)
    cursor = 0
    prefix_ids = np.zeros(0, dtype=np.int32)
    if shared.any():
        prefix_ids = perm[:n_prefix].copy()
        cursor = n_prefix
    tables = np.full((S, MB), -1, dtype=np.int32)
    for s in range(S):
        own = int(private[s])
        ids = perm[cursor: cursor + own]
        cursor += own
        if shared[s]:
            tables[s, :n_prefix] = prefix_ids
            tables[s, n_prefix: n_prefix + own] = ids
        else:
            tables[s, :own] = ids

    gen = value_fn if value_fn is not None else (lambda kind, s, shape, rng: _normal_bf16(rng, shape))

    k_full = np.empty((num_blocks, BLOCK_SIZE, Hkv, D), dtype=np.uint16)
    v_full = np.empty_like(k_full)
    k_full.fill(SENTINEL_BF16)
    v_full.fill(SENTINEL_BF16)

    def scatter(pool, vals, ids, first_token):
        # vals: [n, Hkv, D] for tokens first_token .. first_token+n-1 of a sequence
        n = vals.shape[0]
        if n == 0:
            return
        nfull = n // BLOCK_SIZE
        if nfull:
            pool[ids[first_token // BLOCK_SIZE: first_token // BLOCK_SIZE + nfull]] = \
                vals[: nfull * BLOCK_SIZE].reshape(nfull, BLOCK_SIZE, Hkv, D)
        rem = n - nfull * BLOCK_SIZE
        if rem:
            pool[ids[(first_token + nfull * BLOCK_SIZE) // BLOCK_SIZE], :rem] = vals[nfull * BLOCK_SIZE:]

    pk = pv = None
    if shared.any():
        r = _rng(seed, _S_KV, S)
        pk = gen("pk", S, (prefix_tokens, Hkv, D), r)
        pv = gen("pv", S, (prefix_tokens, Hkv, D), r)
        scatter(k_full, pk, prefix_ids, 0)
        scatter(v_full, pv, prefix_ids, 0)

    dense_k = [None] * S if keep_dense else None
    dense_v = [None] * S if keep_dense else None
    if keep_dense:
        for s in range(S):
            dense_k[s] = np.empty((int(T[s]), Hkv, D), dtype=np.uint16)
            dense_v[s] = np.empty((int(T[s]), Hkv, D), dtype=np.uint16)
            if shared[s]:
                dense_k[s][:prefix_tokens] = pk
                dense_v[s][:prefix_tokens] = pv

    # a sequence's own tokens come in chunks of CHUNK_TOKENS, each from the
    # generator keyed (seed, 7, s, chunk): identical whatever the thread count
    tasks = []
    for s in range(S):
        start = n_prefix * BLOCK_SIZE if shared[s] else 0
        n = int(T[s]) - start
        for c in range(0, max(n, 0), CHUNK_TOKENS):
            tasks.append((s, start, c, min(CHUNK_TOKENS, n - c)))

    def fill(task):
        s, start, c, n = task
        r = _rng(seed, _S_KV, s, c // CHUNK_TOKENS)
        kv = gen("k", s, (n, Hkv, D), r)
        vv = gen("v", s, (n, Hkv, D), r)
        scatter(k_full, kv, tables[s], start + c)
        scatter(v_full, vv, tables[s], start + c)
        if keep_dense:
            dense_k[s][start + c: start + c + n] = kv
            dense_v[s][start + c: start + c + n] = vv

    nthreads = threads or min(16, os.cpu_count() or 1)
    if nthreads > 1 and len(tasks) > 1:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(fill, tasks))
    else:
        for t in tasks:
            fill(t)

    q = gen("q", -1, (S * nq, Hq, D), _rng(seed, _S_Q))

    # this step's new tokens: the last nq of every sequence
    pos = (T[:, None] - nq + np.arange(nq)[None, :]).reshape(-1)          # [S*nq]
    seq = np.repeat(np.arange(S), nq)
    if S:
        phys = tables[seq, pos // BLOCK_SIZE].astype(np.int64)
        slot = phys * BLOCK_SIZE + pos % BLOCK_SIZE
    else:
        phys = np.zeros(0, dtype=np.int64)
        slot = np.zeros(0, dtype=np.int64)
    k_new = k_full[phys, pos % BLOCK_SIZE].copy() if S else np.zeros((0, Hkv, D), np.uint16)
    v_new = v_full[phys, pos % BLOCK_SIZE].copy() if S else np.zeros((0, Hkv, D), np.uint16)
    if keep_full:
        k_cache = k_full.copy()
        v_cache = v_full.copy()
    else:
        k_cache, v_cache = k_full, v_full
        k_full = v_full = None
    if S:
        k_cache[phys, pos % BLOCK_SIZE] = SENTINEL_BF16
        v_cache[phys, pos % BLOCK_SIZE] = SENTINEL_BF16

    return Workload(
        name=name, seed=seed, num_seqs=S, n_query_per_seq=nq, num_q_heads=Hq,
        num_kv_heads=Hkv, head_dim=D, scale=scale, num_blocks=num_blocks,
        max_blocks_per_seq=MB, context_lens=T.astype(np.int32), block_tables=tables,
        q=q, k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
        slot_mapping=slot.astype(np.int64), shared=shared, prefix_blocks=prefix_ids,
        k_full=k_full, v_full=v_full, dense_k=dense_k, dense_v=dense_v,
        meta=dict(prefix_tokens=prefix_tokens, blocks_needed=need))


def permute_pool(w: Workload, seed: int = 5) -> Workload:
    """Return a copy of ``w`` with its physical block ids relabelled by a random permutation.

    Block ``b`` moves to ``pi[b]`` and every table entry ``b`` becomes ``pi[b]``;
    the logical content of every sequence is unchanged.
    """
    pi = _rng(seed, 11).permutation(w.num_blocks).astype(np.int32)
    inv = np.empty_like(pi)
    inv[pi] = np.arange(w.num_blocks, dtype=np.int32)
    out = Workload(**{**w.__dict__})
    out.k_cache = w.k_cache[inv]
    out.v_cache = w.v_cache[inv]
    out.block_tables = np.where(w.block_tables >= 0, pi[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    if w.k_full is not None:
        out.k_full = w.k_full[inv]
        out.v_full = w.v_full[inv]
    out.slot_mapping = (pi[w.slot_mapping // BLOCK_SIZE].astype(np.int64) * BLOCK_SIZE
                        + w.slot_mapping % BLOCK_SIZE)
    out.prefix_blocks = pi[w.prefix_blocks] if w.prefix_blocks.size else w.prefix_blocks
    return out


def unshare_prefix(w: Workload) -> Workload:
    """Return a copy of ``w`` in which every sharer owns a private copy of the prefix.

    The copies go to freshly appended physical blocks at the end of the pool.
    """
    n_prefix = w.meta.get("prefix_tokens", 0) // BLOCK_SIZE
    sharers = np.nonzero(w.shared)[0]
    if n_prefix == 0 or sharers.size == 0:
        return w
    extra = n_prefix * sharers.size
    nb_new = w.num_blocks + extra
    def grow(pool):
        out = np.empty((nb_new,) + pool.shape[1:], dtype=pool.dtype)
        out[: w.num_blocks] = pool
        out[w.num_blocks:] = SENTINEL_BF16
        return out
    k = grow(w.k_cache)
    v = grow(w.v_cache)
    tables = w.block_tables.copy()
    nxt = w.num_blocks
    for s in sharers:
        ids = np.arange(nxt, nxt + n_prefix, dtype=np.int32)
        k[ids] = w.k_cache[w.prefix_blocks]
        v[ids] = w.v_cache[w.prefix_blocks]
        tables[s, :n_prefix] = ids
        nxt += n_prefix
    out = Workload(**{**w.__dict__})
    out.num_blocks = nb_new
    out.k_cache, out.v_cache, out.block_tables = k, v, tables
    out.shared = np.zeros_like(w.shared)
    out.prefix_blocks = np.zeros(0, dtype=np.int32)
    out.k_full = out.v_full = None
    return out


# ----------------------------------------------------------------------------
# FP8 (E4M3) pools standing in for a workload's bf16 pools
# ----------------------------------------------------------------------------
def fp8_pools(w: Workload, seed: Optional[int] = None):
    """uint8 code pools of the same shape as ``w``'s pools, and per-kv-head scales.

    Every slot that holds a token gets a random E4M3 code with an exponent field
    in 1..10 (magnitudes 2^-6 .. 15, i.e. 0.004 .. 3.75 after a scale near 1/4),
    any mantissa and either sign; slots without a token (and this step's new
    slots, which the append fills) hold the NaN code. Codes are drawn as bit
    fields: no value is encoded here. Scales: K 0.25 * (1 + h/16), V
    0.3 * (1 + h/32) for kv head h (float32). Returns (k8, v8, k_scale, v_scale).
    """
    rng = _rng(w.seed if seed is None else seed, _S_FP8)

    def codes(pool):
        r = rng.integers(0, 256, size=pool.shape, dtype=np.uint8)
        field = (((r >> 3) & np.uint8(15)) % np.uint8(10)) + np.uint8(1)
        c = (r & np.uint8(0x87)) | (field << np.uint8(3))
        c[pool == SENTINEL_BF16] = E4M3_NAN
        return c

    k8 = codes(w.k_cache)
    v8 = codes(w.v_cache)
    h = np.arange(w.num_kv_heads, dtype=np.float32)
    k_scale = (np.float32(0.25) * (np.float32(1) + h / np.float32(16))).astype(np.float32)
    v_scale = (np.float32(0.3) * (np.float32(1) + h / np.float32(32))).astype(np.float32)
    return k8, v8, k_scale, v_scale


def sharers_first(w: Workload) -> Workload:
    """The same batch with the sequences that share the prefix moved to the front
    (their order kept), so they form one consecutive group. Rows of q, the new
    tokens and the slots move with their sequence (any n_query_per_seq)."""
    order = np.concatenate([np.nonzero(w.shared)[0], np.nonzero(~w.shared)[0]])
    nq = w.n_query_per_seq
    rows = (order[:, None] * nq + np.arange(nq)[None, :]).reshape(-1)
    w.context_lens = w.context_lens[order].copy()
    w.block_tables = w.block_tables[order].copy()
    w.shared = w.shared[order].copy()
    w.q = w.q[rows].copy()
    w.k_new = w.k_new[rows].copy()
    w.v_new = w.v_new[rows].copy()
    w.slot_mapping = w.slot_mapping[rows].copy()
    return w
