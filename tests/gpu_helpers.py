"""Shared pieces of the GPU tests: moving workloads to the device and comparing
against the fp64 oracle with the stated tolerance."""
from __future__ import annotations

import numpy as np

import paged_kv_cache_101_gb300 as pkv
import workloads as W

# Tolerance of the attention output against the fp64 oracle (bf16 inputs, fp32
# accumulation): every element within ATOL + RTOL * |ref|.
ATOL = 2e-3
RTOL = 1e-2


def bf16_dev(a: np.ndarray, torch, device="cuda"):
    """uint16 bf16 bit patterns -> a torch bfloat16 CUDA tensor (bit-exact)."""
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def bf16_host(t) -> np.ndarray:
    """torch bfloat16 tensor -> uint16 bit patterns on the host."""
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return W.bf16_bits_to_f32(bf16_host(t)).astype(np.float64)
    return t.detach().cpu().numpy().astype(np.float64)


class DeviceStep:
    """A workload's tensors on the GPU, ready for append + attention."""

    def __init__(self, w: W.Workload, torch, out_dtype=None):
        self.w = w
        self.torch = torch
        self.q = bf16_dev(w.q, torch)
        self.k_cache = bf16_dev(w.k_cache, torch)
        self.v_cache = bf16_dev(w.v_cache, torch)
        self.k_new = bf16_dev(w.k_new, torch)
        self.v_new = bf16_dev(w.v_new, torch)
        self.slots = torch.from_numpy(w.slot_mapping).cuda()
        self.tables = torch.from_numpy(w.block_tables).cuda()
        self.lens = torch.from_numpy(w.context_lens).cuda()
        od = out_dtype or torch.bfloat16
        self.out = torch.empty(self.q.shape, dtype=od, device="cuda")

    def append(self):
        pkv.kv_append(self.k_new, self.v_new, self.slots, self.k_cache, self.v_cache)

    def attend(self, ws=None):
        w = self.w
        return pkv.paged_decode_attention(self.q, self.k_cache, self.v_cache, self.tables,
                                          self.lens, w.n_query_per_seq, w.scale, self.out, ws=ws)

    def step(self):
        self.append()
        self.attend()
        return self.out


def compare(got: np.ndarray, ref: np.ndarray, atol=ATOL, rtol=RTOL, what=""):
    """Element-wise gate; returns (max_abs, max_rel over |ref| >= 1e-2)."""
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"max err {err.max():.3e}; first at {idx.tolist()}: "
                             f"got {got[tuple(idx[0])]} ref {ref[tuple(idx[0])]}")
    big = np.abs(ref) >= 1e-2
    max_rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    return float(err.max()), max_rel


def sample_pairs(w: W.Workload, n_random: int = 8, seed: int = 0) -> np.ndarray:
    """A [S, Hkv] mask of (sequence, kv head) pairs the oracle checks at full size:
    every kv head of the longest, shortest and first sequences, of two prefix
    sharers, plus random pairs."""
    S, H = w.num_seqs, w.num_kv_heads
    mask = np.zeros((S, H), dtype=bool)
    T = w.context_lens
    for s in {int(np.argmax(T)), int(np.argmin(T)), 0, S - 1}:
        mask[s, :] = True
    sharers = np.nonzero(w.shared)[0]
    for s in sharers[:2]:
        mask[s, :] = True
    rng = np.random.default_rng(seed)
    for _ in range(n_random):
        mask[rng.integers(S), rng.integers(H)] = True
    return mask


def rows_of(mask: np.ndarray, w: W.Workload):
    """Index arrays (row, q-head) of the output selected by a pair mask."""
    G = w.num_q_heads // w.num_kv_heads
    rows, heads = [], []
    for s, h in np.argwhere(mask):
        for j in range(w.n_query_per_seq):
            for g in range(G):
                rows.append(s * w.n_query_per_seq + j)
                heads.append(h * G + g)
    return np.array(rows), np.array(heads)
