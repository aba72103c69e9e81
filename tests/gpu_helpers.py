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


_REFERENCES = {}


def full_reference(o, w: W.Workload, key: str) -> np.ndarray:
    """The oracle's whole attention output ``[S*nq, Hq, D]`` (fp64) for one decode
    step of ``w`` (append, then attend), computed once per ``key`` in a test run."""
    ref = _REFERENCES.get(key)
    if ref is None:
        ref, _, _ = o.step(w)
        _REFERENCES[key] = ref
    return ref


def report(what: str, max_abs: float, max_rel: float, n: int):
    print(f"{what}: all {n} outputs compared, max_abs={max_abs:.3e} max_rel={max_rel:.3e}")
