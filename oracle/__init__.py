"""ctypes wrapper of the fp64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use this package. It never imports the CUDA
library, and the CUDA library never imports it.

Parity status of every function here: pinned (see the ``tests/test_oracle_*``
files: dense library attention, block-id permutation invariance, softmax weight
sums, shared prefix == copied prefix, closed forms, the block-table diagram of
"07 -- Inference" section 2.2, and the merge algebra of section 5.3; block copy:
the copy-on-write worked example of "ML Interview Prep, Lesson 13" and read-back
of every sequence's tokens through a simulated pool, in ``tests/test_block_manager_oracle.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
LIBRARY = os.path.join(_HERE, "_oracle.so")
BLOCK_SIZE = 16

_lock = threading.Lock()
_lib = None


def build(source: str = SOURCE, output: str = LIBRARY, force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, -O2, OpenMP)."""
    if (not force and os.path.exists(output)
            and os.path.getmtime(output) >= os.path.getmtime(source)):
        return output
    tmp = output + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", source, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, output)
    return output


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    lib.oracle_kv_append.argtypes = [P, P, P, i64, P, P, i64, i32, i32, i32]
    lib.oracle_kv_append.restype = ctypes.c_int
    lib.oracle_copy_blocks.argtypes = [P, P, i64, i32, i32, i32, P, P, i64]
    lib.oracle_copy_blocks.restype = ctypes.c_int
    lib.oracle_paged_attention_varlen.argtypes = [P, P, P, i64, i32, P, i32, P, i32, P, P, P,
                                                  i32, i32, i32, ctypes.c_float, P, i32]
    lib.oracle_paged_attention_varlen.restype = ctypes.c_int
    lib.oracle_e4m3_encode_array.argtypes = [P, i64, P]
    lib.oracle_e4m3_encode_array.restype = None
    lib.oracle_e4m3_decode_array.argtypes = [P, i64, P]
    lib.oracle_e4m3_decode_array.restype = None
    lib.oracle_kv_append_fp8.argtypes = [P, P, P, i64, P, P, i64, i32, i32, i32, P, P]
    lib.oracle_kv_append_fp8.restype = ctypes.c_int
    lib.oracle_paged_attention_fp8.argtypes = [P, P, P, i64, i32, P, i32, P, i32, i32, i32, i32,
                                               i32, ctypes.c_float, P, P, P, P, i32]
    lib.oracle_paged_attention_fp8.restype = ctypes.c_int
    common = [P, P, P, i64, i32, P, i32, P, i32, i32, i32, i32, i32, ctypes.c_float]
    lib.oracle_paged_attention.argtypes = common + [P, P, i32]
    lib.oracle_paged_attention.restype = ctypes.c_int
    lib.oracle_attention_weights.argtypes = common + [i32, i32, i32, P]
    lib.oracle_attention_weights.restype = ctypes.c_int
    lib.oracle_partial_state.argtypes = common + [i32, i32, i32, i32, i32, P, P, P]
    lib.oracle_partial_state.restype = ctypes.c_int
    lib.oracle_merge_states.argtypes = [i32, i32, P, P, P, P]
    lib.oracle_merge_states.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` loads another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(LIBRARY))
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """Python face of one oracle build (the default one, or a test's variant)."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def kv_append(self, k_new, v_new, slot_mapping, k_cache, v_cache):
        """Write the new tokens into (copies of) the pools; returns ``(k, v)``."""
        k_cache = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
        v_cache = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
        NB, bs, Hkv, D = k_cache.shape
        k_new = _c(k_new, np.uint16)
        v_new = _c(v_new, np.uint16)
        slots = _c(slot_mapping, np.int64)
        st = self.lib.oracle_kv_append(_ptr(k_new), _ptr(v_new), _ptr(slots), slots.size,
                                       _ptr(k_cache), _ptr(v_cache), NB, bs, Hkv, D)
        if st not in (0, -1):
            raise RuntimeError(f"oracle_kv_append failed: {st}")
        return k_cache, v_cache

    def copy_blocks(self, k_cache, v_cache, src, dst):
        """Copy whole blocks src[i] -> dst[i] in (copies of) the pools, in order."""
        k_cache = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
        v_cache = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
        NB, bs, Hkv, D = k_cache.shape
        src = _c(src, np.int32)
        dst = _c(dst, np.int32)
        if src.shape != dst.shape:
            raise ValueError("src and dst differ in length")
        st = self.lib.oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), NB, bs, Hkv, D,
                                         _ptr(src), _ptr(dst), src.size)
        if st not in (0, -1):
            raise RuntimeError(f"oracle_copy_blocks failed: {st}")
        return k_cache, v_cache

    def paged_attention_varlen(self, q, k_cache, v_cache, block_tables, context_lens, q_start,
                               scale, tree_mask=None, tree_len=None, threads: int = 0):
        """fp64 ``[q_start[-1], Hq, D]``: per-sequence query counts, causal or tree masks."""
        q = _c(q, np.uint16)
        k_cache = _c(k_cache, np.uint16)
        v_cache = _c(v_cache, np.uint16)
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        qs = _c(q_start, np.int32)
        NB, bs, Hkv, D = k_cache.shape
        S = cl.shape[0]
        Hq = q.shape[1]
        MB = bt.shape[1] if bt.ndim == 2 else 1
        assert qs.shape == (S + 1,) and q.shape[0] >= qs[-1]
        tm = tl = None
        if tree_mask is not None:
            tm = _c(tree_mask, np.uint32)
            tl = _c(tree_len, np.int32)
        out = np.zeros((int(qs[-1]), Hq, D), dtype=np.float64)
        st = self.lib.oracle_paged_attention_varlen(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), NB, bs, _ptr(bt), MB, _ptr(cl), S, _ptr(qs),
            _ptr(tm) if tm is not None else None, _ptr(tl) if tl is not None else None, Hq, Hkv,
            D, ctypes.c_float(float(np.float32(scale))), _ptr(out), int(threads))
        if st != 0:
            raise ValueError(f"oracle_paged_attention_varlen: invalid input (status {st})")
        return out

    # ---- FP8 (E4M3) KV cache
    def e4m3_encode(self, x) -> np.ndarray:
        """uint8 E4M3 codes of float32 values (nearest, ties to even, saturating)."""
        x = _c(x, np.float32)
        out = np.empty(x.shape, dtype=np.uint8)
        self.lib.oracle_e4m3_encode_array(_ptr(x), x.size, _ptr(out))
        return out

    def e4m3_decode(self, c) -> np.ndarray:
        c = _c(c, np.uint8)
        out = np.empty(c.shape, dtype=np.float64)
        self.lib.oracle_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
        return out

    def kv_append_fp8(self, k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale):
        """Quantise the new bf16 rows into (copies of) the uint8 pools."""
        k_cache = np.array(k_cache, dtype=np.uint8, copy=True, order="C")
        v_cache = np.array(v_cache, dtype=np.uint8, copy=True, order="C")
        NB, bs, Hkv, D = k_cache.shape
        k_new = _c(k_new, np.uint16)
        v_new = _c(v_new, np.uint16)
        slots = _c(slot_mapping, np.int64)
        ks = _c(k_scale, np.float32)
        vs = _c(v_scale, np.float32)
        assert ks.size == Hkv and vs.size == Hkv
        st = self.lib.oracle_kv_append_fp8(_ptr(k_new), _ptr(v_new), _ptr(slots), slots.size,
                                           _ptr(k_cache), _ptr(v_cache), NB, bs, Hkv, D,
                                           _ptr(ks), _ptr(vs))
        if st not in (0, -1):
            raise RuntimeError(f"oracle_kv_append_fp8 failed: {st}")
        return k_cache, v_cache

    def paged_attention_fp8(self, q, k_cache, v_cache, block_tables, context_lens,
                            n_query_per_seq, scale, k_scale, v_scale, pair_mask=None,
                            threads: int = 0) -> np.ndarray:
        q = _c(q, np.uint16)
        k_cache = _c(k_cache, np.uint8)
        v_cache = _c(v_cache, np.uint8)
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        ks = _c(k_scale, np.float32)
        vs = _c(v_scale, np.float32)
        NB, bs, Hkv, D = k_cache.shape
        S = cl.shape[0]
        Hq = q.shape[1]
        MB = bt.shape[1] if bt.ndim == 2 else 1
        out = np.full((S * n_query_per_seq, Hq, D), np.nan, dtype=np.float64)
        pm = None
        if pair_mask is not None:
            pm = _c(np.asarray(pair_mask).reshape(S, Hkv), np.uint8)
        st = self.lib.oracle_paged_attention_fp8(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), NB, bs, _ptr(bt), MB, _ptr(cl), S,
            int(n_query_per_seq), Hq, Hkv, D, ctypes.c_float(float(np.float32(scale))),
            _ptr(ks), _ptr(vs), _ptr(pm) if pm is not None else None, _ptr(out), int(threads))
        if st != 0:
            raise ValueError(f"oracle_paged_attention_fp8: invalid input (status {st})")
        return out

    def _common(self, q, k_cache, v_cache, block_tables, context_lens, nq, scale):
        q = _c(q, np.uint16)
        k_cache = _c(k_cache, np.uint16)
        v_cache = _c(v_cache, np.uint16)
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        NB, bs, Hkv, D = k_cache.shape
        S = cl.shape[0]
        Hq = q.shape[1]
        MB = bt.shape[1] if bt.ndim == 2 else 1
        keep = (q, k_cache, v_cache, bt, cl)
        args = [_ptr(q), _ptr(k_cache), _ptr(v_cache), NB, bs, _ptr(bt), MB, _ptr(cl), S,
                int(nq), Hq, Hkv, D, ctypes.c_float(float(np.float32(scale)))]
        return keep, args, (S, Hq, Hkv, D)

    def paged_attention(self, q, k_cache, v_cache, block_tables, context_lens, n_query_per_seq,
                        scale, pair_mask=None, threads: int = 0) -> np.ndarray:
        """fp64 ``[S*nq, Hq, D]``; rows of pairs outside ``pair_mask`` are NaN."""
        keep, args, (S, Hq, Hkv, D) = self._common(q, k_cache, v_cache, block_tables,
                                                   context_lens, n_query_per_seq, scale)
        out = np.full((S * n_query_per_seq, Hq, D), np.nan, dtype=np.float64)
        pm = None
        if pair_mask is not None:
            pm = _c(np.asarray(pair_mask).reshape(S, Hkv), np.uint8)
        st = self.lib.oracle_paged_attention(*args, _ptr(pm) if pm is not None else None,
                                             _ptr(out), int(threads))
        if st != 0:
            raise ValueError(f"oracle_paged_attention: invalid input (status {st})")
        return out

    def attention_weights(self, q, k_cache, v_cache, block_tables, context_lens,
                          n_query_per_seq, scale, s, j, qh) -> np.ndarray:
        keep, args, _ = self._common(q, k_cache, v_cache, block_tables, context_lens,
                                     n_query_per_seq, scale)
        T = int(np.asarray(context_lens)[s])
        w = np.zeros(max(T, 1), dtype=np.float64)
        n = self.lib.oracle_attention_weights(*args, int(s), int(j), int(qh), _ptr(w))
        if n < 0:
            raise ValueError("oracle_attention_weights: invalid input")
        return w[:n]

    def partial_state(self, q, k_cache, v_cache, block_tables, context_lens, n_query_per_seq,
                      scale, s, j, qh, t_begin, t_end):
        keep, args, (_, _, _, D) = self._common(q, k_cache, v_cache, block_tables,
                                                context_lens, n_query_per_seq, scale)
        m = np.zeros(1)
        l = np.zeros(1)
        acc = np.zeros(D)
        st = self.lib.oracle_partial_state(*args, int(s), int(j), int(qh), int(t_begin),
                                           int(t_end), _ptr(m), _ptr(l), _ptr(acc))
        if st != 0:
            raise ValueError("oracle_partial_state: invalid input")
        return float(m[0]), float(l[0]), acc

    def merge_states(self, m, l, acc) -> np.ndarray:
        m = _c(m, np.float64)
        l = _c(l, np.float64)
        acc = _c(acc, np.float64)
        n, D = acc.shape
        out = np.zeros(D)
        self.lib.oracle_merge_states(n, D, _ptr(m), _ptr(l), _ptr(acc), _ptr(out))
        return out

    # convenience on a workloads.Workload
    def step(self, w, pair_mask=None, threads: int = 0):
        """Append this step's tokens, then attend: returns ``(out, k_pool, v_pool)``."""
        k, v = self.kv_append(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache)
        out = self.paged_attention(w.q, k, v, w.block_tables, w.context_lens,
                                   w.n_query_per_seq, w.scale, pair_mask=pair_mask,
                                   threads=threads)
        return out, k, v


def default() -> Oracle:
    return Oracle()
