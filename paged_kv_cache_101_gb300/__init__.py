"""Python binding of libpkv: paged decode attention and KV append on one GB300.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libpkv.so`` (built from ``csrc/`` for sm_103a). There is no CPU or
PyTorch fallback: if the library is missing, every call raises.

    kv_append(k_new, v_new, slot_mapping, k_cache, v_cache)
    paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens,
                           n_query_per_seq, scale, out)
    copy_blocks(k_cache, v_cache, src, dst)      # copy-on-write, on the device
    BlockManager(num_blocks)                     # host: tables, counts, forks

Tensors are torch CUDA tensors on the current device: bf16 K/V/Q laid out as
``include/pkv.h`` describes (pools ``[num_blocks, 16, num_kv_heads, head_dim]``),
int64 slot mapping, int32 block tables and context lengths. Calls are enqueued
on ``torch.cuda.current_stream()``.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK = 0
(PKV_ERR_NULL, PKV_ERR_SHAPE, PKV_ERR_DTYPE, PKV_ERR_ALIGN, PKV_ERR_RANGE, PKV_ERR_WORKSPACE,
 PKV_ERR_CUDA, PKV_ERR_UNSUPPORTED) = range(1, 9)   # pkv_status, include/pkv.h
PKV_ERR_NO_BLOCKS, PKV_ERR_SEQUENCE = 9, 10
PKV_BF16, PKV_FP32 = 0, 1
(PKV_OPT_NUM_CTAS, PKV_OPT_STAGES, PKV_OPT_HEADS_PER_CTA, PKV_OPT_TMA_BOX, PKV_OPT_TAIL,
 PKV_OPT_PACE, PKV_OPT_PACE_MARGIN, PKV_OPT_MATH, PKV_OPT_UMMA,
 PKV_OPT_PREFETCH) = 1, 2, 3, 4, 5, 6, 7, 8, 9, 10
BLOCK_SIZE = 16

# function name -> (argtypes, restype); mirrors include/pkv.h
_P, _I32, _I64, _SZ, _F = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t,
                          ctypes.c_float)
SIGNATURES = {
    "pkv_kv_append": ([_P, _P, _P, _I64, _P, _P, _I64, _I32, _I32, _P], ctypes.c_int),
    "pkv_workspace_size": ([_I32, _I32, _I32, _I32, _I32], _SZ),
    "pkv_paged_decode_attention": ([_P, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32,
                                    _F, _P, _I32, _P, _SZ, _P], ctypes.c_int),
    "pkv_step_arena_layout": ([_I32, _I32, _I32, _I32, _I32, _I32, _P], _SZ),
    "pkv_decode_step": ([_P, _P, _P, _P, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _I32, _I32,
                         _I32, _F, _P, _I32, _P, _SZ, _P, _P, _P], _I32),
    "pkv_decode_step_host": ([_P, _P, _SZ, _P, _P, _I64, _I32, _I32, _I32, _I32, _I32, _I32, _F,
                              _P, _P, _I32, _P, _SZ, _P], ctypes.c_int),
    "pkv_decode_step_host_pipelined": ([_P, _P, _SZ, _P, _P, _I64, _I32, _I32, _I32, _I32, _I32,
                                        _I32, _F, _P, _P, _I32, _P, _SZ, _P, _P, _P, _P, _P, _P,
                                        _P, _P], ctypes.c_int),
    "pkv_status_string": ([_I32], ctypes.c_char_p),
    "pkv_set_option": ([_I32, _I32], _I32),
    "pkv_version": ([], _I32),
    "pkv_set_profiling_events": ([_P, _P], None),
    "pkv_set_trace_buffer": ([_P, _SZ], None),
    "pkv_paged_decode_attention_static": ([_P, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _I32, _I32,
                                           _I32, _F, _P, _I32, _P], ctypes.c_int),
    "pkv_static_error_word": ([_P, _P], ctypes.c_int),
    "pkv_copy_blocks": ([_P, _P, _I64, _I32, _I32, _P, _P, _I32, _P], ctypes.c_int),
    "pkv_paged_decode_attention_varlen": ([_P, _P, _P, _I64, _P, _I32, _I32, _P, _P, _P, _P, _P,
                                           _I32, _I32, _I32, _I32, _I32, _I32, _F, _P, _I32, _P,
                                           _SZ, _P], ctypes.c_int),
    "pkv_workspace_size_cascade": ([_I32, _I32, _I32, _I32, _I32], _SZ),
    "pkv_paged_decode_attention_cascade": ([_P, _P, _P, _I64, _P, _I32, _P, _I32, _I32, _I32, _I32,
                                            _I32, _F, _P, _I32, _I32, _P, _I32, _P, _SZ, _P],
                                           ctypes.c_int),
    "pkv_cascade_pays": ([_P, _I32, _P, _I32, _I32, _I32], _I32),
    "pkv_split_queries": ([_P, _P, _P, _I32, _I32, _P, _P, _P, _P, _I32, _P], ctypes.c_int),
    "pkv_kv_append_fp8": ([_P, _P, _P, _I64, _P, _P, _I64, _I32, _I32, _P, _P, _P], ctypes.c_int),
    "pkv_paged_decode_attention_fp8": ([_P, _P, _P, _I64, _P, _P, _P, _I32, _P, _I32, _I32, _I32,
                                        _I32, _I32, _F, _P, _I32, _P, _SZ, _P], ctypes.c_int),
    # host block manager (include/pkv_block_manager.h)
    "pkv_bm_create": ([_I64], _P),
    "pkv_bm_destroy": ([_P], None),
    "pkv_bm_num_free": ([_P], _I64),
    "pkv_bm_num_blocks": ([_P], _I64),
    "pkv_bm_num_sequences": ([_P], _I64),
    "pkv_bm_refcount": ([_P, _I64], _I32),
    "pkv_bm_add_sequence": ([_P, _I64, _I64], ctypes.c_int),
    "pkv_bm_fork": ([_P, _I64, _I64], ctypes.c_int),
    "pkv_bm_free_sequence": ([_P, _I64], ctypes.c_int),
    "pkv_bm_append": ([_P, _P, _I32, _I32, _P, _P, _P, _P], ctypes.c_int),
    "pkv_bm_sequence_length": ([_P, _I64], _I64),
    "pkv_bm_sequence_blocks": ([_P, _I64, _P, _I64], _I64),
    "pkv_bm_block_tables": ([_P, _P, _I32, _P, _I32, _P], ctypes.c_int),
    "pkv_bm_check": ([_P], _I32),
}

_lib = None
_lib_lock = threading.Lock()


class PkvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: status {status} ({status_string(status)})")


def lib():
    """The loaded libpkv (raises if it was not built: there is no fallback)."""
    global _lib
    if _lib is None:
        with _lib_lock:
            if _lib is None:
                if not os.path.exists(LIBRARY_PATH):
                    raise RuntimeError(
                        f"{LIBRARY_PATH} is missing: build it with "
                        "`python -c 'import __graft_entry__ as g; g.build()'` "
                        "(the CUDA library is the only implementation)")
                handle = ctypes.CDLL(LIBRARY_PATH)
                for name, (argtypes, restype) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.argtypes = argtypes
                    fn.restype = restype
                _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().pkv_status_string(int(status)).decode()


def set_option(option: int, value: int) -> int:
    return int(lib().pkv_set_option(int(option), int(value)))


def set_profiling_events(before, after):
    """Record two torch.cuda.Events around the main attention kernel of later calls
    (None, None turns this off)."""
    if before is None or after is None:
        lib().pkv_set_profiling_events(None, None)
        return
    for ev in (before, after):
        if not ev.cuda_event:
            ev.record()  # torch creates the underlying event lazily
    lib().pkv_set_profiling_events(ctypes.c_void_p(before.cuda_event),
                                   ctypes.c_void_p(after.cuda_event))


def set_trace_buffer(buf):
    """Per-CTA timeline of later attention calls into a zeroed uint64 CUDA tensor
    (8 words per CTA: see include/pkv.h); None turns it off."""
    if buf is None:
        lib().pkv_set_trace_buffer(None, 0)
    else:
        lib().pkv_set_trace_buffer(ctypes.c_void_p(buf.data_ptr()),
                                   buf.numel() * buf.element_size())


def _torch():
    import torch
    return torch


def _stream_handle(device):
    torch = _torch()
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(t, name, dtype, ndim=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def kv_append(k_new, v_new, slot_mapping, k_cache, v_cache):
    """Write new K/V rows ``[n_new, Hkv, D]`` into the pools at ``slot_mapping`` (int64)."""
    torch = _torch()
    _check(k_new, "k_new", torch.bfloat16, 3)
    _check(v_new, "v_new", torch.bfloat16, 3)
    _check(slot_mapping, "slot_mapping", torch.int64, 1)
    _check(k_cache, "k_cache", torch.bfloat16, 4)
    _check(v_cache, "v_cache", torch.bfloat16, 4)
    NB, bs, Hkv, D = k_cache.shape
    if bs != BLOCK_SIZE or v_cache.shape != k_cache.shape:
        raise ValueError("pools must be [num_blocks, 16, Hkv, D] and equal in shape")
    n = slot_mapping.shape[0]
    if k_new.shape != (n, Hkv, D) or v_new.shape != (n, Hkv, D):
        raise ValueError("k_new/v_new must be [n_new, Hkv, D] matching the pool")
    st = lib().pkv_kv_append(k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(), n,
                             k_cache.data_ptr(), v_cache.data_ptr(), NB, Hkv, D,
                             _stream_handle(k_cache.device))
    if st != PKV_OK:
        raise PkvError("pkv_kv_append", st)


def paged_decode_attention_cascade(q, k_cache, v_cache, block_tables, context_lens,
                                   n_query_per_seq, scale, out, prefix_groups, max_group_seqs,
                                   ws=None):
    """``paged_decode_attention`` with shared prefixes attended once per group:
    ``prefix_groups`` is an int32 CUDA tensor [num_groups, 3] of (first sequence,
    sequences, prefix blocks), members consecutive, groups ascending."""
    torch = _torch()
    _check(q, "q", torch.bfloat16, 3)
    _check(k_cache, "k_cache", torch.bfloat16, 4)
    _check(v_cache, "v_cache", torch.bfloat16, 4)
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(context_lens, "context_lens", torch.int32, 1)
    _check(prefix_groups, "prefix_groups", torch.int32, 2)
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bfloat16 or float32")
    _check(out, "out", out.dtype, 3)
    NB, bs, Hkv, D = k_cache.shape
    if bs != BLOCK_SIZE or v_cache.shape != k_cache.shape:
        raise ValueError("pools must be [num_blocks, 16, Hkv, D] and equal in shape")
    if prefix_groups.shape[1] != 3:
        raise ValueError("prefix_groups must be [num_groups, 3]")
    S = context_lens.shape[0]
    nq = int(n_query_per_seq)
    Hq = q.shape[1]
    if q.shape != (S * nq, Hq, D) or out.shape != q.shape or block_tables.shape[0] != S:
        raise ValueError("q/out must be [num_seqs * n_query_per_seq, Hq, D], tables [num_seqs, MB]")
    need = int(lib().pkv_workspace_size_cascade(S, nq, Hq, Hkv, D))
    if ws is None:
        ws = workspace(q.device, need)
    st = lib().pkv_paged_decode_attention_cascade(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), NB, block_tables.data_ptr(),
        block_tables.shape[1], context_lens.data_ptr(), S, nq, Hq, Hkv, D, float(scale),
        prefix_groups.data_ptr(), prefix_groups.shape[0], int(max_group_seqs), out.data_ptr(),
        PKV_FP32 if out.dtype == torch.float32 else PKV_BF16, ws.data_ptr(), ws.numel(),
        _stream_handle(q.device))
    if st != PKV_OK:
        raise PkvError("pkv_paged_decode_attention_cascade", st)
    return out


def split_queries(q_start, context_lens, max_rows, tree_len=None):
    """Host: cut query runs into virtual sequences of at most ``max_rows`` rows
    (see pkv_split_queries). Returns a dict of int32 numpy arrays: q_start
    [V+1], context_lens [V], table_row [V] and, with tree_len, tree_len [V]."""
    import numpy as np
    qs = np.ascontiguousarray(q_start, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    S = cl.size
    tl = None if tree_len is None else np.ascontiguousarray(tree_len, dtype=np.int32)
    nv = ctypes.c_int32(0)
    st = lib().pkv_split_queries(qs.ctypes.data, cl.ctypes.data,
                                 tl.ctypes.data if tl is not None else None, S, int(max_rows),
                                 None, None, None, None, 0, ctypes.byref(nv))
    cap = nv.value
    if st not in (PKV_OK, 5):
        raise PkvError("pkv_split_queries", st)
    vq = np.zeros(cap + 1, np.int32)
    vc = np.zeros(max(cap, 1), np.int32)
    vt = np.zeros(max(cap, 1), np.int32)
    vr = np.zeros(max(cap, 1), np.int32)
    st = lib().pkv_split_queries(qs.ctypes.data, cl.ctypes.data,
                                 tl.ctypes.data if tl is not None else None, S, int(max_rows),
                                 vq.ctypes.data, vc.ctypes.data, vt.ctypes.data, vr.ctypes.data,
                                 cap, ctypes.byref(nv))
    if st != PKV_OK:
        raise PkvError("pkv_split_queries", st)
    V = nv.value
    out = dict(q_start=vq[:V + 1] if V else np.zeros(1, np.int32), context_lens=vc[:V],
               table_row=vr[:V])
    if tl is not None:
        out["tree_len"] = vt[:V]
    return out


def paged_decode_attention_varlen(q, k_cache, v_cache, block_tables, context_lens, q_start,
                                  max_q_len, scale, out, tree_mask=None, tree_len=None,
                                  table_row=None, ws=None):
    """Decode attention with per-sequence query counts (rows q_start[s] ..
    q_start[s+1]-1 of q/out), optional tree masks (uint32 per row, with int32
    windows tree_len) and optional block-table rows (table_row)."""
    torch = _torch()
    _check(q, "q", torch.bfloat16, 3)
    _check(k_cache, "k_cache", torch.bfloat16, 4)
    _check(v_cache, "v_cache", torch.bfloat16, 4)
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(context_lens, "context_lens", torch.int32, 1)
    _check(q_start, "q_start", torch.int32, 1)
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bfloat16 or float32")
    _check(out, "out", out.dtype, 3)
    NB, bs, Hkv, D = k_cache.shape
    if bs != BLOCK_SIZE or v_cache.shape != k_cache.shape:
        raise ValueError("pools must be [num_blocks, 16, Hkv, D] and equal in shape")
    S = context_lens.shape[0]
    if q_start.shape[0] != S + 1 or out.shape != q.shape or q.shape[2] != D:
        raise ValueError("q_start must have num_seqs + 1 entries; q and out [total_q, Hq, D]")
    if (tree_mask is None) != (tree_len is None):
        raise ValueError("tree_mask and tree_len come together")
    if tree_mask is not None:
        _check(tree_mask, "tree_mask", torch.int32, 1)   # uint32 bits stored as int32
        _check(tree_len, "tree_len", torch.int32, 1)
    if table_row is not None:
        _check(table_row, "table_row", torch.int32, 1)
    total_q, Hq = q.shape[0], q.shape[1]
    need = workspace_size(S, int(max_q_len), Hq, Hkv, D)
    if ws is None:
        ws = workspace(q.device, need)
    st = lib().pkv_paged_decode_attention_varlen(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), NB, block_tables.data_ptr(),
        block_tables.shape[1], block_tables.shape[0],
        table_row.data_ptr() if table_row is not None else None, context_lens.data_ptr(),
        q_start.data_ptr(), tree_mask.data_ptr() if tree_mask is not None else None,
        tree_len.data_ptr() if tree_len is not None else None, S, int(max_q_len), total_q, Hq,
        Hkv, D, float(scale), out.data_ptr(),
        PKV_FP32 if out.dtype == torch.float32 else PKV_BF16, ws.data_ptr(), ws.numel(),
        _stream_handle(q.device))
    if st != PKV_OK:
        raise PkvError("pkv_paged_decode_attention_varlen", st)
    return out


def _check_fp8_pools(k_cache, v_cache, k_scale, v_scale):
    torch = _torch()
    _check(k_cache, "k_cache", torch.uint8, 4)
    _check(v_cache, "v_cache", torch.uint8, 4)
    _check(k_scale, "k_scale", torch.float32, 1)
    _check(v_scale, "v_scale", torch.float32, 1)
    NB, bs, Hkv, D = k_cache.shape
    if bs != BLOCK_SIZE or v_cache.shape != k_cache.shape:
        raise ValueError("pools must be [num_blocks, 16, Hkv, D] and equal in shape")
    if k_scale.shape != (Hkv,) or v_scale.shape != (Hkv,):
        raise ValueError("k_scale / v_scale must hold one float per kv head")
    return NB, Hkv, D


def kv_append_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale):
    """Quantise bf16 rows ``[n_new, Hkv, D]`` into E4M3 (uint8) pools with per-head scales."""
    torch = _torch()
    _check(k_new, "k_new", torch.bfloat16, 3)
    _check(v_new, "v_new", torch.bfloat16, 3)
    _check(slot_mapping, "slot_mapping", torch.int64, 1)
    NB, Hkv, D = _check_fp8_pools(k_cache, v_cache, k_scale, v_scale)
    n = slot_mapping.shape[0]
    if k_new.shape != (n, Hkv, D) or v_new.shape != (n, Hkv, D):
        raise ValueError("k_new/v_new must be [n_new, Hkv, D] matching the pool")
    st = lib().pkv_kv_append_fp8(k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(), n,
                                 k_cache.data_ptr(), v_cache.data_ptr(), NB, Hkv, D,
                                 k_scale.data_ptr(), v_scale.data_ptr(),
                                 _stream_handle(k_cache.device))
    if st != PKV_OK:
        raise PkvError("pkv_kv_append_fp8", st)


def paged_decode_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables,
                               context_lens, n_query_per_seq, scale, out, ws=None):
    """Decode attention over E4M3 (uint8) pools with per-head scales; writes ``out``."""
    torch = _torch()
    _check(q, "q", torch.bfloat16, 3)
    NB, Hkv, D = _check_fp8_pools(k_cache, v_cache, k_scale, v_scale)
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(context_lens, "context_lens", torch.int32, 1)
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bfloat16 or float32")
    _check(out, "out", out.dtype, 3)
    S = context_lens.shape[0]
    nq = int(n_query_per_seq)
    Hq = q.shape[1]
    if q.shape != (S * nq, Hq, D) or out.shape != q.shape or block_tables.shape[0] != S:
        raise ValueError("q/out must be [num_seqs * n_query_per_seq, Hq, D], tables [num_seqs, MB]")
    need = workspace_size(S, nq, Hq, Hkv, D)
    if ws is None:
        ws = workspace(q.device, need)
    st = lib().pkv_paged_decode_attention_fp8(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), NB, k_scale.data_ptr(),
        v_scale.data_ptr(), block_tables.data_ptr(), block_tables.shape[1],
        context_lens.data_ptr(), S, nq, Hq, Hkv, D, float(scale), out.data_ptr(),
        PKV_FP32 if out.dtype == torch.float32 else PKV_BF16, ws.data_ptr(), ws.numel(),
        _stream_handle(q.device))
    if st != PKV_OK:
        raise PkvError("pkv_paged_decode_attention_fp8", st)
    return out


def copy_blocks(k_cache, v_cache, src, dst):
    """Copy whole blocks ``src[i] -> dst[i]`` (int32 CUDA tensors) in both pools."""
    torch = _torch()
    _check(k_cache, "k_cache", torch.bfloat16, 4)
    _check(v_cache, "v_cache", torch.bfloat16, 4)
    _check(src, "src", torch.int32, 1)
    _check(dst, "dst", torch.int32, 1)
    NB, bs, Hkv, D = k_cache.shape
    if bs != BLOCK_SIZE or v_cache.shape != k_cache.shape:
        raise ValueError("pools must be [num_blocks, 16, Hkv, D] and equal in shape")
    if src.shape != dst.shape:
        raise ValueError("src and dst must have the same length")
    st = lib().pkv_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), NB, Hkv, D,
                               src.data_ptr(), dst.data_ptr(), src.shape[0],
                               _stream_handle(k_cache.device))
    if st != PKV_OK:
        raise PkvError("pkv_copy_blocks", st)


class BlockManager:
    """Host-side block manager of a pool (free list, block tables, reference
    counts, forks, copy-on-write); a thin face of ``pkv_bm_*``."""

    def __init__(self, num_blocks: int):
        self._h = lib().pkv_bm_create(int(num_blocks))
        if not self._h:
            raise PkvError("pkv_bm_create", 2)
        self.num_blocks = int(num_blocks)

    def close(self):
        if self._h:
            lib().pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _call(self, name, *args):
        st = getattr(lib(), name)(self._h, *args)
        if st != PKV_OK:
            raise PkvError(name, st)

    def num_free(self) -> int:
        return int(lib().pkv_bm_num_free(self._h))

    def num_sequences(self) -> int:
        return int(lib().pkv_bm_num_sequences(self._h))

    def ref(self, block: int) -> int:
        return int(lib().pkv_bm_refcount(self._h, int(block)))

    def add_sequence(self, seq: int, n_tokens: int) -> bool:
        """False when the free blocks do not suffice (nothing changes)."""
        st = lib().pkv_bm_add_sequence(self._h, int(seq), int(n_tokens))
        if st == PKV_ERR_NO_BLOCKS:
            return False
        if st != PKV_OK:
            raise PkvError("pkv_bm_add_sequence", st)
        return True

    def fork(self, parent: int, child: int) -> None:
        self._call("pkv_bm_fork", int(parent), int(child))

    def free(self, seq: int) -> None:
        self._call("pkv_bm_free_sequence", int(seq))

    def append_batch(self, seqs, n_per_seq: int = 1):
        """``(slots, copies)`` for n tokens of each sequence, or None (no change)
        when the free blocks do not suffice; slots is an int64 array, copies a
        list of (src, dst) block pairs."""
        import numpy as np
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        k = ids.size
        slots = np.empty(k * int(n_per_seq), dtype=np.int64)
        src = np.empty(max(k, 1), dtype=np.int32)
        dst = np.empty(max(k, 1), dtype=np.int32)
        nc = ctypes.c_int32(0)
        st = lib().pkv_bm_append(self._h, ids.ctypes.data, k, int(n_per_seq), slots.ctypes.data,
                                 src.ctypes.data, dst.ctypes.data, ctypes.byref(nc))
        if st == PKV_ERR_NO_BLOCKS:
            return None
        if st != PKV_OK:
            raise PkvError("pkv_bm_append", st)
        return slots, [(int(src[i]), int(dst[i])) for i in range(nc.value)]

    def length(self, seq: int) -> int:
        n = int(lib().pkv_bm_sequence_length(self._h, int(seq)))
        if n < 0:
            raise PkvError("pkv_bm_sequence_length", PKV_ERR_SEQUENCE)
        return n

    def table(self, seq: int) -> list:
        import numpy as np
        n = int(lib().pkv_bm_sequence_blocks(self._h, int(seq), None, 0))
        if n < 0:
            raise PkvError("pkv_bm_sequence_blocks", PKV_ERR_SEQUENCE)
        out = np.empty(max(n, 1), dtype=np.int32)
        lib().pkv_bm_sequence_blocks(self._h, int(seq), out.ctypes.data, n)
        return [int(b) for b in out[:n]]

    def block_tables(self, seqs, max_blocks_per_seq: int):
        """int32 ``[len(seqs), max_blocks_per_seq]`` (padded with -1) and int32 lengths."""
        import numpy as np
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        tables = np.empty((ids.size, max(int(max_blocks_per_seq), 1)), dtype=np.int32)
        lens = np.empty(max(ids.size, 1), dtype=np.int32)
        self._call("pkv_bm_block_tables", ids.ctypes.data, ids.size, tables.ctypes.data,
                   int(max_blocks_per_seq), lens.ctypes.data)
        return tables[:, :int(max_blocks_per_seq)], lens[:ids.size]

    def check(self) -> int:
        """0 when the manager's own state is consistent (see pkv_bm_check)."""
        return int(lib().pkv_bm_check(self._h))


def workspace_size(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads, head_dim) -> int:
    return int(lib().pkv_workspace_size(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads,
                                        head_dim))


_workspaces = {}


def workspace(device, nbytes: int):
    """A cached, zero-initialised workspace of at least ``nbytes`` on ``device``."""
    torch = _torch()
    key = torch.device(device).index if torch.device(device).index is not None else \
        torch.cuda.current_device()
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def workspace_error(ws) -> int:
    """The device error word at the start of a workspace (0 = no bounded wait gave up)."""
    return int(ws[:4].view(_torch().int32).item())


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, n_query_per_seq,
                           scale, out, ws=None):
    """Decode attention over the paged pools; writes ``out`` (bf16 or fp32)."""
    torch = _torch()
    _check(q, "q", torch.bfloat16, 3)
    _check(k_cache, "k_cache", torch.bfloat16, 4)
    _check(v_cache, "v_cache", torch.bfloat16, 4)
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(context_lens, "context_lens", torch.int32, 1)
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bfloat16 or float32")
    _check(out, "out", out.dtype, 3)
    NB, bs, Hkv, D = k_cache.shape
    if bs != BLOCK_SIZE or v_cache.shape != k_cache.shape:
        raise ValueError("pools must be [num_blocks, 16, Hkv, D] and equal in shape")
    S = context_lens.shape[0]
    nq = int(n_query_per_seq)
    Hq = q.shape[1]
    if q.shape != (S * nq, Hq, D) or out.shape != q.shape:
        raise ValueError("q and out must be [num_seqs * n_query_per_seq, Hq, D]")
    if block_tables.shape[0] != S:
        raise ValueError("block_tables must have num_seqs rows")
    need = workspace_size(S, nq, Hq, Hkv, D)
    if ws is None:
        ws = workspace(q.device, need)
    st = lib().pkv_paged_decode_attention(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), NB, block_tables.data_ptr(),
        block_tables.shape[1], context_lens.data_ptr(), S, nq, Hq, Hkv, D, float(scale),
        out.data_ptr(), PKV_FP32 if out.dtype == torch.float32 else PKV_BF16, ws.data_ptr(),
        ws.numel(), _stream_handle(q.device))
    if st != PKV_OK:
        raise PkvError("pkv_paged_decode_attention", st)
    return out


def decode_step(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables, context_lens,
                n_query_per_seq, scale, out, ws=None, k_scale=None, v_scale=None):
    """One decode step in one call: append the new rows ``[S * nq, Hkv, D]`` at
    ``slot_mapping``, then attend (bf16 pools; E4M3 uint8 pools with ``k_scale`` and
    ``v_scale``). Same results as ``kv_append`` then ``paged_decode_attention``; the
    attention kernel plans its work while the append runs."""
    torch = _torch()
    _check(q, "q", torch.bfloat16, 3)
    _check(k_new, "k_new", torch.bfloat16, 3)
    _check(v_new, "v_new", torch.bfloat16, 3)
    _check(slot_mapping, "slot_mapping", torch.int64, 1)
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(context_lens, "context_lens", torch.int32, 1)
    if (k_scale is None) != (v_scale is None):
        raise ValueError("give both scales (E4M3 pools) or neither (bf16 pools)")
    if k_scale is not None:
        NB, Hkv, D = _check_fp8_pools(k_cache, v_cache, k_scale, v_scale)
    else:
        _check(k_cache, "k_cache", torch.bfloat16, 4)
        _check(v_cache, "v_cache", torch.bfloat16, 4)
        NB, bs, Hkv, D = k_cache.shape
        if bs != BLOCK_SIZE or v_cache.shape != k_cache.shape:
            raise ValueError("pools must be [num_blocks, 16, Hkv, D] and equal in shape")
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bfloat16 or float32")
    _check(out, "out", out.dtype, 3)
    S = context_lens.shape[0]
    nq = int(n_query_per_seq)
    Hq = q.shape[1]
    if q.shape != (S * nq, Hq, D) or out.shape != q.shape or block_tables.shape[0] != S:
        raise ValueError("q/out must be [num_seqs * n_query_per_seq, Hq, D], tables [num_seqs, MB]")
    if (k_new.shape != (S * nq, Hkv, D) or v_new.shape != k_new.shape
            or slot_mapping.shape[0] != S * nq):
        raise ValueError("k_new/v_new must be [num_seqs * n_query_per_seq, Hkv, D] with one slot "
                         "per row")
    need = workspace_size(S, nq, Hq, Hkv, D)
    if ws is None:
        ws = workspace(q.device, need)
    st = lib().pkv_decode_step(
        q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(),
        k_cache.data_ptr(), v_cache.data_ptr(), NB, block_tables.data_ptr(),
        block_tables.shape[1], context_lens.data_ptr(), S, nq, Hq, Hkv, D, float(scale),
        out.data_ptr(), PKV_FP32 if out.dtype == torch.float32 else PKV_BF16, ws.data_ptr(),
        ws.numel(), None if k_scale is None else k_scale.data_ptr(),
        None if v_scale is None else v_scale.data_ptr(), _stream_handle(q.device))
    if st != PKV_OK:
        raise PkvError("pkv_decode_step", st)
    return out


def paged_decode_attention_static(q, k_cache, v_cache, block_tables, context_lens,
                                  n_query_per_seq, scale, out):
    """``paged_decode_attention`` for callers that cannot allocate device memory: the
    scratch is the library's static 32 MiB device array, shared by every call (so
    calls must not overlap on the GPU)."""
    torch = _torch()
    _check(q, "q", torch.bfloat16, 3)
    _check(k_cache, "k_cache", torch.bfloat16, 4)
    _check(v_cache, "v_cache", torch.bfloat16, 4)
    _check(block_tables, "block_tables", torch.int32, 2)
    _check(context_lens, "context_lens", torch.int32, 1)
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bfloat16 or float32")
    _check(out, "out", out.dtype, 3)
    NB, bs, Hkv, D = k_cache.shape
    S = context_lens.shape[0]
    nq = int(n_query_per_seq)
    Hq = q.shape[1]
    if bs != BLOCK_SIZE or v_cache.shape != k_cache.shape:
        raise ValueError("pools must be [num_blocks, 16, Hkv, D] and equal in shape")
    if q.shape != (S * nq, Hq, D) or out.shape != q.shape or block_tables.shape[0] != S:
        raise ValueError("q/out must be [num_seqs * n_query_per_seq, Hq, D], tables [num_seqs, MB]")
    st = lib().pkv_paged_decode_attention_static(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), NB, block_tables.data_ptr(),
        block_tables.shape[1], context_lens.data_ptr(), S, nq, Hq, Hkv, D, float(scale),
        out.data_ptr(), PKV_FP32 if out.dtype == torch.float32 else PKV_BF16,
        _stream_handle(q.device))
    if st != PKV_OK:
        raise PkvError("pkv_paged_decode_attention_static", st)
    return out


def cascade_pays(context_lens, prefix_groups, num_kv_heads, head_dim) -> bool:
    """The library's rule for choosing the shared-prefix cascade over the plain call
    (host arrays: context lengths [S], groups [num_groups][3]; the pools' kv heads
    and head dim)."""
    import numpy as np
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    groups = np.ascontiguousarray(prefix_groups, dtype=np.int32).reshape(-1, 3)
    r = lib().pkv_cascade_pays(lens.ctypes.data, lens.size, groups.ctypes.data,
                               groups.shape[0], int(num_kv_heads), int(head_dim))
    if r < 0:
        raise ValueError("pkv_cascade_pays: invalid input")
    return bool(r)


def static_error_word(device=None) -> int:
    """The device error word of the static scratch (``paged_decode_attention_static``)
    on ``device``, read after the current stream's work."""
    torch = _torch()
    dev = torch.device(device) if device is not None else torch.device(
        "cuda", torch.cuda.current_device())
    word = ctypes.c_uint32(0)
    with torch.cuda.device(dev):
        st = lib().pkv_static_error_word(ctypes.addressof(word), _stream_handle(dev))
    if st != PKV_OK:
        raise PkvError("pkv_static_error_word", st)
    return int(word.value)


def step_arena_layout(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads, head_dim,
                      max_blocks_per_seq):
    """(total bytes, {name: byte offset}) of one decode step's inputs packed in one
    buffer (q, k_new, v_new, slot_mapping, block_tables, context_lens)."""
    offs = (ctypes.c_size_t * 6)()
    n = lib().pkv_step_arena_layout(num_seqs, n_query_per_seq, num_q_heads, num_kv_heads,
                                    head_dim, max_blocks_per_seq, offs)
    if n == 0:
        raise PkvError("pkv_step_arena_layout", PKV_ERR_UNSUPPORTED)
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    return int(n), dict(zip(names, (int(o) for o in offs)))


def decode_step_host(host_arena, device_arena, k_cache, v_cache, num_seqs, n_query_per_seq,
                     num_q_heads, max_blocks_per_seq, scale, out_device, out_host, ws=None,
                     streams=None, events=None, k_scale=None, v_scale=None):
    """One decode step from host memory (``pkv_decode_step_host``): one copy of the
    packed inputs to ``device_arena``, the KV append, the attention into
    ``out_device``, one copy of the output to ``out_host``; asynchronous on the
    current stream. ``host_arena``/``out_host`` are (pinned) CPU tensors.

    With ``streams = (upload, compute, download)`` (torch CUDA streams) and
    ``events = (uploaded, computed, downloaded)`` (torch CUDA events of this
    buffer slot), it calls ``pkv_decode_step_host_pipelined`` instead: the copies
    and the kernels go on their own streams, ordered by the slot's events, so a
    loop that alternates two slots overlaps copies with kernels. Events that were
    never recorded are recorded once on the compute stream first (torch creates
    them lazily). ``k_scale``/``v_scale`` (float32 ``[Hkv]``) mark E4M3 (uint8)
    pools; they need the pipelined form."""
    torch = _torch()
    fp8 = k_scale is not None or v_scale is not None
    if fp8:
        if streams is None:
            raise ValueError("E4M3 pools (k_scale/v_scale) take the pipelined form: pass streams")
        _check_fp8_pools(k_cache, v_cache, k_scale, v_scale)
    else:
        _check(k_cache, "k_cache", torch.bfloat16, 4)
        _check(v_cache, "v_cache", torch.bfloat16, 4)
    if host_arena.device.type != "cpu" or out_host.device.type != "cpu":
        raise ValueError("host_arena and out_host must be host tensors")
    if device_arena.device.type != "cuda" or not device_arena.is_contiguous():
        raise ValueError("device_arena must be a contiguous CUDA tensor")
    if not host_arena.is_contiguous() or not out_host.is_contiguous():
        raise ValueError("host buffers must be contiguous")
    if out_device.dtype not in (torch.bfloat16, torch.float32) or out_host.dtype != out_device.dtype:
        raise TypeError("out_device/out_host must both be bfloat16 or both float32")
    NB, bs, Hkv, D = k_cache.shape
    if bs != BLOCK_SIZE or v_cache.shape != k_cache.shape:
        raise ValueError("pools must be [num_blocks, 16, Hkv, D] and equal in shape")
    nbytes = min(host_arena.numel() * host_arena.element_size(),
                 device_arena.numel() * device_arena.element_size())
    if out_host.numel() != out_device.numel():
        raise ValueError("out_host and out_device differ in size")
    if ws is None:
        ws = workspace(k_cache.device, workspace_size(num_seqs, n_query_per_seq, num_q_heads,
                                                      Hkv, D))
    odt = PKV_FP32 if out_device.dtype == torch.float32 else PKV_BF16
    if streams is None:
        st = lib().pkv_decode_step_host(
            host_arena.data_ptr(), device_arena.data_ptr(), nbytes, k_cache.data_ptr(),
            v_cache.data_ptr(), NB, max_blocks_per_seq, num_seqs, n_query_per_seq, num_q_heads,
            Hkv, D, float(scale), out_device.data_ptr(), out_host.data_ptr(), odt, ws.data_ptr(),
            ws.numel(), _stream_handle(k_cache.device))
        if st != PKV_OK:
            raise PkvError("pkv_decode_step_host", st)
        return out_host
    if events is None or len(streams) != 3 or len(events) != 3:
        raise ValueError("streams and events: three of each (upload, compute, download)")
    for ev in events:
        if not ev.cuda_event:
            ev.record(streams[1])
    st = lib().pkv_decode_step_host_pipelined(
        host_arena.data_ptr(), device_arena.data_ptr(), nbytes, k_cache.data_ptr(),
        v_cache.data_ptr(), NB, max_blocks_per_seq, num_seqs, n_query_per_seq, num_q_heads, Hkv,
        D, float(scale), out_device.data_ptr(), out_host.data_ptr(), odt, ws.data_ptr(),
        ws.numel(), k_scale.data_ptr() if fp8 else None, v_scale.data_ptr() if fp8 else None,
        *[s.cuda_stream for s in streams], *[ev.cuda_event for ev in events])
    if st != PKV_OK:
        raise PkvError("pkv_decode_step_host_pipelined", st)
    return out_host
