"""Byte and FLOP counts of paged decode attention and the KV append.

Pure arithmetic on shapes; used by the benchmark to turn a measured time into
GB/s and a roofline fraction.

* KV bytes per token: ``2 * layers * kv_heads * head_dim * bytes_per_element``
  (the 2 is K and V) -- "07 -- Inference" section 2.1; "ML Interview Prep,
  Lesson 13" section 3.2.
* Bytes per block: ``block_size`` times that ("Chapter 18", section 18.2.2).
* Blocks for ``n`` tokens: ``ceil(n / block_size)``; the waste is under one
  block ("ML Interview Prep, Lesson 13", section 3.5, waste bound).
* Decode attention: ``4 t d_h n_h`` FLOPs against ``2 t d_h n_kv b`` bytes, an
  intensity of ``n_h / n_kv`` FLOP/byte in bf16 ("ML Interview Prep, Lesson
  13", section 3.3 theorem, steps 4-6).

The algorithmic bytes of one attention call are those the method cannot avoid:
Q, the visible K and V, the block-table entries in use and the context lengths
read, plus the output written. With a shared prefix, ``unique=True`` counts the
shared blocks' tokens once (they need to leave HBM only once, "Chapter 18"
section 18.2.2: sharers read the same physical blocks).
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

BLOCK_SIZE = 16


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_element: int = 2) -> int:
    return 2 * layers * kv_heads * head_dim * bytes_per_element


def bytes_per_block(block_size: int, layers: int, kv_heads: int, head_dim: int,
                    bytes_per_element: int = 2) -> int:
    return block_size * kv_bytes_per_token(layers, kv_heads, head_dim, bytes_per_element)


def blocks_for_tokens(n: int, block_size: int = BLOCK_SIZE) -> int:
    return -(-int(n) // block_size)


def waste_tokens(n: int, block_size: int = BLOCK_SIZE) -> int:
    return block_size * blocks_for_tokens(n, block_size) - int(n)


def attention_bytes(context_lens: Sequence[int], n_query_per_seq: int, num_q_heads: int,
                    num_kv_heads: int, head_dim: int, out_bytes_per_element: int = 2,
                    shared_prefix_tokens: int = 0, n_sharers: int = 0,
                    unique: bool = False, kv_bytes_per_element: int = 2) -> int:
    """Algorithmic bytes of one ``paged_decode_attention`` call (bf16 Q and output;
    K/V elements of ``kv_bytes_per_element``: 2 for bf16, 1 for E4M3 pools, whose
    per-head scales add 8 bytes per kv head)."""
    T = np.asarray(context_lens, dtype=np.int64)
    S = int(T.size)
    tokens = int(T.sum())
    if unique and n_sharers > 1:
        tokens -= (n_sharers - 1) * int(shared_prefix_tokens)
    kv = tokens * num_kv_heads * head_dim * 2 * kv_bytes_per_element
    if kv_bytes_per_element == 1:
        kv += num_kv_heads * 8
    q = S * n_query_per_seq * num_q_heads * head_dim * 2
    out = S * n_query_per_seq * num_q_heads * head_dim * out_bytes_per_element
    table_entries = int(((T + BLOCK_SIZE - 1) // BLOCK_SIZE).sum())
    if unique and n_sharers > 1:
        table_entries -= (n_sharers - 1) * (int(shared_prefix_tokens) // BLOCK_SIZE)
    tables = table_entries * 4 + S * 4
    return kv + q + out + tables


def append_bytes(n_new: int, num_kv_heads: int, head_dim: int, kv_bytes_per_element: int = 2) -> int:
    """K and V of the new tokens read once (bf16) and written once (at the pool's
    element size), plus the slot ids."""
    return n_new * num_kv_heads * head_dim * 2 * (2 + kv_bytes_per_element) + n_new * 8


def attention_flops(context_lens: Sequence[int], n_query_per_seq: int, num_q_heads: int,
                    head_dim: int) -> int:
    """``4 * head_dim`` FLOPs per (query row, visible token) pair."""
    T = np.asarray(context_lens, dtype=np.int64)
    nq = n_query_per_seq
    visible = 0
    for j in range(nq):
        visible += int(np.maximum(T - nq + j + 1, 0).sum())
    return 4 * head_dim * num_q_heads * visible


def workload_bytes(w, unique: bool = True, out_bytes_per_element: int = 2,
                   kv_bytes_per_element: int = 2) -> int:
    """``attention_bytes`` of a ``workloads.Workload``."""
    n_sh = int(np.asarray(w.shared).sum())
    return attention_bytes(w.context_lens, w.n_query_per_seq, w.num_q_heads, w.num_kv_heads,
                           w.head_dim, out_bytes_per_element,
                           shared_prefix_tokens=w.meta.get("prefix_tokens", 0),
                           n_sharers=n_sh, unique=unique,
                           kv_bytes_per_element=kv_bytes_per_element)
