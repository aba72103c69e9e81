"""Byte/FLOP counting used by the benchmark, against the pages' worked numbers."""
import json
import math
import os

import numpy as np
import pytest

import workloads as W
from paged_kv_cache_101_gb300 import roofline as R

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "kv_bytes.json")))


@pytest.mark.parametrize("case", G["bytes_per_token"], ids=lambda c: c["model"])
def test_bytes_per_token(case):
    assert R.kv_bytes_per_token(case["layers"], case["kv_heads"], case["head_dim"]) == case["bytes"]


@pytest.mark.parametrize("case", G["bytes_per_block"], ids=lambda c: str(c["bytes"]))
def test_bytes_per_block(case):
    got = R.bytes_per_block(case["block_size"], case["layers"], case["kv_heads"], case["head_dim"])
    assert got == case["bytes"]


def test_prefix_bytes():
    for c in G["prefix_bytes"]:
        assert c["tokens"] * R.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"]) == c["bytes"]


def test_blocks_and_waste():
    for c in G["blocks_for_tokens"]:
        assert R.blocks_for_tokens(c["tokens"], c["block_size"]) == c["blocks"]
        if "last_block_tokens" in c:
            assert c["tokens"] - (c["blocks"] - 1) * c["block_size"] == c["last_block_tokens"]
    for n in range(1, 200):
        assert 0 <= R.waste_tokens(n) <= 15


def test_context_bytes():
    for c in G["context_bytes"]:
        gib = c["per_token_bytes"] * c["tokens"] / 2**30
        if "gib" in c:
            assert gib == c["gib"]
        else:
            assert round(gib, 1) == c["gib_rounded_1dp"]


def test_attention_bytes_by_enumeration():
    """Count the bytes of a small workload one element at a time."""
    sh = np.array([True, False, True])
    w = W.make_custom(3, 2, 8, 2, 64, [40, 19, 70], seed=3, shared=sh, prefix_tokens=32)
    kv_logical = kv_unique = 0
    seen = set()
    entries_logical = 0
    for s in range(3):
        T = int(w.context_lens[s])
        for t in range(T):
            kv_logical += 2 * 2 * 64 * 2            # K and V, 2 heads, 64 dims, 2 bytes
            key = (int(w.block_tables[s, t // 16]), t % 16)
            if key not in seen:
                seen.add(key)
                kv_unique += 2 * 2 * 64 * 2
        entries_logical += math.ceil(T / 16)
    qo = 2 * (3 * 2 * 8 * 64 * 2)
    logical = kv_logical + qo + entries_logical * 4 + 3 * 4
    assert R.workload_bytes(w, unique=False) == logical
    unique_entries = w.unique_blocks()
    assert R.workload_bytes(w, unique=True) == kv_unique + qo + unique_entries * 4 + 3 * 4


def test_intensity_theorem():
    """KV-only intensity of decode attention is n_h / n_kv FLOP per byte (bf16)."""
    for Hq, Hkv in ((32, 32), (32, 8), (64, 8)):
        T = [4096, 8192]
        flops = R.attention_flops(T, 1, Hq, 128)
        kv = sum(T) * Hkv * 128 * 2 * 2
        assert flops / kv == pytest.approx(Hq / Hkv, rel=1e-3)
