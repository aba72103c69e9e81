"""The samples the bench times the oracle on (CPU baseline and reference arm).

- A sample of the first sequences carries only the pool blocks they use: the oracle's
  step on it equals, bit for bit, its step on the same sequences over the whole pool.
- A token-budget sample cuts its last sequence to a shorter context with the new
  tokens at that context's end (their slots come from the block table), and stays a
  valid decode step.
- The reference arm's run time is bounded for any step count (a tiny workload here).
"""
import copy
import os
import sys

import numpy as np
import pytest

import oracle
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


def first_sequences(w, keep):
    """The same sequences over the whole pool (no compaction)."""
    w = copy.deepcopy(w)
    nq = w.n_query_per_seq
    w.context_lens = w.context_lens[:keep].copy()
    w.block_tables = w.block_tables[:keep].copy()
    for f in ("q", "k_new", "v_new", "slot_mapping"):
        setattr(w, f, getattr(w, f)[:keep * nq].copy())
    w.shared = w.shared[:keep].copy()
    w.num_seqs = keep
    return w


def test_compact_pool_gives_the_same_step(o):
    full = W.make_workload("llama3_70b_mix")           # sharers: a shared prefix in the pool
    s, desc = bench.sample_workload("llama3_70b_mix", 6, w=copy.deepcopy(full))
    assert s.num_blocks < full.num_blocks and desc == "first 6 of 256 sequences"
    ref = first_sequences(full, 6)
    a, ka, va = o.step(s)
    b, _, _ = o.step(ref)
    assert np.array_equal(a, b)
    # the appended rows land in the compacted pool where the tables point
    nq = s.n_query_per_seq
    for i in range(s.num_seqs):
        T = int(s.context_lens[i])
        for j in range(nq):
            pos = T - nq + j
            slot = int(s.block_tables[i, pos // 16]) * 16 + pos % 16
            assert int(s.slot_mapping[i * nq + j]) == slot


def test_token_budget_cuts_the_last_sequence(o):
    full = W.make_workload("spec_verify")
    budget = int(full.context_lens[0]) + 700
    s, desc = bench.sample_workload("spec_verify", 16, max_tokens=budget, w=full)
    assert s.num_seqs == 2 and int(s.context_lens.sum()) <= budget
    assert "cut to its first" in desc
    L, nq = int(s.context_lens[1]), s.n_query_per_seq
    for j in range(nq):                                # new tokens at the cut context's end
        pos = L - nq + j
        assert int(s.slot_mapping[nq + j]) == int(s.block_tables[1, pos // 16]) * 16 + pos % 16
    out, _, _ = o.step(s)
    assert out.shape == (2 * nq, s.num_q_heads, s.head_dim) and np.isfinite(out).all()


def test_reference_arm_bounded_for_many_steps(monkeypatch):
    monkeypatch.setattr(bench, "REF_BUDGET_S", 3.0)
    args = bench.argparse.Namespace(workload="llama3_8b_decode", kv_dtype="bf16", steps=400,
                                    warmup=3)
    res = bench.run_reference(args)
    assert res["steps"] == 400 and res["value"] > 0
    assert "cut to its first" in res["config"]["sample"]
