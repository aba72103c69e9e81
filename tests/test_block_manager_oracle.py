"""Pins of the Python block-manager model (oracle/block_manager.py) and of the
oracle's block copy, against what the pages fix:

- the worked examples of copy-on-write under parallel sampling
  (tests/golden/cow_worked_examples.json, each with its citation);
- the allocation rule "a new block only when the last one is full", checked at
  every token of a long run ("LLM Serving: Continuous Batching &
  PagedAttention", section 4.1: token 16 takes one new block);
- the waste bound (exactly ceil(n/16) blocks), conservation of blocks, counts
  equal to holders, and read-back of every sequence's tokens through a
  simulated pool, after each of thousands of random operations (the exercise of
  "ML Interview Prep, Lesson 13", section 10, item 3: no leaked block, no
  double free);
- planted mistakes in a copy of the model, each caught by one of the above.
"""
import re

import numpy as np
import pytest

import bm_harness as H
import oracle
from oracle import block_manager as BMmod
from oracle.block_manager import BlockManagerModel


@pytest.mark.parametrize("ex", H.worked_examples(), ids=lambda e: f"prompt{e['prompt_tokens']}")
def test_worked_example(ex):
    H.run_worked_example(BlockManagerModel, ex)


def test_new_block_exactly_when_last_is_full():
    bm = BlockManagerModel(64)
    assert bm.add_sequence(0, 16)                 # one full block
    assert bm.num_free() == 63
    for t in range(16, 16 * 40):                  # token index t is appended
        before = bm.num_free()
        slots, copies = bm.append(0)
        assert copies == []
        took = before - bm.num_free()
        assert took == (1 if t % 16 == 0 else 0), t
        assert slots[0] % 16 == t % 16
        assert slots[0] // 16 == bm.table(0)[t // 16]


def test_empty_sequence_takes_its_first_block_on_append():
    bm = BlockManagerModel(4)
    assert bm.add_sequence(7, 0)
    assert bm.table(7) == [] and bm.num_free() == 4
    (slot,), _ = bm.append(7)
    assert bm.num_free() == 3 and slot == bm.table(7)[0] * 16


def test_refused_append_changes_nothing():
    bm = BlockManagerModel(3)
    assert bm.add_sequence(0, 20)                 # 2 blocks, 1 free
    bm.fork(0, 1)
    # seq 0 copies its shared last block (1 block) and seq 1 then writes in
    # place; 13 more tokens each would need more blocks than the pool has
    assert bm.append_batch([0, 1], 13) is None
    assert bm.num_free() == 1 and bm.table(0) == bm.table(1)
    assert [bm.ref(b) for b in bm.table(0)] == [2, 2]


def test_no_sharing_uses_sum_of_ceils():
    rng = np.random.default_rng(3)
    bm = BlockManagerModel(10_000)
    lens = rng.integers(0, 3000, size=50)
    for s, n in enumerate(lens):
        assert bm.add_sequence(s, int(n))
    assert 10_000 - bm.num_free() == sum(-(-int(n) // 16) for n in lens)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_fuzz_model(seed):
    stats = H.fuzz(BlockManagerModel, num_blocks=96, n_ops=3000, seed=seed)
    # the run must have exercised every path
    for k in ("add", "fork", "append", "free", "copies", "append_refused", "fill"):
        assert stats[k] > 0, (k, stats)


def test_oracle_copy_blocks_moves_whole_blocks():
    o = oracle.Oracle()
    rng = np.random.default_rng(5)
    k = rng.integers(0, 65536, size=(12, 16, 2, 64), dtype=np.uint16)
    v = rng.integers(0, 65536, size=(12, 16, 2, 64), dtype=np.uint16)
    src, dst = [3, 0, 7], [9, 11, 1]
    k2, v2 = o.copy_blocks(k, v, src, dst)
    for a, b in zip(src, dst):
        assert (k2[b] == k[a]).all() and (v2[b] == v[a]).all()
    untouched = [i for i in range(12) if i not in dst]
    assert (k2[untouched] == k[untouched]).all() and (v2[untouched] == v[untouched]).all()
    # a pair outside the pool copies nothing
    k3, v3 = o.copy_blocks(k, v, [12, -1], [0, 1])
    assert (k3 == k).all() and (v3 == v).all()


# ---- planted mistakes: each must be caught
MUTANTS = {
    "no_copy_on_write": ("if self.refcount[last] > 1:", "if self.refcount[last] > 99:"),
    "copy_keeps_count": ("                self.refcount[last] -= 1\n", ""),
    "copy_not_reported": ("copies.append((last, new))", "pass"),
    "new_block_one_late": ("if t % self.block_size == 0:", "if t % self.block_size == 1 or t == 0:"),
    "fork_no_count": ("            self.refcount[b] += 1\n", "            pass\n"),
    "release_early": ("if self.refcount[b] == 0:", "if self.refcount[b] <= 1:"),
    "slot_offset": ("+ t % self.block_size\n", "+ (t + 1) % self.block_size\n"),
    "prompt_floor": ("need = -(-n_tokens // self.block_size)", "need = n_tokens // self.block_size"),
}


def _mutant_class(old, new):
    src = open(BMmod.__file__).read()
    assert src.count(old) == 1, old
    ns = {"__name__": "bm_mutant"}
    exec(compile(src.replace(old, new), "bm_mutant", "exec"), ns)
    return ns["BlockManagerModel"]


def _pins(cls):
    for ex in H.worked_examples():
        H.run_worked_example(cls, ex)
    H.fuzz(cls, num_blocks=64, n_ops=600, seed=11)


def test_pins_pass_on_the_model():
    _pins(BlockManagerModel)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    cls = _mutant_class(*MUTANTS[name])
    with pytest.raises(Exception):
        _pins(cls)


def test_mutant_texts_apply():
    src = open(BMmod.__file__).read()
    for old, _ in MUTANTS.values():
        assert src.count(old) == 1, old
    assert re.search(r"class BlockManagerModel", src)
