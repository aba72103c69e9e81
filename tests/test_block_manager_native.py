"""The library's C++ block manager (include/pkv_block_manager.h), on the host:
the worked examples, thousands of random operations with the invariants and
read-back checks of bm_harness, the manager's own audit, and lockstep
agreement with the Python model (oracle/block_manager.py) on every result,
with physical ids compared only up to a consistent renaming."""
import ctypes
import threading

import numpy as np
import pytest

import bm_harness as H
import paged_kv_cache_101_gb300 as pkv
from oracle.block_manager import BlockManagerModel
from paged_kv_cache_101_gb300 import _build

SEQ, NOBLK, SHAPE, RANGE, NULL = pkv.PKV_ERR_SEQUENCE, pkv.PKV_ERR_NO_BLOCKS, 2, 5, 1


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return pkv.lib()


class Audited(pkv.BlockManager):
    """The native manager, audited by pkv_bm_check after every mutation."""

    def _audit(self):
        assert self.check() == 0, f"pkv_bm_check = {self.check()}"

    def add_sequence(self, seq, n):
        r = super().add_sequence(seq, n)
        self._audit()
        return r

    def fork(self, parent, child):
        super().fork(parent, child)
        self._audit()

    def free(self, seq):
        super().free(seq)
        self._audit()

    def append_batch(self, seqs, n=1):
        r = super().append_batch(seqs, n)
        self._audit()
        return r


class Lockstep:
    """Runs every operation on the model and the native manager; results must
    agree up to one fixed bijection between their physical block ids."""

    def __init__(self, num_blocks):
        self.m = BlockManagerModel(num_blocks)
        self.n = Audited(num_blocks)
        self.to_native = {}

    def _same_block(self, bm, bn):
        prev = self.to_native.setdefault(bm, bn)
        assert prev == bn, f"model block {bm} maps to {prev} and {bn}"

    def _same_table(self, seq):
        tm, tn = self.m.table(seq), self.n.table(seq)
        assert len(tm) == len(tn)
        for a, b in zip(tm, tn):
            self._same_block(a, b)
            assert self.m.ref(a) == self.n.ref(b)

    def add_sequence(self, seq, n):
        a, b = self.m.add_sequence(seq, n), self.n.add_sequence(seq, n)
        assert a == b
        if a:
            self._same_table(seq)
        return b

    def fork(self, parent, child):
        self.m.fork(parent, child)
        self.n.fork(parent, child)
        self._same_table(child)

    def free(self, seq):
        self.m.free(seq)
        self.n.free(seq)
        assert self.m.num_free() == self.n.num_free()

    def append_batch(self, seqs, n=1):
        a, b = self.m.append_batch(seqs, n), self.n.append_batch(seqs, n)
        assert (a is None) == (b is None)
        if a is None:
            return None
        (sm, cm), (sn, cn) = a, b
        assert len(sm) == len(sn) and len(cm) == len(cn)
        for x, y in zip(sm, sn):
            assert x % 16 == y % 16
            self._same_block(x // 16, int(y) // 16)
        for (pa, pb), (qa, qb) in zip(cm, cn):
            self._same_block(pa, qa)
            self._same_block(pb, qb)
        for s in seqs:
            self._same_table(s)
        assert self.m.num_free() == self.n.num_free()
        return b

    def num_free(self):
        return self.n.num_free()

    def table(self, seq):
        return self.n.table(seq)

    def length(self, seq):
        assert self.m.length(seq) == self.n.length(seq)
        return self.n.length(seq)

    def ref(self, block):
        return self.n.ref(block)


@pytest.mark.parametrize("ex", H.worked_examples(), ids=lambda e: f"prompt{e['prompt_tokens']}")
def test_worked_example_native(ex):
    bm = H.run_worked_example(Audited, ex)
    assert bm.check() == 0


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_fuzz_native(seed):
    stats = H.fuzz(Audited, num_blocks=96, n_ops=3000, seed=seed)
    for k in ("add", "fork", "append", "free", "copies", "append_refused", "fill"):
        assert stats[k] > 0, (k, stats)


@pytest.mark.parametrize("seed", [10, 11])
def test_lockstep_with_model(seed):
    H.fuzz(Lockstep, num_blocks=128, n_ops=2500, seed=seed, check_every=5)


def test_block_tables_for_the_attention_call():
    bm = pkv.BlockManager(64)
    assert bm.add_sequence(5, 40)                    # 3 blocks
    assert bm.add_sequence(9, 0)
    bm.fork(5, 6)
    tables, lens = bm.block_tables([6, 9, 5], 4)
    assert lens.tolist() == [40, 0, 40]
    assert tables[0].tolist() == bm.table(5) + [-1] and tables[1].tolist() == [-1] * 4
    assert (tables[2] == tables[0]).all()
    with pytest.raises(pkv.PkvError) as e:
        bm.block_tables([5], 2)                      # 3 blocks do not fit 2 columns
    assert e.value.status == RANGE
    with pytest.raises(pkv.PkvError) as e:
        bm.block_tables([77], 4)
    assert e.value.status == SEQ


def test_errors_change_nothing():
    bm = pkv.BlockManager(8)
    assert bm.add_sequence(1, 100)                   # 7 blocks
    assert not bm.add_sequence(2, 33)                # needs 3, 1 free
    assert bm.num_free() == 1 and bm.num_sequences() == 1
    with pytest.raises(pkv.PkvError) as e:
        bm.add_sequence(1, 3)
    assert e.value.status == SEQ
    with pytest.raises(pkv.PkvError) as e:
        bm.fork(1, 1)
    assert e.value.status == SEQ
    with pytest.raises(pkv.PkvError) as e:
        bm.fork(42, 3)
    assert e.value.status == SEQ
    with pytest.raises(pkv.PkvError) as e:
        bm.append_batch([1, 1], 1)                   # repeated id
    assert e.value.status == SEQ
    with pytest.raises(pkv.PkvError) as e:
        bm.free(2)
    assert e.value.status == SEQ
    bm.fork(1, 2)
    # both share a 4-token last block: seq 1 copies (1 block), seq 2 writes in
    # place; 13 more tokens each cross into new blocks -> not enough
    assert bm.append_batch([1, 2], 13) is None
    assert bm.num_free() == 1 and bm.table(1) == bm.table(2) and bm.check() == 0
    slots, copies = bm.append_batch([1, 2], 1)
    assert len(copies) == 1 and bm.num_free() == 0 and bm.check() == 0
    assert copies[0][0] == bm.table(2)[-1] and copies[0][1] == bm.table(1)[-1]


def test_raw_abi_edge_cases():
    L = pkv.lib()
    assert not L.pkv_bm_create(0) and not L.pkv_bm_create(-3) and not L.pkv_bm_create(1 << 31)
    assert L.pkv_bm_num_free(None) == -1 and L.pkv_bm_check(None) == -1
    assert L.pkv_bm_refcount(None, 0) == -1
    assert L.pkv_bm_add_sequence(None, 0, 1) == NULL
    h = L.pkv_bm_create(4)
    try:
        assert L.pkv_bm_add_sequence(h, 0, -1) == SHAPE
        assert L.pkv_bm_refcount(h, 4) == -1 and L.pkv_bm_refcount(h, -1) == -1
        nc = ctypes.c_int32(7)
        # empty batches are no-ops and may pass NULL arrays
        assert L.pkv_bm_append(h, None, 0, 1, None, None, None, ctypes.byref(nc)) == 0
        assert nc.value == 0
        assert L.pkv_bm_append(h, None, 3, 1, None, None, None, ctypes.byref(nc)) == NULL
        assert L.pkv_bm_append(h, None, -1, 1, None, None, None, None) == SHAPE
        assert L.pkv_bm_sequence_length(h, 0) == -1
        assert L.pkv_bm_add_sequence(h, 0, 20) == 0
        buf = (ctypes.c_int32 * 1)()
        assert L.pkv_bm_sequence_blocks(h, 0, buf, 1) == 2   # count, capacity 1 written
        assert buf[0] == 0
        assert L.pkv_bm_num_blocks(h) == 4
    finally:
        L.pkv_bm_destroy(h)
    L.pkv_bm_destroy(None)


def test_threads_share_one_manager():
    bm = pkv.BlockManager(4096)
    errors = []

    def worker(base):
        try:
            rng = np.random.default_rng(base)
            mine = []
            for i in range(300):
                s = base * 10_000 + i
                if bm.add_sequence(s, int(rng.integers(1, 40))):
                    mine.append(s)
                if mine and rng.random() < 0.5:
                    bm.append_batch([mine[-1]], int(rng.integers(1, 5)))
                if len(mine) > 8:
                    bm.free(mine.pop(0))
            for s in mine:
                bm.free(s)
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    ts = [threading.Thread(target=worker, args=(k,)) for k in range(1, 7)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    assert bm.check() == 0 and bm.num_free() == 4096 and bm.num_sequences() == 0
