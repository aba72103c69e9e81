"""Plain Python model of the paged KV block manager.

TEST INFRASTRUCTURE. Only ``tests/`` use this module; it shares no code with
the library's C++ block manager, and neither imports the other.

What it models, step by step as the pages state it:

- The KV memory is a pool of fixed-size physical blocks of 16 token slots;
  every sequence has a block table whose entry i names the physical block of
  its tokens 16i .. 16i+15, and a sequence takes a new block only when its
  last block is full ("ML Interview Prep, Lesson 13", section 3.5 "Paged
  attention"; "LLM Serving: Continuous Batching & PagedAttention", section 4.1:
  the block for token 16 comes from the free-frame list).
- A free list hands blocks out; a reference count per block says how many
  sequences hold it; releasing a block lowers its count and a block whose count
  reaches zero goes back to the free list ("LLM Serving: Continuous Batching &
  PagedAttention", section 7, block manager; "ML Interview Prep, Lesson 13",
  section 3.5, step loop item 1).
- Sharing: parallel sampling forks a sequence, and the fork holds the same
  physical blocks with their counts raised ("ML Interview Prep, Lesson 13",
  section 3.5 "Sharing"; "LLM Serving: Continuous Batching & PagedAttention",
  section 4.2).
- Copy-on-write: before a sequence writes into a block whose count is above 1,
  it gets a private copy and the shared block's count drops by one (same
  passages). The copy is reported as a (source, destination) pair, to be
  carried out on the device before the new rows are written.

Readings where the pages leave a step open:

- A sequence of n tokens holds exactly ceil(n / 16) blocks (the waste bound of
  "ML Interview Prep, Lesson 13", section 3.5); a sequence created with 0
  tokens holds none and its first append takes one.
- Several tokens appended in one call (speculative verification) are placed one
  after another; a call that cannot get every block it needs changes nothing
  and returns ``None``. A batch append is all-or-nothing the same way and
  handles the sequences in the order given, so of several sequences sharing a
  partly filled last block the ones handled first get copies and the last one
  writes in place (the worked example of "ML Interview Prep, Lesson 13",
  section 8, question 4).
- The free list is a stack whose first pops give blocks 0, 1, 2, ...; the
  choice of physical ids is not part of the method, so tests compare the
  sharing structure and counts, never the ids themselves.
"""
from __future__ import annotations

import copy

import numpy as np

BLOCK_SIZE = 16


class OutOfBlocks(Exception):
    pass


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int = BLOCK_SIZE):
        self.block_size = block_size
        self.num_blocks = num_blocks
        self.free_list = list(range(num_blocks - 1, -1, -1))
        self.refcount = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lengths: dict[int, int] = {}

    # ---- the free list and the reference counts
    def _allocate(self) -> int:
        if not self.free_list:
            raise OutOfBlocks
        b = self.free_list.pop()
        self.refcount[b] = 1
        return b

    def _release(self, b: int) -> None:
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            self.free_list.append(b)

    def num_free(self) -> int:
        return len(self.free_list)

    # ---- sequences
    def add_sequence(self, seq: int, n_tokens: int) -> bool:
        """A new sequence holding ceil(n_tokens/16) fresh blocks (its prompt)."""
        if seq in self.tables:
            raise KeyError(f"sequence {seq} exists")
        need = -(-n_tokens // self.block_size)
        if need > len(self.free_list):
            return False
        self.tables[seq] = [self._allocate() for _ in range(need)]
        self.lengths[seq] = n_tokens
        return True

    def fork(self, parent: int, child: int) -> None:
        """``child`` shares every block of ``parent`` (parallel sampling)."""
        if child in self.tables:
            raise KeyError(f"sequence {child} exists")
        table = self.tables[parent]
        for b in table:
            self.refcount[b] += 1
        self.tables[child] = list(table)
        self.lengths[child] = self.lengths[parent]

    def free(self, seq: int) -> None:
        """The sequence ends: release each of its blocks."""
        for b in self.tables.pop(seq):
            self._release(b)
        del self.lengths[seq]

    def _append_one(self, seq: int, copies: list) -> int:
        table = self.tables[seq]
        t = self.lengths[seq]
        if t % self.block_size == 0:
            table.append(self._allocate())          # the last block is full (or none yet)
        else:
            last = table[-1]
            if self.refcount[last] > 1:             # shared: private copy first
                new = self._allocate()
                copies.append((last, new))
                self.refcount[last] -= 1
                table[-1] = new
        self.lengths[seq] = t + 1
        return table[t // self.block_size] * self.block_size + t % self.block_size

    def append_batch(self, seqs, n_per_seq: int = 1):
        """Slots for n tokens of each sequence (in the order given) and the copy
        pairs, or None (and no change) when the free blocks do not suffice."""
        if len(set(seqs)) != len(seqs):
            raise KeyError("a sequence appears twice in one batch")
        saved = (copy.deepcopy(self.tables), dict(self.lengths), list(self.refcount),
                 list(self.free_list))
        slots, copies = [], []
        try:
            for s in seqs:
                for _ in range(n_per_seq):
                    slots.append(self._append_one(s, copies))
        except OutOfBlocks:
            self.tables, self.lengths, self.refcount, self.free_list = saved
            return None
        return slots, copies

    def append(self, seq: int, n: int = 1):
        return self.append_batch([seq], n)

    # ---- read-only views
    def table(self, seq: int) -> list[int]:
        return list(self.tables[seq])

    def length(self, seq: int) -> int:
        return self.lengths[seq]

    def ref(self, block: int) -> int:
        return self.refcount[block]

    # ---- what the attention kernel reads
    def block_tables(self, seqs, max_blocks_per_seq: int):
        """int32 [len(seqs), max_blocks_per_seq] padded with -1, and int32 lengths."""
        tables = np.full((len(seqs), max_blocks_per_seq), -1, dtype=np.int32)
        lens = np.zeros(len(seqs), dtype=np.int32)
        for i, s in enumerate(seqs):
            t = self.tables[s]
            tables[i, :len(t)] = t
            lens[i] = self.lengths[s]
        return tables, lens
