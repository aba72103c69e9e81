"""Checks shared by the block-manager tests (the Python model and the library's
C++ manager go through the same ones).

A manager here is any object with add_sequence(seq, n) -> bool, fork(parent,
child), free(seq), append_batch(seqs, n) -> (slots, copies) | None,
num_free(), table(seq), length(seq) and ref(block).

Nothing here trusts the manager: the invariants are recomputed from its block
tables, and a simulated pool (slot -> token value) receives the prompt writes,
the copy-on-write pairs and the appended tokens exactly as the device would,
so every live sequence must read back its own logical token stream.
"""
from __future__ import annotations

import json
import os
from collections import Counter

import numpy as np

BS = 16
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "cow_worked_examples.json")


def ceil_div(a, b):
    return -(-a // b)


class Pool:
    """The device pool as the host sees it: slot -> token value."""

    def __init__(self):
        self.slots: dict[int, int] = {}

    def write_prompt(self, table, tokens):
        for i, v in enumerate(tokens):
            self.slots[table[i // BS] * BS + i % BS] = v

    def apply(self, slots, copies, values):
        # all copies first (pkv_copy_blocks), then the new rows (pkv_kv_append)
        snapshot = {a: [self.slots.get(a * BS + o) for o in range(BS)] for a, _ in copies}
        for a, b in copies:
            for o in range(BS):
                v = snapshot[a][o]
                if v is None:
                    self.slots.pop(b * BS + o, None)
                else:
                    self.slots[b * BS + o] = v
        for s, v in zip(slots, values):
            self.slots[s] = v

    def read(self, table, n):
        return [self.slots.get(table[i // BS] * BS + i % BS) for i in range(n)]


def check_state(bm, live: dict, num_blocks: int, pool: Pool | None = None):
    """Invariants of the manager against the sequences the test knows are live."""
    refs = Counter()
    for s, toks in live.items():
        t = bm.table(s)
        assert bm.length(s) == len(toks), f"seq {s}: length {bm.length(s)} != {len(toks)}"
        # waste bound: exactly ceil(n/16) blocks, so less than one block of waste
        assert len(t) == ceil_div(len(toks), BS), f"seq {s}: {len(t)} blocks for {len(toks)} tokens"
        assert all(0 <= b < num_blocks for b in t), f"seq {s}: block id out of the pool"
        refs.update(t)
        if pool is not None:
            got = pool.read(t, len(toks))
            assert got == toks, f"seq {s}: read back differs at {next(i for i, (a, b) in enumerate(zip(got, toks)) if a != b)}"
    for b in range(num_blocks):
        assert bm.ref(b) == refs.get(b, 0), f"block {b}: count {bm.ref(b)} != {refs.get(b, 0)} holders"
    # no leak and no double free: the free blocks are exactly the unheld ones
    assert bm.num_free() == num_blocks - len(refs), \
        f"{bm.num_free()} free + {len(refs)} held != {num_blocks}"


def canonical(bm, seqs):
    """Sharing structure with physical ids renamed by first appearance."""
    names = {}
    out = []
    for s in seqs:
        row = []
        for b in bm.table(s):
            names.setdefault(b, len(names))
            row.append(names[b])
        out.append((bm.length(s), tuple(row)))
    return out


def worked_examples():
    with open(GOLDEN) as f:
        g = json.load(f)
    assert g["block_size"] == BS
    return g["examples"]


def run_worked_example(make, ex):
    """Fork `samples` outputs of one prompt, then let each write its first token."""
    n, k = ex["prompt_tokens"], ex["samples"]
    nb = 4 * k * ceil_div(n, BS) + 64
    bm = make(nb)
    pool = Pool()
    prompt = list(range(1000, 1000 + n))
    assert bm.add_sequence(0, n)
    pool.write_prompt(bm.table(0), prompt)
    for c in range(1, k):
        bm.fork(0, c)
    held = nb - bm.num_free()
    assert held == ex["blocks_with_sharing"] == ex["prompt_blocks"]
    assert k * held == ex["blocks_without_sharing"]
    assert len(bm.table(0)) - (n % BS != 0) == ex["full_prompt_blocks"]
    assert n - (len(bm.table(0)) - 1) * BS == ex["tokens_in_last_prompt_block"]
    assert all(bm.ref(b) == ex["shared_refcount"] for b in bm.table(0))
    res = bm.append_batch(list(range(k)), 1)
    assert res is not None
    slots, copies = res
    assert len(copies) == ex["private_copies_after_first_token"]
    assert nb - bm.num_free() == ex["blocks_after_first_token"]
    firsts = [-1 - c for c in range(k)]
    pool.apply(slots, copies, firsts)
    live = {c: prompt + [firsts[c]] for c in range(k)}
    check_state(bm, live, nb, pool)
    return bm


def fuzz(make, num_blocks: int, n_ops: int, seed: int, max_nq: int = 4, check_every: int = 1):
    """Random add / fork / batch-append / free operations; invariants after each."""
    rng = np.random.default_rng(seed)
    bm = make(num_blocks)
    pool = Pool()
    live: dict[int, list[int]] = {}
    next_seq = 0
    next_tok = 0
    stats = Counter()
    for op_i in range(n_ops):
        op = rng.choice(["add", "fork", "append", "append", "append", "free", "fill"],
                        p=[0.18, 0.12, 0.22, 0.22, 0.12, 0.12, 0.02])
        if op == "add" or not live:
            n = int(rng.integers(0, 80))
            toks = list(range(next_tok, next_tok + n))
            next_tok += n
            free_before = bm.num_free()
            if bm.add_sequence(next_seq, n):
                live[next_seq] = toks
                pool.write_prompt(bm.table(next_seq), toks)
                stats["add"] += 1
            else:
                assert ceil_div(n, BS) > free_before
                assert bm.num_free() == free_before
                stats["add_refused"] += 1
            next_seq += 1
        elif op == "fork":
            parent = int(rng.choice(list(live)))
            bm.fork(parent, next_seq)
            live[next_seq] = list(live[parent])
            next_seq += 1
            stats["fork"] += 1
        elif op == "append":
            k = int(rng.integers(1, min(len(live), 8) + 1))
            seqs = [int(s) for s in rng.choice(list(live), size=k, replace=False)]
            nq = int(rng.integers(1, max_nq + 1))
            before = {s: bm.table(s) for s in seqs}
            free_before = bm.num_free()
            res = bm.append_batch(seqs, nq)
            if res is None:
                assert bm.num_free() == free_before
                assert all(bm.table(s) == before[s] for s in seqs)
                stats["append_refused"] += 1
            else:
                slots, copies = res
                assert len(slots) == k * nq
                assert len(copies) <= k
                dsts = [b for _, b in copies]
                assert len(set(dsts)) == len(dsts)
                assert not set(dsts) & {a for a, _ in copies}
                vals = list(range(next_tok, next_tok + len(slots)))
                next_tok += len(slots)
                pool.apply(slots, copies, vals)
                for i, s in enumerate(seqs):
                    live[s] += vals[i * nq:(i + 1) * nq]
                stats["append"] += 1
                stats["copies"] += len(copies)
        elif op == "free":
            s = int(rng.choice(list(live)))
            bm.free(s)
            del live[s]
            stats["free"] += 1
        elif op == "fill":
            # every free block must be handed out once, none of them held
            nfree = bm.num_free()
            held = {b for s in live for b in bm.table(s)}
            assert bm.add_sequence(next_seq, nfree * BS)
            got = bm.table(next_seq)
            assert len(set(got)) == nfree and not set(got) & held
            assert bm.num_free() == 0
            assert not bm.add_sequence(next_seq + 1, 1)
            bm.free(next_seq)
            next_seq += 2
            stats["fill"] += 1
        if op_i % check_every == 0:
            check_state(bm, live, num_blocks, pool)
    check_state(bm, live, num_blocks, pool)
    for s in list(live):
        bm.free(s)
    assert bm.num_free() == num_blocks
    assert all(bm.ref(b) == 0 for b in range(num_blocks))
    return stats
