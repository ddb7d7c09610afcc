"""Pins of the block-manager model against the pages' semantics and invariants."""
from __future__ import annotations

import os
import random

import pytest

from oracle.alloc_model import BlockAllocatorModel, RefCountError

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def check_invariants(m: BlockAllocatorModel):
    N, B = m.num_blocks, m.block_size
    counts = [0] * N
    for sq in m.seqs.values():
        for b in sq["blocks"]:
            counts[b] += 1
        # on-demand blocks: exactly ceil(len / B), so waste is < 1 block
        assert len(sq["blocks"]) == -(-sq["len"] // B)
    assert counts == m.ref
    assert len(set(m.free)) == len(m.free)
    assert all(m.ref[b] == 0 for b in m.free)
    assert m.num_free() + sum(1 for r in m.ref if r > 0) == N
    # prefix records: one block per prefix and back, every initialized free block has one
    assert len(set(m.init)) == len(m.init) and not set(m.init) & set(m.free)
    assert all(m.ref[b] == 0 and b in m.key_of for b in m.init)
    assert all(m.key_of[b] == k for k, b in m.record.items()) and len(m.key_of) == len(m.record)
    assert all(len(k) % B == 0 and len(k) > 0 for k in m.record)


def test_free_list_hands_out_from_the_end():
    m = BlockAllocatorModel(10, 4)
    m.add_seq(0)
    slots, pairs = m.append_slots([0])
    assert m.table(0) == [9] and slots == [36] and pairs == []
    for _ in range(4):
        m.append_slots([0])
    assert m.table(0) == [9, 8]


def test_empty_pool_raises_and_changes_nothing():
    m = BlockAllocatorModel(2, 4)
    for s in range(3):
        m.add_seq(s)
    m.append_slots([0, 1])
    before = (list(m.free), list(m.ref), {k: dict(v, blocks=list(v["blocks"])) for k, v in m.seqs.items()})
    with pytest.raises(MemoryError):
        m.append_slots([0, 2])  # seq 0 fits in its block, seq 2 needs a new one
    assert (m.free, m.ref) == (before[0], before[1])
    assert m.length(0) == 1 and m.length(2) == 0


def test_prefix_sharing_table_of_the_blog_example():
    B = 16
    m = BlockAllocatorModel(32, B)
    m.add_seq(0)
    for _ in range(3 * B):          # a system prompt filling three blocks
        m.append_slots([0])
    m.fork(0, 1)
    for _ in range(2 * B):
        _, pairs = m.append_slots([0, 1])
        assert pairs == []          # full shared blocks are never copied
    a, b = m.table(0), m.table(1)
    rows = {}
    with open(os.path.join(GOLDEN, "prefix_sharing_table.txt"), encoding="utf-8") as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, *v = line.split()
                rows[k] = v
    names = {}
    for seq, tbl in (("A", a), ("B", b)):
        for name, blk in zip(rows[seq], tbl):
            assert names.setdefault(name, blk) == blk
    assert len(set(names.values())) == len(names)  # distinct names, distinct blocks
    for name, blk in names.items():
        want = int(rows["shared_refcount"][0]) if name.startswith("shared") else int(rows["private_refcount"][0])
        assert m.ref[blk] == want
    check_invariants(m)


def test_parallel_sampling_copy_on_write():
    """Prompt of 1000 tokens (62 full blocks + 8 slots), 8 samples: the
    first 7 writers copy the shared partial block, the last writes in
    place; full shared blocks are never copied."""
    B = 16
    m = BlockAllocatorModel(200, B)
    m.add_seq(0)
    for _ in range(1000):
        m.append_slots([0])
    shared_last = m.table(0)[-1]
    for c in range(1, 8):
        m.fork(0, c)
    assert m.ref[shared_last] == 8
    slots, pairs = m.append_slots(list(range(8)))
    assert len(pairs) == 7
    assert all(src == shared_last for src, _ in pairs)
    assert len({dst for _, dst in pairs}) == 7
    assert m.ref[shared_last] == 1
    # the one sequence still holding the original writes at slot 1000 % 16 of it
    assert (shared_last * B + 1000 % B) in slots
    for s in range(8):
        assert m.table(s)[:62] == m.table(0)[:62]
    check_invariants(m)


def test_shared_blocks_are_freed_only_at_zero():
    B = 4
    m = BlockAllocatorModel(16, B)
    m.add_seq(0)
    for _ in range(10):
        m.append_slots([0])
    m.fork(0, 1)
    prompt = m.table(0)
    m.free_seq(0)
    assert all(m.ref[b] == 1 for b in prompt)
    assert not any(b in m.free for b in prompt)
    m.free_seq(1)
    assert all(b in m.free for b in prompt)
    check_invariants(m)
    with pytest.raises(RefCountError):
        m._release(prompt[0])


def test_random_operation_sequences_keep_invariants():
    rng = random.Random(0)
    for trial in range(20):
        B = rng.choice([1, 2, 4, 16])
        m = BlockAllocatorModel(rng.randint(8, 64), B)
        nxt = 0
        for _ in range(300):
            op = rng.random()
            live = list(m.seqs)
            if op < 0.15 or not live:
                m.add_seq(nxt)
                nxt += 1
            elif op < 0.25:
                m.fork(rng.choice(live), nxt)
                nxt += 1
            elif op < 0.35:
                m.free_seq(rng.choice(live))
            else:
                batch = rng.sample(live, rng.randint(1, len(live)))
                try:
                    m.append_slots(batch)
                except MemoryError:
                    pass
            check_invariants(m)


# -- prefix caching (continuous-batching page, "Prefix 캐싱" / "제거") ------------

def test_prefix_cache_shares_completed_blocks_of_a_common_prompt():
    """B = 4.  Request A's prompt is 1..10 (two full blocks + 2 tokens);
    request B's prompt shares A's first 8 ids and then differs."""
    m = BlockAllocatorModel(16, 4, prefix_cache=True)
    assert m.add_seq_prefix(0, range(1, 11)) == 0  # nothing recorded yet
    for t in range(1, 11):
        m.append_slots([0], [t])
    assert m.table(0) == [15, 14, 13]  # taken from the end of the free list
    assert m.prefix_stats() == (2, 0)  # blocks [1..4] and [1..8] are full: recorded
    assert m.add_seq_prefix(1, [1, 2, 3, 4, 5, 6, 7, 8, 99, 98]) == 8
    assert m.table(1) == [15, 14] and m.ref[15] == m.ref[14] == 2
    for t in (99, 98):
        m.append_slots([1], [t])
    assert m.table(1) == [15, 14, 12]  # a block of its own after the shared prefix
    # a prompt that differs inside the first block shares nothing
    assert m.add_seq_prefix(2, [1, 2, 3, 5, 5, 6, 7, 8]) == 0
    # one that repeats the first block only
    assert m.add_seq_prefix(3, [1, 2, 3, 4, 0, 0]) == 4 and m.table(3) == [15]
    check_invariants(m)


def test_freed_blocks_stay_matchable_until_demoted_most_recent_first():
    m = BlockAllocatorModel(4, 2, prefix_cache=True)
    m.add_seq_prefix(0, [7, 7, 8, 8])
    for t in (7, 7, 8, 8):
        m.append_slots([0], [t])
    assert m.table(0) == [3, 2] and m.prefix_stats() == (2, 0)
    m.free_seq(0)  # released in logical order: 3 then 2 -> initialized, 2 most recent
    assert m.free == [0, 1] and m.init == [3, 2] and m.num_free() == 4
    # a new request with the same prompt takes both back without prefill
    assert m.add_seq_prefix(1, [7, 7, 8, 8, 9]) == 4 and m.table(1) == [3, 2] and m.init == []
    m.free_seq(1)
    assert m.init == [3, 2]
    # fill the pool with unrelated tokens: the free list goes first (1, 0), then
    # the most recently freed initialized block (2) loses its record
    m.add_seq(5)
    for _ in range(6):
        m.append_slots([5])
    assert m.table(5) == [1, 0, 2] and m.init == [3] and m.prefix_stats() == (1, 1)
    # the [7, 7] block is still recorded; the [7, 7, 8, 8] one is gone
    assert m.add_seq_prefix(6, [7, 7, 8, 8]) == 2 and m.table(6) == [3]
    check_invariants(m)


def test_random_prefix_cache_sequences_keep_invariants():
    rng = random.Random(5)
    for trial in range(15):
        B = rng.choice([1, 2, 4])
        m = BlockAllocatorModel(rng.randint(6, 40), B, prefix_cache=True)
        families = [[rng.randint(0, 3) for _ in range(rng.randint(1, 12))] for _ in range(4)]
        nxt = 0
        for _ in range(300):
            op = rng.random()
            live = list(m.seqs)
            if op < 0.15 or not live:
                prompt = list(rng.choice(families)) + [rng.randint(0, 3) for _ in range(rng.randint(0, 3))]
                n = m.add_seq_prefix(nxt, prompt)
                assert n % B == 0 and n <= len(prompt)
                nxt += 1
            elif op < 0.22:
                m.fork(rng.choice(live), nxt)
                nxt += 1
            elif op < 0.32:
                m.free_seq(rng.choice(live))
            else:
                batch = rng.sample(live, rng.randint(1, len(live)))
                try:
                    m.append_slots(batch, [rng.randint(0, 3) for _ in batch])
                except MemoryError:
                    pass
            check_invariants(m)
