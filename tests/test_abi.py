"""Host-side checks of the C-ABI library (no GPU needed).

The library loads, exports every function include/pa.h declares, rejects
bad arguments before launching anything, and its host block allocator and
slot helper agree operation by operation with the oracle's model.
"""
from __future__ import annotations

import ctypes
import os
import random
import re

import numpy as np
import pytest

import oracle
from oracle.alloc_model import BlockAllocatorModel

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_35_gb300 as pa

    return pa


def header_functions():
    text = open(os.path.join(ROOT, "include", "pa.h"), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_function(pa):
    names = header_functions()
    assert len(names) >= 20
    L = ctypes.CDLL(pa.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    assert sorted(pa.SIGNATURES) == names


def test_status_strings_and_version(pa):
    assert pa.lib().pa_version() >= 100
    for st in range(9):
        assert pa.status_string(st) not in ("", "unknown status")
    assert pa.status_string(99) == "unknown status"


def test_bad_arguments_are_rejected_before_launch(pa):
    L = pa.lib()
    fake = ctypes.c_void_p(0x1000)
    # unsupported head_dim / block size / dtype
    args = [fake, pa.PA_F16, fake, fake, fake, fake, 4, fake, 64, 2, 4, 96, 16, 8, 0.1, pa.PA_F16, fake, 1 << 20, 0,
            fake, None]
    assert L.pa_decode(*args) == pa.PA_ERR_UNSUPPORTED
    args[11] = 128
    args[12] = 24
    assert L.pa_decode(*args) == pa.PA_ERR_UNSUPPORTED
    args[12] = 16
    args[15] = 7
    assert L.pa_decode(*args) == pa.PA_ERR_UNSUPPORTED
    args[15] = pa.PA_F16
    args[17] = 16  # workspace too small
    assert L.pa_decode(*args) == pa.PA_ERR_WORKSPACE
    # 2^20 partitions of the longest sequence (max_context_len 2^24, partition 16): unsupported
    big = list(args)
    big[8], big[17], big[18] = 1 << 24, 1 << 40, 16
    assert L.pa_decode(*big) == pa.PA_ERR_UNSUPPORTED
    args[17] = 1 << 20
    args[18] = 24  # partition not a multiple of 16
    assert L.pa_decode(*args) == pa.PA_ERR_INVALID_ARG
    args[18] = 0
    args[16] = None
    assert L.pa_decode(*args) == pa.PA_ERR_INVALID_ARG
    args[9] = 0  # no sequences: nothing to do
    assert L.pa_decode(*args) == pa.PA_OK
    # prefill (every case must be refused before a launch: the pointers are fake):
    # head_dim 96, block size 40 (not a multiple of 16), block size past 65536
    pargs = [fake, pa.PA_BF16, fake, fake, fake, fake, fake, fake, 8, 2, 100, 64, 4, 96, 16, 8, 0.1, pa.PA_BF16, fake,
             None]
    assert L.pa_prefill_chunk(*pargs) == pa.PA_ERR_UNSUPPORTED
    pargs[13] = 128
    for bad_block in (40, 65552):
        pargs[14] = bad_block
        assert L.pa_prefill_chunk(*pargs) == pa.PA_ERR_UNSUPPORTED
    # scatter / copy with nothing to do
    assert L.pa_reshape_and_cache(fake, fake, fake, fake, fake, 0, 4, 64, 16, 8, pa.PA_F16, fake, None) == pa.PA_OK
    assert L.pa_copy_blocks(fake, fake, fake, 0, 4, 64, 16, 8, pa.PA_F16, fake, None) == pa.PA_OK
    assert L.pa_copy_blocks(fake, fake, fake, 1, 4, 64, 16, 8, 9, fake, None) == pa.PA_ERR_UNSUPPORTED
    assert L.pa_get_error(None, None, None) == pa.PA_ERR_INVALID_ARG


def test_partition_and_workspace_sizes(pa):
    assert pa.pa_decode_partition_size(64, 40, 2048) == 512    # 5120 units at 1024: < 16 waves
    assert pa.pa_decode_partition_size(256, 32, 16384) == 1024  # 131072 units at 1024
    assert pa.pa_decode_partition_size(16, 40, 1024) == 1024    # one partition per sequence, 640 pairs
    assert pa.pa_decode_partition_size(8, 40, 1024) == 512      # 320 pairs: split, 640 units at 512
    assert pa.pa_decode_partition_size(32, 40, 4096) == 512     # 5120 units at 1024
    assert pa.pa_decode_partition_size(1, 40, 4096) == 256      # 640 units; 512 would give 320
    assert pa.pa_decode_partition_size(1, 40, 1024) == 64       # 640 units; 128 would give 320
    assert pa.pa_decode_partition_size(1, 8, 4096) == 64        # 512 units; 128 would give 256
    assert pa.pa_decode_partition_size(1, 1, 4096) == 64        # floor
    assert pa.pa_decode_partition_size(0, 40, 4096) == 512
    for S, H, mx in ((1, 1, 1), (3, 7, 100), (1000, 64, 100000), (380, 1, 1025)):
        P = pa.pa_decode_partition_size(S, H, mx)
        assert P in (64, 128, 256, 512, 1024)
    for S, H, D, mx in ((64, 40, 128, 2048), (256, 32, 128, 16384), (4, 4, 64, 46)):
        n = pa.pa_decode_workspace_bytes(S, H, D, mx, 0)
        P = pa.pa_decode_partition_size(S, H, mx)
        parts = -(-mx // P)
        assert n >= 4 * S * H * parts * (D + 2) and n % 256 == 0
    assert pa.pa_decode_workspace_bytes(4, 4, 64, 100, 24) == 0
    assert pa.pa_decode_workspace_bytes(4, 4, 64, 100, 2048) == 0
    # a work item holds fewer than 2^20 partitions of one sequence
    assert pa.pa_decode_workspace_bytes(1, 1, 128, (1 << 24) - 16, 16) > 0   # 2^20 - 1 partitions
    assert pa.pa_decode_workspace_bytes(1, 1, 128, 1 << 24, 16) == 0          # 2^20 partitions
    assert pa.pa_decode_workspace_bytes(1, 1, 128, (1 << 30) - 1024, 1024) > 0  # 2^20 - 1 partitions
    assert pa.pa_decode_workspace_bytes(1, 1, 128, 2 ** 31 - 1, 1024) == 0      # 2^21: refused, no overflow


def test_slot_mapping_matches_the_oracle(pa):
    rng = np.random.default_rng(0)
    for B in (16, 256):
        tables = rng.permutation(400)[:120].reshape(6, 20).astype(np.int32)
        seq = rng.integers(0, 6, 300).astype(np.int32)
        pos = rng.integers(0, 20 * B, 300).astype(np.int32)
        got = pa.pa_slot_mapping(tables, seq, pos, B)
        want = [oracle.slot_of(tables[s], int(p), B) for s, p in zip(seq, pos)]
        assert got.tolist() == want
    tables = np.array([[3, -1]], dtype=np.int32)
    with pytest.raises(pa.PAError):
        pa.pa_slot_mapping(tables, [0], [16], 16)


def _compare(model: BlockAllocatorModel, alloc, seq_ids):
    assert alloc.num_free() == model.num_free()
    assert alloc.num_seqs() == len(model.seqs)
    for b in range(model.num_blocks):
        assert alloc.ref(b) == model.ref[b]
    for s in seq_ids:
        if s in model.seqs:
            tbl, ln = alloc.block_table(s)
            assert tbl == model.table(s) and ln == model.length(s)


def test_allocator_matches_model_on_random_operations(pa):
    rng = random.Random(1)
    for trial in range(12):
        N = rng.randint(4, 48)
        B = rng.choice([1, 4, 16, 256])
        model = BlockAllocatorModel(N, B)
        alloc = pa.BlockAllocator(N, B)
        nxt = 0
        for _ in range(250):
            live = list(model.seqs)
            op = rng.random()
            if op < 0.15 or not live:
                model.add_seq(nxt)
                alloc.add_seq(nxt)
                nxt += 1
            elif op < 0.25:
                p = rng.choice(live)
                model.fork(p, nxt)
                alloc.fork(p, nxt)
                nxt += 1
            elif op < 0.33:
                s = rng.choice(live)
                model.free_seq(s)
                alloc.free_seq(s)
            else:
                batch = rng.sample(live, rng.randint(1, len(live)))
                try:
                    want_slots, want_pairs = model.append_slots(batch)
                except MemoryError:
                    with pytest.raises(pa.PAError) as ei:
                        alloc.append_slots(batch)
                    assert ei.value.status == pa.PA_ERR_NO_FREE_BLOCKS
                else:
                    slots, pairs = alloc.append_slots(batch)
                    assert slots.tolist() == want_slots
                    assert [tuple(p) for p in pairs.tolist()] == want_pairs
            _compare(model, alloc, range(nxt))
        alloc.close()


def test_prefix_cache_allocator_matches_model_on_random_operations(pa):
    """Prompts drawn from a few families over a 4-token vocabulary, so that
    prefixes repeat, blocks are shared, freed, kept initialized, revived and
    demoted; every step is compared with the model (slots, copy pairs, reused
    tokens, tables, counts, cache statistics)."""
    rng = random.Random(7)
    for trial in range(12):
        N = rng.randint(6, 48)
        B = rng.choice([1, 2, 4, 16])
        model = BlockAllocatorModel(N, B, prefix_cache=True)
        alloc = pa.BlockAllocator(N, B, prefix_cache=True)
        families = [[rng.randint(0, 3) for _ in range(rng.randint(1, 3 * B + 2))] for _ in range(4)]
        nxt = 0
        for _ in range(300):
            live = list(model.seqs)
            op = rng.random()
            if op < 0.15 or not live:
                prompt = list(rng.choice(families)) + [rng.randint(0, 3) for _ in range(rng.randint(0, B))]
                assert alloc.add_seq_prefix(nxt, prompt) == model.add_seq_prefix(nxt, prompt)
                nxt += 1
            elif op < 0.22:
                p = rng.choice(live)
                model.fork(p, nxt)
                alloc.fork(p, nxt)
                nxt += 1
            elif op < 0.30:
                s = rng.choice(live)
                model.free_seq(s)
                alloc.free_seq(s)
            else:
                batch = rng.sample(live, rng.randint(1, len(live)))
                ids = None if rng.random() < 0.05 else [rng.randint(0, 3) for _ in batch]
                try:
                    want_slots, want_pairs = model.append_slots(batch, ids)
                except MemoryError:
                    with pytest.raises(pa.PAError) as ei:
                        alloc.append_slots(batch) if ids is None else alloc.append_tokens(batch, ids)
                    assert ei.value.status == pa.PA_ERR_NO_FREE_BLOCKS
                else:
                    slots, pairs = alloc.append_slots(batch) if ids is None else alloc.append_tokens(batch, ids)
                    assert slots.tolist() == want_slots
                    assert [tuple(p) for p in pairs.tolist()] == want_pairs
            _compare(model, alloc, range(nxt))
            assert alloc.prefix_stats() == model.prefix_stats()
        alloc.close()


def test_beam_search_fork_and_prune_match_model(pa):
    """Beam search as the summary's section 6 describes it, on both the C++
    allocator and the model: each step every new beam forks a surviving
    parent, the old beams are freed (pruned branches return their blocks at
    reference count 0) and every beam appends a token (copy-on-write of a
    shared partial block).  Compared after every step."""
    rng = random.Random(11)
    for width, B in ((2, 4), (4, 16), (6, 1)):
        model = BlockAllocatorModel(400, B)
        alloc = pa.BlockAllocator(400, B)
        for m in (model, alloc):
            m.add_seq(0)
        for _ in range(37):
            assert alloc.append_slots([0])[0].tolist() == model.append_slots([0])[0]
        beams, nxt = [0], 1
        for _ in range(60):
            parents = [rng.choice(beams) for _ in range(width)]
            new = list(range(nxt, nxt + width))
            nxt += width
            for p_, c in zip(parents, new):
                model.fork(p_, c)
                alloc.fork(p_, c)
            for b in beams:
                model.free_seq(b)
                alloc.free_seq(b)
            want_slots, want_pairs = model.append_slots(new)
            slots, pairs = alloc.append_slots(new)
            assert slots.tolist() == want_slots and [tuple(x) for x in pairs.tolist()] == want_pairs
            beams = new
            _compare(model, alloc, beams)
        # only the surviving beams' blocks are held
        held = {b for s in beams for b in model.table(s)}
        assert alloc.num_free() == 400 - len(held)
        alloc.close()


def test_prefix_groups_follow_the_tables(pa):
    """pa_alloc_prefix_groups on beam-search states: the groups cover the
    batch in order, hold 1..max_group sequences, and their prefixes are
    multiples of 16 within every member's length over which every member's
    table equals the first member's; the run rule (extend while the next
    sequence shares a full leading block; prefix = the common filled leading
    blocks) is restated here from its definition."""
    rng = random.Random(5)
    for width, B, max_group in ((8, 16, 8), (5, 4, 3), (6, 32, 8), (4, 1, 2)):
        model = BlockAllocatorModel(600, B)
        alloc = pa.BlockAllocator(600, B)
        for m in (model, alloc):
            m.add_seq(0)
        for _ in range(70):
            model.append_slots([0])
            alloc.append_slots([0])
        beams, nxt = [0], 1
        for step in range(12):
            parents = [rng.choice(beams) for _ in range(width)]
            new = list(range(nxt, nxt + width))
            nxt += width
            for p_, c in zip(parents, new):
                model.fork(p_, c)
                alloc.fork(p_, c)
            for b in beams:
                model.free_seq(b)
                alloc.free_seq(b)
            for _ in range(rng.randint(1, 9)):
                model.append_slots(new)
                alloc.append_slots(new)
            beams = new
            order = beams[:]
            rng.shuffle(order)
            starts, prefixes = alloc.prefix_groups(order, max_group)
            tables = [model.table(s) for s in order]
            lens = [model.length(s) for s in order]
            # the run rule, restated
            want_s, want_p, i = [0], [], 0
            while i < len(order):
                def full(k):
                    return min(lens[k] // B, len(tables[k]))
                common, j = full(i), i + 1
                while j < len(order) and j - i < max_group and common > 0:
                    c, lim = 0, min(common, full(j))
                    while c < lim and tables[j][c] == tables[i][c]:
                        c += 1
                    if c == 0:
                        break
                    common, j = c, j + 1
                want_p.append((common * B if j - i > 1 else 0) // 16 * 16)
                want_s.append(j)
                i = j
            assert starts.tolist() == want_s and prefixes.tolist() == want_p
            # what pa_decode_grouped requires of a group
            for g in range(len(prefixes)):
                g0, g1, pre = int(starts[g]), int(starts[g + 1]), int(prefixes[g])
                assert 1 <= g1 - g0 <= max_group and pre % 16 == 0
                nb = -(-pre // B)
                for k in range(g0, g1):
                    assert pre <= lens[k] and tables[k][:nb] == tables[g0][:nb]
        alloc.close()
    with pytest.raises(pa.PAError):
        pa.BlockAllocator(8, 16).prefix_groups([3])  # unknown sequence


def test_prefix_groups_of_prefix_cached_requests(pa):
    """Requests that reuse a cached prompt through the prefix cache hold its
    blocks too: pa_alloc_prefix_groups groups them (8 at most) with the cached
    prompt's full blocks as the prefix."""
    B, L = 16, 1000
    alloc = pa.BlockAllocator(2000, B, prefix_cache=True)
    prompt = list(range(7, 7 + L))
    assert alloc.add_seq_prefix(0, prompt) == 0  # empty cache: the first request appends its prompt
    for t in prompt:
        alloc.append_tokens([0], [t])
    reused = []
    for r in range(1, 11):
        n0 = alloc.add_seq_prefix(r, prompt + [5000 + r])
        reused.append(n0)
        for t in (prompt + [5000 + r])[n0:]:
            alloc.append_tokens([r], [t])
    assert reused == [(L // B) * B] * 10  # every full prompt block is reused
    starts, prefixes = alloc.prefix_groups(range(11))
    assert starts.tolist() == [0, 8, 11]
    assert prefixes.tolist() == [(L // B) * B] * 2
    alloc.close()


def test_grouped_workspace_sizes(pa):
    for S, H, D, mx in ((64, 40, 128, 1256), (4, 4, 64, 46), (256, 32, 128, 16384)):
        plain = pa.pa_decode_workspace_bytes(S, H, D, mx, 0)
        grouped = pa.pa_decode_grouped_workspace_bytes(S, H, D, mx, 0)
        parts = -(-mx // pa.pa_decode_partition_size(S, H, mx)) + 1  # a prefix adds at most one partition
        assert grouped > plain and grouped >= 4 * S * H * parts * (D + 2) + 4 * S and grouped % 256 == 0
    assert pa.pa_decode_grouped_workspace_bytes(4, 4, 64, 100, 24) == 0
    assert pa.pa_decode_grouped_workspace_bytes(1, 1, 128, (1 << 24) - 16, 16) == 0  # 2^20 partitions with the extra


def test_allocator_errors(pa):
    a = pa.BlockAllocator(2, 4)
    a.add_seq(0)
    with pytest.raises(pa.PAError):
        a.add_seq(0)
    with pytest.raises(pa.PAError):
        a.fork(5, 6)
    with pytest.raises(pa.PAError):
        a.append_slots([0, 0])
    a.add_seq(1)
    a.add_seq(2)
    a.append_slots([0, 1])
    with pytest.raises(pa.PAError) as ei:
        a.append_slots([2])
    assert ei.value.status == pa.PA_ERR_NO_FREE_BLOCKS
    assert a.block_table(2) == ([], 0)
    tables, lens = a.block_tables([0, 1, 2], 3)
    assert tables[2].tolist() == [-1, -1, -1] and lens.tolist() == [1, 1, 0]
    assert a.ref(-1) == -1 and a.ref(2) == -1


def test_shared_prefix_copy_pairs_match_model(pa):
    """The 8-sample shared-prompt flow: 7 copy pairs, the 8th writes in place."""
    B = 16
    model = BlockAllocatorModel(200, B)
    alloc = pa.BlockAllocator(200, B)
    for m in (model, alloc):
        m.add_seq(0)
    for _ in range(1000):
        model.append_slots([0])
        alloc.append_slots([0])
    for c in range(1, 8):
        model.fork(0, c)
        alloc.fork(0, c)
    ws, wp = model.append_slots(list(range(8)))
    gs, gp = alloc.append_slots(list(range(8)))
    assert gs.tolist() == ws and [tuple(p) for p in gp.tolist()] == wp and len(wp) == 7
    _compare(model, alloc, range(8))
