"""The KV-memory waste simulator: its contiguous allocator, reservations and
waste accounting against hand-worked cases, the ordering of the policies on
a random trace, and the sharing measurements on cases worked by hand."""
from __future__ import annotations

import pytest

from paged_kv_cache_35_gb300 import memsim
from paged_kv_cache_35_gb300.memsim import FirstFit, Request


def test_first_fit_places_lowest_hole_and_merges_on_free():
    ff = FirstFit(100)
    assert ff.alloc(30) == 0 and ff.alloc(30) == 30 and ff.alloc(30) == 60
    assert ff.alloc(20) is None  # 10 free
    ff.free(30, 30)
    assert ff.holes == [(30, 30), (90, 10)]
    assert ff.alloc(40) is None and ff.free_total() == 40  # 40 free, no 40-slot hole
    ff.free(0, 30)
    assert ff.holes == [(0, 60), (90, 10)]
    ff.free(60, 30)
    assert ff.holes == [(0, 100)]


def test_reservations_of_the_three_baselines():
    r = Request(0, prompt=100, output=37)
    assert memsim.reservation("orca_max", r, 2048) == 2048
    assert memsim.reservation("orca_pow2", r, 2048) == 100 + 64
    assert memsim.reservation("orca_pow2", Request(1, 10, 64), 2048) == 74
    assert memsim.reservation("orca_pow2", Request(2, 2000, 40), 2048) == 2048  # capped
    assert memsim.reservation("orca_oracle", r, 2048) == 137


def test_accounting_by_hand_orca_max_and_paged():
    """A: prompt 4, output 2; B: prompt 1, output 3; max_len 16, 32 slots.
    Orca-Max: regions of 16 each.  After step 1 A holds 5 tokens (final 6),
    B 2 (final 4): reserved (6-5)+(4-2) = 3, internal (16-6)+(16-4) = 22.
    Step 2: 6 and 3 tokens, reserved 0+1, internal 22; A leaves.  Step 3: B
    holds 4, reserved 0, internal 12.  Paged, blocks of 4: step 1 uses
    2+1 blocks for 7 tokens (5 unfilled), step 2 the same 12 slots for 9
    tokens (3), step 3 one block for 4 tokens (0)."""
    trace = [Request(0, 4, 2), Request(1, 1, 3)]
    m = memsim.simulate("orca_max", trace, 32, max_len=16)
    assert (m.steps, m.completed, m.batch_steps) == (3, 2, 5)
    assert (m.token_slot_steps, m.reserved_steps, m.internal_steps, m.external_steps) == (20, 4, 56, 0)
    p = memsim.simulate("paged", trace, 32, block_size=4, max_len=16)
    assert (p.steps, p.completed, p.preemptions) == (3, 2, 0)
    assert (p.token_slot_steps, p.reserved_steps, p.internal_steps, p.external_steps) == (20, 0, 8, 0)


def test_external_fragmentation_counts_free_space_that_cannot_be_used():
    """Orca-Oracle, max_len 20.

    Case 1 (40 slots): A (10+2), B (5+3) and C (10+10) take [0,12), [12,20)
    and [20,40); D (6+14) waits.  While A and B run nothing is free; A leaves
    after step 2, leaving a 12-slot hole, too small in total for D (20), so
    nothing counts; B leaves after step 3 and D then fits [0,20).

    Case 2 (30 slots): E (2+2), F (2+4), G (4+14) take [0,4), [4,10),
    [10,28); H (3+3) needs 6 and waits with 2 slots free (less than 6: not
    counted).  E leaves after step 2: 4 + 2 = 6 slots are free but in two
    holes, so steps 3 and 4 count 6 each; F leaves after step 4 and H fits
    [0,10) at step 5."""
    trace = [Request(0, 10, 2), Request(1, 5, 3), Request(2, 10, 10), Request(3, 6, 14)]
    m = memsim.simulate("orca_oracle", trace, 40, max_len=20)
    assert m.external_steps == 0 and m.completed == 4
    trace = [Request(0, 2, 2), Request(1, 2, 4), Request(2, 4, 14), Request(3, 3, 3)]
    m = memsim.simulate("orca_oracle", trace, 30, max_len=20)
    assert m.external_steps == 12 and m.completed == 4


def test_policies_order_on_a_long_tailed_trace():
    tr = memsim.synthetic_trace("long_tail", 150, seed=3)
    frac = {p: memsim.simulate(p, tr, 16384).summary()["token_fraction"] for p in memsim.POLICIES}
    assert frac["orca_max"] < frac["orca_pow2"] < frac["orca_oracle"] < frac["paged"]
    assert frac["paged"] > 0.9


def test_sharing_measurements_by_hand():
    # prompt of 2 full blocks, two samples of 16 tokens: shared peak 2 + 2
    # blocks, unshared 3 + 3
    x = memsim.sharing_parallel_sampling(2, 32, [16, 16], block_size=16)
    assert (x["shared_peak_blocks"], x["unshared_blocks"]) == (4, 6)
    assert x["saving"] == pytest.approx(1 / 3)
    # one sample, one beam: nothing to share
    assert memsim.sharing_parallel_sampling(1, 20, [5], 16)["saving"] == 0.0
    assert memsim.sharing_beam_search(1, 20, 30, 0, 16)["saving"] == 0.0
    # more beams share more
    s = [memsim.sharing_beam_search(w, 100, 60, 1, 16)["saving"] for w in (2, 4, 6)]
    assert 0 < s[0] < s[1] < s[2] < 1
