"""pa_decode_grouped against the oracle.

Groups of sequences share the blocks of a common prefix (the parallel samples
or beams of one prompt, [summary] section 6, Figures 9-10, and [blog] "Prefix Sharing"):
their tables hold the same block ids over the prefix.  The grouped call reads
each prefix once for its group; the oracle reassembles every sequence on its
own from the same tables and attends over it in fp64, so the grouping is
checked against the plain definition, per sequence, within the gate.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import pa_workloads as W
from oracle.alloc_model import BlockAllocatorModel
from tests.gpu_common import TORCH_OUT, assert_attn_close, bits_equal

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_35_gb300 as pa

    torch.cuda.set_device(0)
    return pa


def grouped_case(groups, H, D, B, dtype, seed, singles=()):
    """groups: [(prefix tokens, [member contexts])]; singles: contexts of
    sequences outside every group.  Member tables hold the same blocks over
    the prefix's blocks, then blocks of their own; block ids are a seeded
    permutation of the pool.  Returns host tensors and the group arrays."""
    ctxs, tables_rows, starts, prefixes = [], [], [0], []
    need = 0
    for pre, members in groups:
        nsh = -(-pre // B)
        need += nsh + sum(-(-c // B) - nsh for c in members)
    need += sum(-(-c // B) for c in singles)
    NB = need + 7
    perm = W.randint(0, 1 << 30, NB, seed + 1).argsort().tolist()
    nxt = 0

    def take(k):
        nonlocal nxt
        ids = perm[nxt:nxt + k]
        nxt += k
        return ids

    for pre, members in groups:
        shared = take(-(-pre // B))
        for c in members:
            assert c >= pre
            tables_rows.append(shared + take(-(-c // B) - len(shared)))
            ctxs.append(c)
        starts.append(starts[-1] + len(members))
        prefixes.append(pre)
    for c in singles:
        tables_rows.append(take(-(-c // B)))
        ctxs.append(c)
    S = len(ctxs)
    MB = max(1, max(len(r) for r in tables_rows))
    tables = torch.full((S, MB), -1, dtype=torch.int32)
    for s, r in enumerate(tables_rows):
        tables[s, :len(r)] = torch.tensor(r, dtype=torch.int32)
    dt = DT[dtype]
    q = W.normal((S, H, D), seed + 2, dt)
    kp = W.normal((NB, H, B, D), seed + 3, dt)
    vp = W.normal((NB, H, B, D), seed + 4, dt)
    return (q, kp, vp, tables, torch.tensor(ctxs, dtype=torch.int32), torch.tensor(starts, dtype=torch.int32),
            torch.tensor(prefixes, dtype=torch.int32))


def oracle_ref(case, dtype):
    q, kp, vp, tables, ctx, _, _ = case
    D = q.shape[2]
    return oracle.decode(q, kp, vp, tables, ctx, kp.shape[2], 1 / np.sqrt(D), dtype)


def grouped_call(pa, case, out_dtype="f32", partition=0, starts=None, prefixes=None):
    """Runs pa_decode_grouped; returns (out, device error flags)."""
    q, kp, vp, tables, ctx, gs, gp = case
    gs = gs if starts is None else starts
    gp = gp if prefixes is None else prefixes
    dev = torch.device("cuda")
    S, H, D = q.shape
    mx = int(ctx.max())
    out = torch.empty(S, H, D, dtype=TORCH_OUT[out_dtype], device=dev)
    ws = pa.decode_grouped_workspace(S, H, D, mx, partition, device=dev)
    err = pa.new_error_flag(dev)
    pa.pa_decode_grouped(out, q.to(dev), kp.to(dev), vp.to(dev), tables.to(dev), ctx.to(dev), mx, 1 / np.sqrt(D),
                         gs.to(dev), gp.to(dev), ws, err, partition_size=partition)
    torch.cuda.synchronize()
    flags = int(err.item())
    return out, flags


# prefixes: none, one tile, whole blocks, longer than a partition; members
# ending at the prefix, one token past it, and far past it
MIXED_GROUPS = [
    (0, [40, 41]),
    (16, [16, 17, 100]),
    (256, [256, 257, 300, 511, 512, 513, 700, 1029]),
    (1024, [1024, 1100, 1500, 2047, 2048, 2100]),
    (96, [500]),
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B", [16, 32, 256])
def test_grouped_matches_the_oracle(pa, dtype, D, B):
    case = grouped_case(MIXED_GROUPS, H=3, D=D, B=B, dtype=dtype, seed=11, singles=(1, 33, 700))
    out, flags = grouped_call(pa, case)
    assert flags == 0
    assert_attn_close(out, oracle_ref(case, dtype), "f32", f"grouped {dtype} D={D} B={B}")


@pytest.mark.parametrize("partition", [16, 64, 256, 512, 1024])
def test_grouped_partition_sizes(pa, partition):
    case = grouped_case(MIXED_GROUPS, H=2, D=128, B=16, dtype="f16", seed=12, singles=(5,))
    out, flags = grouped_call(pa, case, partition=partition)
    assert flags == 0
    assert_attn_close(out, oracle_ref(case, "f16"), "f32", f"grouped, partition {partition}")


@pytest.mark.parametrize("out_dtype", ["f16", "bf16"])
def test_grouped_output_dtypes(pa, out_dtype):
    case = grouped_case(MIXED_GROUPS[:3], H=4, D=128, B=16, dtype="bf16", seed=13)
    out, flags = grouped_call(pa, case, out_dtype=out_dtype)
    assert flags == 0
    assert_attn_close(out, oracle_ref(case, "bf16"), out_dtype, f"grouped, {out_dtype} output")


def test_groups_without_prefixes(pa):
    """Groups whose prefix is 0, and sequences outside every group: each
    sequence is decoded on its own (one-column units)."""
    case = grouped_case([(0, [40, 700, 1029]), (0, [1, 16])], H=3, D=128, B=16, dtype="f16", seed=14,
                        singles=(17, 2048))
    out, flags = grouped_call(pa, case)
    assert flags == 0
    assert_attn_close(out, oracle_ref(case, "f16"), "f32", "no shared prefixes")
    q, kp, vp, tables, ctx, _, _ = case
    none = (q, kp, vp, tables, ctx, torch.zeros(1, dtype=torch.int32), torch.zeros(0, dtype=torch.int32))
    out0, flags = grouped_call(pa, none)  # num_groups == 0: pa_decode itself
    assert flags == 0
    assert_attn_close(out0, oracle_ref(case, "f16"), "f32", "no groups at all")


def test_grouped_is_deterministic(pa):
    case = grouped_case(MIXED_GROUPS, H=3, D=128, B=16, dtype="bf16", seed=15)
    a, fa = grouped_call(pa, case)
    b, fb = grouped_call(pa, case)
    assert fa == 0 and fb == 0
    assert torch.equal(a, b)


def test_single_key_prefix_rows_are_v0(pa):
    """A group whose members attend over 16 prefix tokens of which one key
    dominates returns that key's V row for every member."""
    case = list(grouped_case([(16, [16, 16, 16])], H=1, D=128, B=16, dtype="f16", seed=16))
    q, kp, vp, tables, ctx = case[:5]
    blk = int(tables[0, 0])
    kp[blk, 0] = 0
    kp[blk, 0, 5] = 8.0  # with every query all ones, key 5 scores 8 * sqrt(128) above the others
    q[:, 0] = 1.0
    out, flags = grouped_call(pa, tuple(case))
    assert flags == 0
    ref = oracle_ref(tuple(case), "f16")
    assert_attn_close(out, ref, "f32", "dominant key")
    assert np.abs(ref[:, 0] - vp[blk, 0, 5].double().numpy()).max() < 1e-9


def test_bad_groups_are_flagged_and_decoded_whole(pa):
    """A group that breaks a rule raises PA_FLAG_BAD_GROUP; its members are
    decoded whole and every output still matches the oracle."""
    case = grouped_case([(256, [300, 400]), (128, [200, 250, 260])], H=2, D=128, B=16, dtype="f16", seed=17)
    ref = oracle_ref(case, "f16")
    q, kp, vp, tables, ctx, gs, gp = case
    # the second member's table points one prefix block at another block that
    # holds the same bits: same sequences, but not the same block ids
    used = set(tables.flatten().tolist())
    spare = next(b for b in range(int(kp.shape[0])) if b not in used)
    kp2, vp2, t2 = kp.clone(), vp.clone(), tables.clone()
    kp2[spare], vp2[spare] = kp[int(tables[0, 3])], vp[int(tables[0, 3])]
    t2[1, 3] = spare
    out, flags = grouped_call(pa, (q, kp2, vp2, t2, ctx, gs, gp))
    assert flags & pa.PA_FLAG_BAD_GROUP
    assert_attn_close(out, ref, "f32", "a member table that differs over the prefix")
    for name, starts, prefixes in [
        ("prefix above a member's context", None, torch.tensor([256, 208], dtype=torch.int32)),
        ("prefix not a multiple of 16", None, torch.tensor([256, 120], dtype=torch.int32)),
        ("range past the batch", torch.tensor([0, 2, 9], dtype=torch.int32), None),
        ("empty range", torch.tensor([0, 2, 2], dtype=torch.int32), None),
    ]:
        out, flags = grouped_call(pa, case, starts=starts, prefixes=prefixes)
        assert flags & pa.PA_FLAG_BAD_GROUP, name
        assert_attn_close(out, ref, "f32", name)


def test_groups_of_more_than_eight_are_refused(pa):
    case = grouped_case([(64, [64 + i for i in range(9)])], H=1, D=64, B=16, dtype="f16", seed=18)
    out, flags = grouped_call(pa, case)
    assert flags & pa.PA_FLAG_BAD_GROUP
    assert_attn_close(out, oracle_ref(case, "f16"), "f32", "nine members")


def test_parallel_sampling_workload_grouped(pa):
    """The 8 prompts x 8 samples workload built through the library's
    allocator (fork, copy-on-write of the partial prompt block, suffixes),
    grouped by pa_alloc_prefix_groups; every sequence against the oracle."""
    sc = W.shared_prefix()
    dev = torch.device("cuda")
    P, N, L, B = sc.num_prompts, sc.samples, sc.prompt_len, sc.block_size
    H, D = sc.num_heads, sc.head_dim
    n = P * N
    alloc = pa.BlockAllocator(sc.num_blocks, B)
    for p in range(P):
        alloc.add_seq(p * N)
    prompt_slots = np.stack([alloc.append_slots([p * N for p in range(P)])[0] for _ in range(L)], axis=1)
    for p in range(P):
        for j in range(1, N):
            alloc.fork(p * N, p * N + j)
    kp, vp = sc.pool_init_k.to(dev), sc.pool_init_v.to(dev)
    err = pa.new_error_flag()
    pa.pa_reshape_and_cache(sc.prompt_k.reshape(P * L, H, D).to(dev), sc.prompt_v.reshape(P * L, H, D).to(dev), kp, vp,
                            torch.from_numpy(prompt_slots.reshape(-1)).to(dev), err)
    suffix = sc.suffix_lens.tolist()
    ms = sc.suffix_k.shape[1]
    suffix_slots = np.full((n, ms), -1, dtype=np.int64)
    for r in range(max(suffix)):
        active = [s for s in range(n) if suffix[s] > r]
        slots, pairs = alloc.append_slots(active)
        suffix_slots[active, r] = slots
        if len(pairs):
            pa.pa_copy_blocks(kp, vp, torch.from_numpy(pairs).to(dev), err)
    pa.pa_reshape_and_cache(sc.suffix_k.reshape(n * ms, H, D).to(dev), sc.suffix_v.reshape(n * ms, H, D).to(dev),
                            kp, vp, torch.from_numpy(suffix_slots.reshape(-1)).to(dev), err)
    assert pa.pa_get_error(err) == 0
    mb = max(len(alloc.block_table(s)[0]) for s in range(n))
    tables, lens = alloc.block_tables(range(n), mb)
    starts, prefixes = alloc.prefix_groups(range(n))
    # the prompt's full blocks (the partial one was copied on write) are shared
    assert starts.tolist() == list(range(0, n + 1, N))
    assert prefixes.tolist() == [(L // B) * B] * P
    mx = int(lens.max())
    out = torch.empty(n, H, D, dtype=torch.float16, device=dev)
    ws = pa.decode_grouped_workspace(n, H, D, mx, device=dev)
    pa.pa_decode_grouped(out, sc.q.to(dev), kp, vp, torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev),
                         mx, sc.scale, torch.from_numpy(starts).to(dev), torch.from_numpy(prefixes).to(dev), ws, err)
    assert pa.pa_get_error(err) == 0

    # the oracle: its own allocator model, scatter, copies and attention
    model = BlockAllocatorModel(sc.num_blocks, B)
    for p in range(P):
        model.add_seq(p * N)
    o_prompt = np.stack([model.append_slots([p * N for p in range(P)])[0] for _ in range(L)], axis=1)
    for p in range(P):
        for j in range(1, N):
            model.fork(p * N, p * N + j)
    kb, vb = oracle.pool_bits(sc.pool_init_k), oracle.pool_bits(sc.pool_init_v)
    oracle.reshape_and_cache(sc.prompt_k.reshape(P * L, H, D), sc.prompt_v.reshape(P * L, H, D), kb, vb,
                             o_prompt.reshape(-1), B)
    o_suffix = np.full((n, ms), -1, dtype=np.int64)
    for r in range(max(suffix)):
        active = [s for s in range(n) if suffix[s] > r]
        slots, pairs = model.append_slots(active)
        o_suffix[active, r] = slots
        if pairs:
            oracle.copy_blocks(kb, vb, pairs, B)
    oracle.reshape_and_cache(sc.suffix_k.reshape(n * ms, H, D), sc.suffix_v.reshape(n * ms, H, D), kb, vb,
                             o_suffix.reshape(-1), B)
    o_tables = np.full((n, mb), -1, dtype=np.int32)
    for s in range(n):
        o_tables[s, :len(model.table(s))] = model.table(s)
    o_lens = np.array([model.length(s) for s in range(n)], dtype=np.int32)
    assert np.array_equal(tables, o_tables) and np.array_equal(lens, o_lens)
    assert bits_equal(kp, kb) and bits_equal(vp, vb)
    ref = oracle.decode(sc.q, kb, vb, o_tables, o_lens, B, sc.scale, "f16")
    assert_attn_close(out, ref, "f16", "grouped parallel-sampling decode")


def test_bad_block_in_a_shared_prefix(pa):
    """A block id out of range inside a group's shared prefix (in every
    member's table, so the group stays valid) raises PA_FLAG_BAD_BLOCK and
    leaves that 16-token tile out of each member's sum; other sequences are
    untouched."""
    case = grouped_case([(64, [100, 130]), (32, [50, 60])], H=2, D=128, B=16, dtype="f16", seed=19, singles=(40,))
    q, kp, vp, tables, ctx, gs, gp = case
    NB = int(kp.shape[0])
    bad = tables.clone()
    bad[0, 1] = NB + 5
    bad[1, 1] = NB + 5
    out, flags = grouped_call(pa, (q, kp, vp, bad, ctx, gs, gp))
    assert flags == pa.PA_FLAG_BAD_BLOCK
    assert torch.isfinite(out).all()
    ref = oracle_ref(case, "f16")
    assert_attn_close(out[2:], ref[2:], "f32", "sequences without the bad entry")
    # the group's members without their second page: the oracle over the
    # tables with that entry taken out and 16 fewer tokens
    kept, shorter = tables.clone(), ctx.clone()
    for s in (0, 1):
        row = tables[s].tolist()
        kept[s] = torch.tensor(row[:1] + row[2:] + row[:1], dtype=kept.dtype)
        shorter[s] -= 16
    ref2 = oracle.decode(q, kp, vp, kept, shorter, 16, 1 / np.sqrt(128), "f16")
    assert_attn_close(out[:2], ref2[:2], "f32", "members whose shared second page is out of range")


N_FUZZ = 60


@pytest.mark.parametrize("case", range(N_FUZZ))
def test_grouped_random_cases(pa, case):
    """Seeded random layouts: 1-4 groups of 1-8 sequences with prefixes of 0-640
    tokens (multiples of 16), members ending at the prefix or past it, sequences
    outside every group (empty ones included), both dtypes, head_dim 64 / 128,
    block sizes that are multiples of 16, partition lengths, output dtypes; the
    output starts as NaN so that an unwritten row fails."""
    rng = np.random.default_rng(3000 + case)
    D = int(rng.choice([64, 128]))
    B = int(rng.choice([16, 32, 48, 64, 128, 256]))
    H = int(rng.integers(1, 6))
    dtype = str(rng.choice(["f16", "bf16"]))
    out_dtype = str(rng.choice(["f32", dtype]))
    P = int(rng.choice([0, 16, 64, 112, 512, 1024]))
    groups = []
    for _ in range(int(rng.integers(1, 5))):
        pre = 16 * int(rng.integers(0, 41))
        members = [pre + (0 if rng.random() < 0.2 else int(rng.integers(1, 700))) for _ in range(int(rng.integers(1, 9)))]
        groups.append((pre, members))
    singles = tuple(int(rng.choice([0, 1, 17, int(rng.integers(1, 900))])) for _ in range(int(rng.integers(0, 4))))
    case_t = grouped_case(groups, H=H, D=D, B=B, dtype=dtype, seed=4000 + case, singles=singles)
    q, kp, vp, tables, ctx, gs, gp = case_t
    dev = torch.device("cuda")
    S = q.shape[0]
    mx = max(1, int(ctx.max()))
    out = torch.full((S, H, D), float("nan"), dtype=TORCH_OUT[out_dtype], device=dev)
    ws = pa.decode_grouped_workspace(S, H, D, mx, P, device=dev)
    err = pa.new_error_flag(dev)
    pa.pa_decode_grouped(out, q.to(dev), kp.to(dev), vp.to(dev), tables.to(dev), ctx.to(dev), mx, 1 / np.sqrt(D),
                         gs.to(dev), gp.to(dev), ws, err, partition_size=P)
    assert pa.pa_get_error(err) == 0, f"case {case}"
    assert_attn_close(out, oracle_ref(case_t, dtype), out_dtype, f"grouped random case {case}")
