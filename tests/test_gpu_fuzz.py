"""Seeded randomized parity of paged decode and chunked prefill against the
CPU oracle: random shapes (sequences, heads, head_dim 64 / 128, block sizes
that are multiples of 16), dtypes, output dtypes, partition lengths, context
mixes (empty, one token, ragged, page-aligned) and chunk layouts, each case
drawn from a fixed seed so that a failure is reproducible by its index."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import pa_workloads as W
from tests.gpu_common import TORCH_OUT, assert_attn_close, oracle_slots

pytestmark = pytest.mark.gpu

N_DECODE = 100
N_PREFILL = 100


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_35_gb300 as pa

    torch.cuda.set_device(0)
    return pa


def _ctx_mix(rng, n, B):
    """Context lengths mixing the edge cases with random ones."""
    pool = [0, 1, B - 1, B, B + 1, 2 * B, 127, 128, 129, 511, 512, 513]
    out = []
    for _ in range(n):
        if rng.random() < 0.4:
            out.append(int(rng.choice(pool)))
        else:
            out.append(int(rng.integers(1, 1300)))
    return out


@pytest.mark.parametrize("case", range(N_DECODE))
def test_decode_random_cases(pa, case):
    rng = np.random.default_rng(1000 + case)
    D = int(rng.choice([64, 128]))
    B = int(rng.choice([16, 32, 48, 64, 128, 256]))
    H = int(rng.integers(1, 6))
    S = int(rng.integers(1, 9))
    dtype = str(rng.choice(["f16", "bf16"]))
    out_dtype = str(rng.choice(["f32", dtype]))
    P = int(rng.choice([0, 16, 64, 112, 512, 1024]))
    ctx = torch.tensor(_ctx_mix(rng, S, B), dtype=torch.int32)
    w = W._decode_workload(f"fuzz{case}", ctx, ctx - 1 + (ctx == 0).to(torch.int32), H, D, B, dtype,
                           seed=50 + case)
    dev = torch.device("cuda")
    mx = max(1, int(ctx.max()))
    out = torch.full((S, H, D), float("nan"), dtype=TORCH_OUT[out_dtype], device=dev)
    ws = pa.decode_workspace(S, H, D, mx, P)
    err = pa.new_error_flag()
    pa.pa_decode(out, w.q.to(dev), w.k_pool.to(dev), w.v_pool.to(dev), w.block_tables.to(dev), ctx.to(dev), mx,
                 w.scale, ws, err, partition_size=P)
    assert pa.pa_get_error(err) == 0
    ref = oracle.decode(w.q, w.k_pool, w.v_pool, w.block_tables, ctx, B, w.scale, dtype)
    assert_attn_close(out, ref, out_dtype, f"case {case}: S={S} H={H} D={D} B={B} {dtype} P={P} ctx={ctx.tolist()}")


@pytest.mark.parametrize("case", range(10))
def test_decode_random_cases_with_a_bad_page(pa, case):
    """One table entry of one sequence out of range: the call flags it and the
    sequence's output is the oracle over the same sequence without that page
    (its entry taken out of the table, its context shorter by the page's
    tokens); the other sequences are unaffected."""
    rng = np.random.default_rng(3000 + case)
    D = int(rng.choice([64, 128]))
    B = int(rng.choice([16, 32, 48, 64]))
    H = int(rng.integers(1, 4))
    S = int(rng.integers(2, 6))
    dtype = str(rng.choice(["f16", "bf16"]))
    P = int(rng.choice([0, 16, 64, 512]))
    ctx = torch.tensor([int(rng.integers(B + 1, 900)) for _ in range(S)], dtype=torch.int32)
    w = W._decode_workload(f"badpage{case}", ctx, ctx - 1, H, D, B, dtype, seed=90 + case)
    s_bad = int(rng.integers(0, S))
    n_pages = (int(ctx[s_bad]) + B - 1) // B
    j = int(rng.integers(0, n_pages))
    tables = w.block_tables.clone()
    tables[s_bad, j] = w.num_blocks + int(rng.integers(0, 5))
    dev = torch.device("cuda")
    mx = int(ctx.max())
    out = torch.full((S, H, D), float("nan"), dtype=torch.float32, device=dev)
    ws = pa.decode_workspace(S, H, D, mx, P)
    err = pa.new_error_flag()
    pa.pa_decode(out, w.q.to(dev), w.k_pool.to(dev), w.v_pool.to(dev), tables.to(dev), ctx.to(dev), mx, w.scale, ws,
                 err, partition_size=P)
    assert pa.pa_get_error(err) == pa.PA_FLAG_BAD_BLOCK
    kept = w.block_tables.clone()
    row = w.block_tables[s_bad].tolist()
    kept[s_bad] = torch.tensor(row[:j] + row[j + 1:] + row[:1], dtype=kept.dtype)
    shorter = ctx.clone()
    shorter[s_bad] = int(ctx[s_bad]) - (min((j + 1) * B, int(ctx[s_bad])) - j * B)
    ref = oracle.decode(w.q, w.k_pool, w.v_pool, kept, shorter, B, w.scale, dtype)
    assert_attn_close(out, ref, "f32", f"case {case}: S={S} H={H} D={D} B={B} {dtype} P={P} bad page {j} of seq {s_bad}")


@pytest.mark.parametrize("case", range(N_PREFILL))
def test_prefill_random_cases(pa, case):
    rng = np.random.default_rng(2000 + case)
    D = int(rng.choice([64, 128]))
    B = int(rng.choice([16, 32, 48, 80, 128, 256]))
    H = int(rng.integers(1, 4))
    C = int(rng.integers(1, 5))
    dtype = str(rng.choice(["f16", "bf16"]))
    out_dtype = str(rng.choice(["f32", dtype]))
    lens = [int(rng.choice([1, 2, 127, 128, 129, int(rng.integers(1, 400))])) for _ in range(C)]
    before = [int(rng.choice([0, 1, B, int(rng.integers(0, 700))])) for _ in range(C)]
    m = W.small_prefill(chunk_lens=tuple(lens), ctx_before=tuple(before), H=H, D=D, B=B, dtype=dtype,
                        seed=70 + case)
    w = m.decode
    dev = torch.device("cuda")
    kp, vp = w.k_pool.to(dev), w.v_pool.to(dev)
    seq_idx = np.concatenate([np.full(n, c) for c, n in enumerate(lens)])
    pos = np.concatenate([np.arange(c0, c0 + n) for c0, n in zip(before, lens)])
    slots = pa.pa_slot_mapping(m.chunk_tables, seq_idx, pos, B)
    err = pa.new_error_flag()
    pa.pa_reshape_and_cache(m.chunk_k.to(dev), m.chunk_v.to(dev), kp, vp, torch.from_numpy(slots).to(dev), err)
    T = sum(lens)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    out = torch.full((T, H, D), float("nan"), dtype=TORCH_OUT[out_dtype], device=dev)
    pa.pa_prefill_chunk(out, m.chunk_q.to(dev), cu.to(dev), m.ctx_before.to(dev), kp, vp, m.chunk_tables.to(dev),
                        max(lens), w.scale, err)
    assert pa.pa_get_error(err) == 0
    kb, vb = oracle.pool_bits(w.k_pool), oracle.pool_bits(w.v_pool)
    oracle.reshape_and_cache(m.chunk_k, m.chunk_v, kb, vb, oracle_slots(m.chunk_tables, seq_idx, pos, B), B)
    ref = oracle.prefill(m.chunk_q, cu, m.ctx_before, kb, vb, m.chunk_tables, B, w.scale, dtype)
    assert_attn_close(out, ref, out_dtype,
                      f"case {case}: C={C} H={H} D={D} B={B} {dtype} lens={lens} before={before}")
