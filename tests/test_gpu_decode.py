"""GPU parity of the slot scatter, the block copy and paged decode attention
against the CPU oracle (small and ragged cases, every dtype combination,
several partition sizes, the bit-exact special cases and the error flags)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import pa_workloads as W
from tests.gpu_common import TORCH_OUT, assert_attn_close, bits_equal, oracle_slots

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_35_gb300 as pa

    torch.cuda.set_device(0)
    return pa


def run_decode(pa, w, ctx=None, out_dtype="f32", partition_size=0, tables=None, kp=None, vp=None, q=None):
    dev = torch.device("cuda")
    ctx = w.context_lens if ctx is None else ctx
    tables = w.block_tables if tables is None else tables
    kp = w.k_pool.to(dev) if kp is None else kp
    vp = w.v_pool.to(dev) if vp is None else vp
    q = w.q.to(dev) if q is None else q
    mx = max(1, int(ctx.max()))
    out = torch.full((w.num_seqs, w.num_heads, w.head_dim), float("nan"), dtype=TORCH_OUT[out_dtype], device=dev)
    ws = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, mx, partition_size)
    err = pa.new_error_flag()
    pa.pa_decode(out, q, kp, vp, tables.to(dev), ctx.to(dev), mx, w.scale, ws, err, partition_size=partition_size)
    flags = pa.pa_get_error(err)
    return out, flags


def oracle_decode(w, ctx=None, tables=None, kp=None, vp=None):
    return oracle.decode(w.q, w.k_pool if kp is None else kp, w.v_pool if vp is None else vp,
                         w.block_tables if tables is None else tables, w.context_lens if ctx is None else ctx,
                         w.block_size, w.scale, w.dtype)


# -- scatter and copy ---------------------------------------------------------------

def test_reshape_and_cache_is_bit_exact(pa):
    w = W.tiny_decode()
    dev = torch.device("cuda")
    kp, vp = w.k_pool.to(dev), w.v_pool.to(dev)
    slots = pa.pa_slot_mapping(w.block_tables, np.arange(w.num_seqs), w.new_pos, w.block_size)
    sm = torch.from_numpy(slots).to(dev)
    sm[1] = -1  # padding token: skipped
    err = pa.new_error_flag()
    pa.pa_reshape_and_cache(w.k_new.to(dev), w.v_new.to(dev), kp, vp, sm, err)
    assert pa.pa_get_error(err) == 0
    kb, vb = oracle.pool_bits(w.k_pool), oracle.pool_bits(w.v_pool)
    oslots = oracle_slots(w.block_tables, range(w.num_seqs), w.new_pos, w.block_size)
    oslots[1] = -1
    oracle.reshape_and_cache(w.k_new, w.v_new, kb, vb, oslots, w.block_size)
    assert bits_equal(kp, kb) and bits_equal(vp, vb)


def test_reshape_and_cache_flags_slot_outside_pool(pa):
    w = W.tiny_decode()
    dev = torch.device("cuda")
    kp, vp = w.k_pool.to(dev), w.v_pool.to(dev)
    sm = torch.tensor([0, w.num_blocks * w.block_size, 5, -7], dtype=torch.int64, device=dev)
    err = pa.new_error_flag()
    pa.pa_reshape_and_cache(w.k_new.to(dev), w.v_new.to(dev), kp, vp, sm, err)
    assert pa.pa_get_error(err) == pa.PA_FLAG_BAD_SLOT
    kb, vb = oracle.pool_bits(w.k_pool), oracle.pool_bits(w.v_pool)
    oracle.reshape_and_cache(w.k_new[[0, 2]], w.v_new[[0, 2]], kb, vb, np.array([0, 5]), w.block_size)
    assert bits_equal(kp, kb) and bits_equal(vp, vb)


@pytest.mark.parametrize("dtype,B", [("f16", 16), ("bf16", 256)])
def test_copy_blocks_is_bit_exact(pa, dtype, B):
    dt = W.DTYPES[dtype]
    NB, H, D = 24, 5, 128
    kp0 = W.normal((NB, H, B, D), 31, dt)
    vp0 = W.normal((NB, H, B, D), 32, dt)
    pairs = torch.tensor([[3, 17], [4, 0], [23, 9], [9 + 0, 11]], dtype=torch.int32)
    pairs = pairs[[0, 1, 2]]  # sources and destinations disjoint
    dev = torch.device("cuda")
    kp, vp = kp0.to(dev), vp0.to(dev)
    err = pa.new_error_flag()
    pa.pa_copy_blocks(kp, vp, pairs.to(dev), err)
    assert pa.pa_get_error(err) == 0
    kb, vb = oracle.pool_bits(kp0), oracle.pool_bits(vp0)
    oracle.copy_blocks(kb, vb, pairs.numpy(), B)
    assert bits_equal(kp, kb) and bits_equal(vp, vb)
    bad = torch.tensor([[1, NB]], dtype=torch.int32, device=dev)
    pa.pa_copy_blocks(kp, vp, bad, err)
    assert pa.pa_get_error(err) == pa.PA_FLAG_BAD_BLOCK
    assert bits_equal(kp, kb) and bits_equal(vp, vb)


# -- decode parity -----------------------------------------------------------------

def test_tiny_config_decode_scatter_decode(pa):
    """4 sequences, contexts {1,16,17,45}, 32-block pool: decode, write the
    next token of each sequence, decode again over one more token."""
    w = W.tiny_decode()
    dev = torch.device("cuda")
    kp, vp = w.k_pool.to(dev), w.v_pool.to(dev)
    out, flags = run_decode(pa, w, kp=kp, vp=vp, out_dtype="f16")
    assert flags == 0
    assert_attn_close(out, oracle_decode(w), "f16", "tiny decode")
    slots = pa.pa_slot_mapping(w.block_tables, np.arange(4), w.new_pos, w.block_size)
    err = pa.new_error_flag()
    pa.pa_reshape_and_cache(w.k_new.to(dev), w.v_new.to(dev), kp, vp, torch.from_numpy(slots).to(dev), err)
    assert pa.pa_get_error(err) == 0
    ctx2 = w.context_lens + 1
    out2, flags = run_decode(pa, w, ctx=ctx2, kp=kp, vp=vp, out_dtype="f32")
    assert flags == 0
    kb, vb = oracle.pool_bits(w.k_pool), oracle.pool_bits(w.v_pool)
    oracle.reshape_and_cache(w.k_new, w.v_new, kb, vb, oracle_slots(w.block_tables, range(4), w.new_pos, 16), 16)
    assert_attn_close(out2, oracle_decode(w, ctx=ctx2, kp=kb, vp=vb), "f32", "tiny decode after write")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("out_dtype", ["f16", "bf16", "f32"])
def test_decode_small_ragged(pa, dtype, D, out_dtype):
    w = W.small_decode(dtype=dtype, D=D, H=3)
    out, flags = run_decode(pa, w, out_dtype=out_dtype)
    assert flags == 0
    assert_attn_close(out, oracle_decode(w), out_dtype, f"{dtype} D={D} -> {out_dtype}")


@pytest.mark.parametrize("P", [16, 64, 112, 512, 1024])
def test_decode_partition_sizes_agree(pa, P):
    w = W.small_decode(ctx=(1, 17, 255, 256, 257, 1029, 2100), H=2, dtype="bf16")
    out, flags = run_decode(pa, w, out_dtype="f32", partition_size=P)
    assert flags == 0
    assert_attn_close(out, oracle_decode(w), "f32", f"partition {P}")


@pytest.mark.parametrize("B", [16, 32, 48, 256, 1024, 4096])
def test_decode_block_sizes(pa, B):
    w = W.small_decode(ctx=(1, 31, 300, 777, 5000), H=2, B=B, dtype="f16")
    out, flags = run_decode(pa, w, out_dtype="f32")
    assert flags == 0
    assert_attn_close(out, oracle_decode(w), "f32", f"block {B}")


def test_decode_context_one_is_v0_bitwise(pa):
    w = W.small_decode(ctx=(1, 1, 1), H=4, D=128, dtype="bf16")
    out, flags = run_decode(pa, w, out_dtype="bf16")
    assert flags == 0
    for s in range(3):
        blk = int(w.block_tables[s, 0])
        assert torch.equal(out[s].cpu(), w.v_pool[blk, :, 0, :])


def test_decode_one_hot_key_locates_every_position_bitwise(pa):
    """k_j = 12 q for one position j makes every other weight underflow to 0
    in fp32: the output must be exactly the V row the oracle finds at j."""
    w = W.small_decode(ctx=(45, 45), H=2, D=64, dtype="f16")
    dev = torch.device("cuda")
    vp = w.v_pool.to(dev)
    for j in range(45):
        kp_host = w.k_pool.clone()
        for s in range(2):
            slot = oracle.slot_of(w.block_tables[s].numpy(), j, w.block_size)
            kp_host[slot // 16, :, slot % 16, :] = (12.0 * w.q[s].float()).half()
        out, flags = run_decode(pa, w, out_dtype="f16", kp=kp_host.to(dev), vp=vp, partition_size=16)
        assert flags == 0
        for s in range(2):
            slot = oracle.slot_of(w.block_tables[s].numpy(), j, w.block_size)
            assert torch.equal(out[s].cpu(), w.v_pool[slot // 16, :, slot % 16, :]), (j, s)


def test_decode_block_permutation_invariance_bitwise(pa):
    w = W.small_decode(ctx=(300, 1029, 17), H=2, dtype="f16")
    out1, _ = run_decode(pa, w, out_dtype="f32")
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(5))
    kp2 = torch.empty_like(w.k_pool)
    vp2 = torch.empty_like(w.v_pool)
    kp2[perm] = w.k_pool
    vp2[perm] = w.v_pool
    t2 = torch.where(w.block_tables >= 0, perm[w.block_tables.clamp(min=0).long()].to(torch.int32), w.block_tables)
    out2, flags = run_decode(pa, w, out_dtype="f32", tables=t2, kp=kp2.cuda(), vp=vp2.cuda())
    assert flags == 0
    assert torch.equal(out1, out2)


def test_decode_is_deterministic(pa):
    w = W.small_decode(ctx=(700, 2100, 5, 1500), H=5, dtype="bf16")
    a, _ = run_decode(pa, w, out_dtype="f32")
    b, _ = run_decode(pa, w, out_dtype="f32")
    assert torch.equal(a, b)


def test_decode_empty_context_and_bad_entries(pa):
    w = W.small_decode(ctx=(0, 40, 33), H=2, dtype="f16")
    out, flags = run_decode(pa, w, out_dtype="f32")
    assert flags == 0
    assert torch.count_nonzero(out[0]) == 0
    assert_attn_close(out, oracle_decode(w), "f32", "empty context")
    bad = w.block_tables.clone()
    bad[2, 1] = w.num_blocks + 5
    out, flags = run_decode(pa, w, out_dtype="f32", tables=bad)
    assert flags == pa.PA_FLAG_BAD_BLOCK
    assert torch.isfinite(out).all()
    assert_attn_close(out[:2], oracle_decode(w)[:2], "f32", "rows without a bad entry")
    # sequence 2 (33 tokens, 16-token pages) without its second page: the
    # oracle over the table with that entry taken out and 17 tokens
    kept = w.block_tables.clone()
    row = w.block_tables[2].tolist()
    kept[2] = torch.tensor(row[:1] + row[2:] + row[:1], dtype=kept.dtype)
    shorter = w.context_lens.clone()
    shorter[2] = 17
    ref = oracle_decode(w, ctx=shorter, tables=kept)
    assert_attn_close(out[2:], ref[2:], "f32", "the row whose second page is out of range")
    too_long = w.context_lens.clone()
    too_long[1] = w.max_blocks_per_seq * w.block_size + 1
    out, flags = run_decode(pa, w, ctx=too_long, out_dtype="f32")
    assert flags & pa.PA_FLAG_BAD_LENGTH
    assert torch.count_nonzero(out[1]) == 0


def test_decode_many_heads_short_contexts(pa):
    """More (sequence, head) units than resident CTAs, all single-partition."""
    w = W.small_decode(ctx=tuple(range(1, 200, 7)), H=40, dtype="f16")
    out, flags = run_decode(pa, w, out_dtype="f16")
    assert flags == 0
    assert_attn_close(out, oracle_decode(w), "f16", "many heads")


def test_decode_many_small_units_stress(pa):
    """Hundreds of one- and two-tile units per CTA (partition 16 and 32):
    unit boundaries are everywhere, so consumer warps run ahead of one
    another constantly.  Repeated launches must give bitwise identical
    outputs that match the oracle."""
    g = torch.Generator().manual_seed(11)
    ctx = tuple(int(x) for x in torch.randint(1, 120, (48,), generator=g))
    w = W.small_decode(ctx=ctx, H=24, D=128, dtype="f16")
    ref = oracle_decode(w)
    dev = torch.device("cuda")
    kp, vp, q = w.k_pool.to(dev), w.v_pool.to(dev), w.q.to(dev)
    for P in (16, 32):
        first, flags = run_decode(pa, w, out_dtype="f32", partition_size=P, kp=kp, vp=vp, q=q)
        assert flags == 0
        assert_attn_close(first, ref, "f32", f"stress partition {P}")
        for _ in range(30):
            again, flags = run_decode(pa, w, out_dtype="f32", partition_size=P, kp=kp, vp=vp, q=q)
            assert flags == 0
            assert torch.equal(first, again)
