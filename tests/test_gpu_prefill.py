"""GPU parity of the tcgen05 chunked-prefill kernel against the CPU oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import pa_workloads as W
from tests.gpu_common import TORCH_OUT, assert_attn_close, oracle_slots

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_35_gb300 as pa

    torch.cuda.set_device(0)
    return pa


def chunk_positions(m):
    seq_idx = np.concatenate([np.full(n, c) for c, n in enumerate(m.chunk_lens.tolist())])
    pos = np.concatenate([np.arange(c0, c0 + n) for c0, n in zip(m.ctx_before.tolist(), m.chunk_lens.tolist())])
    return seq_idx, pos


def cu_lens(m):
    return torch.cat([torch.zeros(1, dtype=torch.int32), m.chunk_lens.cumsum(0).to(torch.int32)])


def run_prefill(pa, m, out_dtype="f32", tables=None, ctx_before=None):
    """Write the chunks' K/V with pa_reshape_and_cache, then pa_prefill_chunk."""
    w = m.decode
    dev = torch.device("cuda")
    kp, vp = w.k_pool.to(dev), w.v_pool.to(dev)
    tables = m.chunk_tables if tables is None else tables
    ctx_before = m.ctx_before if ctx_before is None else ctx_before
    seq_idx, pos = chunk_positions(m)
    slots = pa.pa_slot_mapping(m.chunk_tables, seq_idx, pos, w.block_size)
    err = pa.new_error_flag()
    pa.pa_reshape_and_cache(m.chunk_k.to(dev), m.chunk_v.to(dev), kp, vp, torch.from_numpy(slots).to(dev), err)
    assert pa.pa_get_error(err) == 0
    T = int(m.chunk_lens.sum())
    out = torch.full((T, w.num_heads, w.head_dim), float("nan"), dtype=TORCH_OUT[out_dtype], device=dev)
    pa.pa_prefill_chunk(out, m.chunk_q.to(dev), cu_lens(m).to(dev), ctx_before.to(dev), kp, vp, tables.to(dev),
                        int(m.chunk_lens.max()), w.scale, err)
    flags = pa.pa_get_error(err)
    return out, flags, kp, vp


def oracle_prefill(m):
    w = m.decode
    kb, vb = oracle.pool_bits(w.k_pool), oracle.pool_bits(w.v_pool)
    seq_idx, pos = chunk_positions(m)
    oracle.reshape_and_cache(m.chunk_k, m.chunk_v, kb, vb, oracle_slots(m.chunk_tables, seq_idx, pos, w.block_size),
                             w.block_size)
    ref = oracle.prefill(m.chunk_q, cu_lens(m), m.ctx_before, kb, vb, m.chunk_tables, w.block_size, w.scale, w.dtype)
    return ref, kb, vb


@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_prefill_small_ragged_bf16(pa, out_dtype):
    m = W.small_prefill()
    out, flags, _, _ = run_prefill(pa, m, out_dtype)
    assert flags == 0
    ref, _, _ = oracle_prefill(m)
    assert_attn_close(out, ref, out_dtype, "prefill bf16")


@pytest.mark.parametrize("B", [16, 32, 48, 80, 128, 144, 256, 384])
def test_prefill_block_sizes(pa, B):
    m = W.small_prefill(chunk_lens=(200, 64), ctx_before=(300, 0), H=2, B=B)
    out, flags, _, _ = run_prefill(pa, m, "f32")
    assert flags == 0
    ref, _, _ = oracle_prefill(m)
    assert_attn_close(out, ref, "f32", f"prefill block {B}")


def test_prefill_fp16_tile_aligned_chunks(pa):
    m = W.small_prefill(chunk_lens=(128, 256, 1), ctx_before=(128, 0, 511), H=2, B=16, dtype="f16")
    out, flags, _, _ = run_prefill(pa, m, "f16")
    assert flags == 0
    ref, _, _ = oracle_prefill(m)
    assert_attn_close(out, ref, "f16", "prefill fp16")


def test_prefill_bf16_values_outside_the_fp16_range(pa):
    """A bf16 pool's V tiles go through the P V product in fp16, which holds
    bf16 values exactly only below 2^16.  Place V values of 65280 (the largest
    bf16 value below 2^16), 2^16 and beyond, in the cached context and among
    the chunk's own tokens, in one or both halves of a key tile: rows that
    see them must stay within the gate relative to the largest |v| they see,
    every other row within the plain gate."""
    m = W.small_prefill(chunk_lens=(200, 150), ctx_before=(300, 40), H=2, B=16)
    w = m.decode
    B = w.block_size
    big = []  # (chunk, head, position, value)
    for c, h, p, val in ((0, 0, 5, 3.0e5), (0, 0, 140, 65280.0), (0, 1, 200, -65536.0), (0, 1, 330, 1.0e6),
                         (1, 0, 10, 65280.0), (1, 1, 100, -2.5e5), (1, 1, 170, 7.0e4)):
        c0 = int(m.ctx_before[c])
        if p < c0:  # cached context: straight into the pool
            blk = int(m.chunk_tables[c, p // B])
            w.v_pool[blk, h, p % B, 3] = val
        else:       # one of the chunk's tokens, written by the scatter
            t = int(m.chunk_lens[:c].sum()) + p - c0
            m.chunk_v[t, h, 3] = val
        big.append((c, h, p, abs(float(torch.tensor(val, dtype=torch.bfloat16).float()))))
    out, flags, _, _ = run_prefill(pa, m, "f32")
    assert flags == 0
    ref, _, _ = oracle_prefill(m)
    g = out.cpu().double().numpy()
    assert np.isfinite(g).all()
    # largest |v| each output row (token, head) attends to
    scale = np.ones(g.shape[:2])
    starts = [0] + np.cumsum(m.chunk_lens.numpy()).tolist()
    for c, h, p, a in big:
        c0 = int(m.ctx_before[c])
        first = max(p - c0, 0)  # chunk rows at positions >= p see key p
        rows = slice(starts[c] + first, starts[c + 1])
        scale[rows, h] = np.maximum(scale[rows, h], a)
    err = np.abs(g - ref).max(axis=2)
    worst = float((err / scale).max())
    assert worst <= 2e-3, f"relative error {worst:.3e}"
    assert float(err[scale == 1.0].max()) <= 2e-3


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("hot", [0, 150, 207, 263, 499])
def test_prefill_one_hot_key_is_bitwise(pa, hot, dtype):
    """Every query of the chunk equals q0 and the key at position `hot` is
    32 q0 (per head), so for each row that sees it every other weight
    underflows to 0: the output row is V[hot] bit for bit.  Sweeping `hot`
    over the cached context and the chunk's own tokens (several key tiles and
    16-token pages) checks the paged indexing of the prefill kernel exactly.
    Rows before `hot` are checked against the oracle within the gate."""
    m = W.small_prefill(chunk_lens=(300,), ctx_before=(200,), H=2, B=16, dtype=dtype)
    w = m.decode
    B, c0 = w.block_size, int(m.ctx_before[0])
    g = torch.Generator().manual_seed(11)
    q0 = torch.randn(w.num_heads, w.head_dim, generator=g).to(m.chunk_q.dtype)
    m.chunk_q[:] = q0
    key = (32.0 * q0.float()).to(m.chunk_q.dtype)
    if hot < c0:
        blk = int(m.chunk_tables[0, hot // B])
        w.k_pool[blk, :, hot % B, :] = key
        v_hot = w.v_pool[blk, :, hot % B, :].float()
    else:
        m.chunk_k[hot - c0] = key
        v_hot = m.chunk_v[hot - c0].float()
    out, flags, _, _ = run_prefill(pa, m, "f32")
    assert flags == 0
    got = out.cpu()
    first = max(hot - c0, 0)  # chunk rows at positions >= hot see the key
    assert torch.equal(got[first:], v_hot.expand(300 - first, -1, -1)), "one-hot rows differ from V[hot]"
    if first > 0:
        ref, _, _ = oracle_prefill(m)
        assert_attn_close(got[:first], ref[:first], "f32", f"rows before key {hot}")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_prefill_single_key_row_is_v0_bitwise(pa, dtype):
    """A chunk at context 0: its first row attends to one key, its own
    token, so its output is that token's V row exactly (exp(0) = 1)."""
    m = W.small_prefill(chunk_lens=(5, 130), ctx_before=(0, 0), H=3, B=16, dtype=dtype)
    out, flags, _, _ = run_prefill(pa, m, "f32")
    assert flags == 0
    got = out.cpu()
    assert torch.equal(got[0], m.chunk_v[0].float())
    assert torch.equal(got[5], m.chunk_v[5].float())


def test_prefill_rows_match_decode_at_their_positions(pa):
    """Cross-kernel: chunk row i equals pa_decode of the same query with a
    context of ctx_before + i + 1 tokens."""
    m = W.small_prefill(chunk_lens=(150,), ctx_before=(333,), H=2, B=16)
    out, flags, kp, vp = run_prefill(pa, m, "f32")
    assert flags == 0
    w = m.decode
    rows = torch.arange(0, 150, 7)
    ctx = (m.ctx_before[0] + rows + 1).to(torch.int32)
    tables = m.chunk_tables.expand(len(rows), -1).contiguous()
    q = m.chunk_q[rows].contiguous()
    dev = torch.device("cuda")
    dout = torch.empty(len(rows), w.num_heads, w.head_dim, dtype=torch.float32, device=dev)
    ws = pa.decode_workspace(len(rows), w.num_heads, w.head_dim, int(ctx.max()))
    err = pa.new_error_flag()
    pa.pa_decode(dout, q.to(dev), kp, vp, tables.to(dev), ctx.to(dev), int(ctx.max()), w.scale, ws, err)
    assert pa.pa_get_error(err) == 0
    assert float((dout.cpu() - out[rows].cpu()).abs().max()) <= 2e-3


def test_prefill_flags_bad_table_entry(pa):
    m = W.small_prefill(chunk_lens=(40,), ctx_before=(100,), H=1, B=16)
    bad = m.chunk_tables.clone()
    bad[0, 2] = -3
    out, flags, _, _ = run_prefill(pa, m, "f32", tables=bad)
    assert flags == pa.PA_FLAG_BAD_BLOCK
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("B,bad_page,dtype,D", [(16, 3, "bf16", 128), (48, 1, "bf16", 128), (16, 2, "f16", 64),
                                               (32, 5, "f16", 128)])
def test_prefill_skips_the_keys_of_a_bad_page(pa, B, bad_page, dtype, D):
    """Keys in a page whose table entry is out of range are skipped, and the
    call flags it.  The reference is the oracle over the sequence with that
    page's entry taken out of the table: there row p sits at p (before the
    page), at the page's first position minus one (inside it) or at p - B
    (after it); each row runs as a one-row chunk at that position."""
    m = W.small_prefill(chunk_lens=(300,), ctx_before=(0,), H=2, B=B, D=D, dtype=dtype)
    w = m.decode
    bad = m.chunk_tables.clone()
    bad[0, bad_page] = -3
    out, flags, _, _ = run_prefill(pa, m, "f32", tables=bad)
    assert flags == pa.PA_FLAG_BAD_BLOCK

    kb, vb = oracle.pool_bits(w.k_pool), oracle.pool_bits(w.v_pool)
    seq_idx, pos = chunk_positions(m)
    oracle.reshape_and_cache(m.chunk_k, m.chunk_v, kb, vb, oracle_slots(m.chunk_tables, seq_idx, pos, B), B)
    row = m.chunk_tables[0].tolist()
    kept = row[:bad_page] + row[bad_page + 1:] + [row[0]]
    T = int(m.chunk_lens[0])
    lo, hi = bad_page * B, (bad_page + 1) * B
    at = [p if p < lo else (lo - 1 if p < hi else p - B) for p in range(T)]
    ref = oracle.prefill(m.chunk_q, torch.arange(T + 1, dtype=torch.int32), torch.tensor(at, dtype=torch.int32), kb,
                         vb, torch.tensor([kept] * T, dtype=torch.int32), B, w.scale, w.dtype)
    assert_attn_close(out, ref, "f32", f"prefill, page {bad_page} of {B} tokens out of range")


def test_prefill_skips_a_chunk_whose_context_overruns_its_table(pa):
    """A chunk whose last position lies past its table's capacity is flagged
    and skipped (its output rows are not written); the chunks beside it are
    computed as usual."""
    m = W.small_prefill(chunk_lens=(100, 50, 80), ctx_before=(10, 20, 30), H=2, B=16)
    cb = m.ctx_before.clone()
    cb[1] = m.chunk_tables.shape[1] * 16
    out, flags, _, _ = run_prefill(pa, m, "f32", ctx_before=cb)
    assert flags == pa.PA_FLAG_BAD_LENGTH
    assert torch.isnan(out[100:150]).all()
    keep = torch.cat([torch.arange(0, 100), torch.arange(150, 230)])
    ref, _, _ = oracle_prefill(m)
    assert_attn_close(out[keep.cuda()], ref[keep.numpy()], "f32", "chunks beside the skipped one")


def test_prefill_with_every_chunk_skipped_ends_cleanly(pa):
    """No runnable item at all: every CTA sees only the end of the list."""
    m = W.small_prefill(chunk_lens=(40, 9), ctx_before=(0, 0), H=2, B=16)
    cb = torch.full_like(m.ctx_before, m.chunk_tables.shape[1] * 16)
    out, flags, _, _ = run_prefill(pa, m, "bf16", ctx_before=cb)
    assert flags == pa.PA_FLAG_BAD_LENGTH
    assert torch.isnan(out.float()).all()


def test_prefill_many_items_per_cta(pa):
    """Ten or so (query tile, head) items per CTA of the persistent grid, with
    an empty chunk and chunks of one row among them: every item's output must
    come out right whatever ran on the same CTA before it."""
    m = W.small_prefill(chunk_lens=(700, 0, 300, 513, 129, 1, 255), ctx_before=(40, 77, 0, 1500, 129, 2047, 333),
                        H=16, B=16)
    out, flags, _, _ = run_prefill(pa, m, "f32")
    assert flags == 0
    ref, _, _ = oracle_prefill(m)
    assert_attn_close(out, ref, "f32", "prefill many items")


@pytest.mark.parametrize("n_chunks", [1000, 1100])
def test_prefill_many_short_chunks(pa, n_chunks):
    """More (chunk, query tile) pairs than the in-kernel ranking handles
    (1100) and just under it (1000): both work orders give the same result."""
    g = torch.Generator().manual_seed(5)
    cl = tuple(int(x) for x in torch.randint(1, 4, (n_chunks,), generator=g))
    cb = tuple(int(x) for x in torch.randint(0, 200, (n_chunks,), generator=g))
    m = W.small_prefill(chunk_lens=cl, ctx_before=cb, H=2, B=16)
    out, flags, _, _ = run_prefill(pa, m, "bf16")
    assert flags == 0
    ref, _, _ = oracle_prefill(m)
    assert_attn_close(out, ref, "bf16", f"prefill {n_chunks} short chunks")


@pytest.mark.parametrize("dtype,out_dtype,B", [("bf16", "f32", 16), ("f16", "f16", 256), ("bf16", "bf16", 48)])
def test_prefill_head_dim_64(pa, dtype, out_dtype, B):
    """head_dim 64: one swizzled 64-column half per tile, K = 64 for S and
    N = 64 for P V; ragged chunks over several key tiles, one chunk at
    context 0 (rows with one or two keys)."""
    m = W.small_prefill(chunk_lens=(300, 77, 1), ctx_before=(150, 0, 700), H=3, D=64, B=B, dtype=dtype)
    out, flags, _, _ = run_prefill(pa, m, out_dtype)
    assert flags == 0
    ref, _, _ = oracle_prefill(m)
    assert_attn_close(out, ref, out_dtype, f"prefill head_dim 64 {dtype} block {B}")


@pytest.mark.parametrize("B", [16, 1024])
def test_prefill_long_chunk(pa, B):
    """One 2048-query chunk at context 0 (16 query tiles, causal over up to
    16 key tiles), 4 heads.  The oracle scatters the chunk's K/V into its own
    copy of the pools; the GPU's scattered pools must equal them bit for bit,
    and every row of the output must match the oracle's attention over them."""
    m = W.small_prefill(chunk_lens=(2048,), ctx_before=(0,), H=4, B=B)
    out, flags, kp, vp = run_prefill(pa, m, "f32")
    assert flags == 0
    ref, kb, vb = oracle_prefill(m)
    assert np.array_equal(oracle.pool_bits(kp.cpu()), kb) and np.array_equal(oracle.pool_bits(vp.cpu()), vb)
    assert_attn_close(out, ref, "f32", f"prefill 2048-query chunk, block {B}")


def test_prefill_head_groups(pa):
    """A launch of at least eight rounds of the grid deals its heads in groups
    (here 4 chunks x 4 query tiles x 80 heads = 1280 items: two groups of 40
    heads, the second taking its query tiles shortest first).  The order is
    only a schedule: every row must match the oracle."""
    m = W.small_prefill(chunk_lens=(512, 512, 512, 512), ctx_before=(0, 50, 130, 300), H=80, B=16)
    out, flags, _, _ = run_prefill(pa, m, "f32")
    assert flags == 0
    ref, _, _ = oracle_prefill(m)
    assert_attn_close(out, ref, "f32", "prefill with head groups")
