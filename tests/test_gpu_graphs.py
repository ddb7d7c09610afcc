"""Decode graphs: pa_decode recorded per padded (sequence count, KV length)
shape and replayed.  A replay must give, bit for bit, what pa_decode gives
for the padded shape; padding rows must come out as zero rows; a shape seen
before must not be recorded again; shapes past the creation maxima are
refused; one step is also checked against the oracle."""
from __future__ import annotations

import pytest
import torch

import oracle
import pa_workloads as W
from tests.gpu_common import assert_attn_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_35_gb300 as pa

    torch.cuda.set_device(0)
    return pa


@pytest.fixture(scope="module")
def work():
    return W.llama13b_decode(device="cuda")


def _pad(x, n):
    return (x + n - 1) // n * n


def _direct(pa, w, rows, s_pad, c_pad, err):
    """pa_decode on the padded shape, built by hand."""
    dev = torch.device("cuda")
    S = len(rows)
    q = torch.zeros(s_pad, w.num_heads, w.head_dim, dtype=w.q.dtype, device=dev)
    q[:S] = w.q[rows]
    tables = torch.full((s_pad, w.max_blocks_per_seq), -1, dtype=torch.int32, device=dev)
    tables[:S] = w.block_tables.to(dev)[rows]
    ctx = torch.zeros(s_pad, dtype=torch.int32, device=dev)
    ctx[:S] = w.context_lens.to(dev)[rows]
    out = torch.empty(s_pad, w.num_heads, w.head_dim, dtype=w.q.dtype, device=dev)
    ws = pa.decode_workspace(s_pad, w.num_heads, w.head_dim, c_pad)
    pa.pa_decode(out, q, w.k_pool, w.v_pool, tables, ctx, c_pad, w.scale, ws, err)
    return out


def test_replays_match_pa_decode_at_the_padded_shape(pa, work):
    w = work
    dev = torch.device("cuda")
    err = pa.new_error_flag()
    g = pa.DecodeGraphs(w.k_pool, w.v_pool, max_seqs=64, max_context_len=2048,
                        max_blocks_per_seq=w.max_blocks_per_seq, scale=w.scale, err_flag=err, seq_interval=8,
                        kv_interval=256)
    gen = torch.Generator().manual_seed(9)
    seen = set()
    for S in (5, 8, 13, 64, 5, 3, 13, 40):
        rows = torch.randperm(w.num_seqs, generator=gen)[:S].to(dev)
        ctx = w.context_lens.to(dev)[rows]
        c = int(ctx.max())
        g.q[:S] = w.q[rows]
        g.tables[:S] = w.block_tables.to(dev)[rows]
        g.context_lens[:S] = ctx
        g.run(S, c)
        s_pad, c_pad = _pad(S, 8), _pad(c, 256)
        seen.add((s_pad, c_pad))
        assert g.count == len(seen)
        ref = _direct(pa, w, rows, s_pad, c_pad, err)
        torch.cuda.synchronize()
        assert torch.equal(g.out[:S].view(torch.int16), ref[:S].view(torch.int16)), S
        assert (g.out[S:s_pad] == 0).all(), S  # padding rows (stale ones from a larger step included)
    assert pa.pa_get_error(err) == 0
    # one replayed step against the oracle
    S = 13
    rows = torch.arange(S, device=dev)
    g.q[:S] = w.q[rows]
    g.tables[:S] = w.block_tables.to(dev)[rows]
    g.context_lens[:S] = w.context_lens.to(dev)[rows]
    g.run(S, int(w.context_lens[:S].max()))
    torch.cuda.synchronize()
    kb, vb = oracle.pool_bits(w.k_pool.cpu()), oracle.pool_bits(w.v_pool.cpu())
    ref = oracle.decode(w.q[:S].cpu(), kb, vb, w.block_tables[:S], w.context_lens[:S], w.block_size, w.scale, "f16")
    assert_attn_close(g.out[:S], ref, "f16", "decode graph replay")
    g.close()


def test_shapes_past_the_maxima_are_refused(pa, work):
    w = work
    err = pa.new_error_flag()
    g = pa.DecodeGraphs(w.k_pool, w.v_pool, max_seqs=16, max_context_len=1000,
                        max_blocks_per_seq=w.max_blocks_per_seq, scale=w.scale, err_flag=err, seq_interval=8,
                        kv_interval=256)
    for S, c in ((17, 500), (8, 1025)):  # 17 pads to 24 > 16; 1025 pads to 1280 > 1024
        with pytest.raises(pa.PAError) as e:
            g.run(S, c)
        assert e.value.status == pa.PA_ERR_INVALID_ARG
    g.run(0, 0)  # an empty step is a no-op
    assert g.count == 0
    g.close()
