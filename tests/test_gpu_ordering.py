"""Stream ordering of back-to-back calls.  The decode's planning kernel
starts early behind the slot scatter (programmatic dependent launch) and the
mixed step's decode starts early behind its prefill; both must still see
every write queued before them.  Each step here writes a new token whose key
makes it dominate its row (weight ~1), so the output row must equal that
token's value: a decode that read the pool before the scatter landed would
return the previous step's value instead.  40 steps back to back on one
stream, no host synchronisation until the end."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import pa_workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_35_gb300 as pa

    torch.cuda.set_device(0)
    return pa


def _dominant_key(q, scale):
    """A key row whose score against q is ~60 above any N(0,1) key's."""
    qf = q.float()
    return (qf / qf.norm(dim=-1, keepdim=True) * (80.0 / scale) / qf.norm(dim=-1, keepdim=True)).to(q.dtype)


def test_decode_sees_the_scatter_queued_right_before_it(pa):
    w = W.llama13b_decode(device="cuda", num_seqs=16)
    dev = torch.device("cuda")
    S, H, D, B = w.num_seqs, w.num_heads, w.head_dim, w.block_size
    slots = torch.from_numpy(pa.pa_slot_mapping(w.block_tables, np.arange(S), w.new_pos, B)).to(dev)
    tables, ctx = w.block_tables.to(dev), w.context_lens.to(dev)
    mx = int(w.context_lens.max())
    ws = pa.decode_workspace(S, H, D, mx)
    err = pa.new_error_flag()
    k_new = _dominant_key(w.q, w.scale)
    steps = 40
    g = torch.Generator(device=dev).manual_seed(5)
    vals = [torch.randn(S, H, D, generator=g, device=dev).to(w.q.dtype) for _ in range(steps)]
    outs = [torch.empty(S, H, D, dtype=torch.float32, device=dev) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        pa.pa_reshape_and_cache(k_new, vals[i], w.k_pool, w.v_pool, slots, err)
        pa.pa_decode(outs[i], w.q, w.k_pool, w.v_pool, tables, ctx, mx, w.scale, ws, err)
    assert pa.pa_get_error(err) == 0
    for i in range(steps):
        assert torch.allclose(outs[i], vals[i].float(), atol=2e-3, rtol=0), i


def test_mixed_step_sees_the_scatter_queued_right_before_it(pa):
    m = W.mixed_prefill(device="cuda", num_decode=8, chunk_len=128, ctx_before=(500,))
    w = m.decode
    dev = torch.device("cuda")
    S, H, D, B = w.num_seqs, w.num_heads, w.head_dim, w.block_size
    d_slots = pa.pa_slot_mapping(w.block_tables, np.arange(S), w.new_pos, B)
    pos = np.arange(500, 628)
    c_slots = pa.pa_slot_mapping(m.chunk_tables, np.zeros(128, dtype=np.int64), pos, B)
    slots = torch.from_numpy(np.concatenate([d_slots, c_slots])).to(dev)
    tables, ctx = w.block_tables.to(dev), w.context_lens.to(dev)
    mx = int(w.context_lens.max())
    ws = pa.decode_workspace(S, H, D, mx)
    err = pa.new_error_flag()
    cu = torch.tensor([0, 128], dtype=torch.int32, device=dev)
    cb = torch.tensor([500], dtype=torch.int32, device=dev)
    ctab = m.chunk_tables.to(dev)
    # decode rows: the new token dominates; chunk rows: every chunk key is the
    # dominant key of the chunk's first query, so that row's output is the
    # value of the chunk's first token (the only chunk key it may see)
    k_dec = _dominant_key(w.q, w.scale)
    q_chunk = m.chunk_q
    k_chunk = _dominant_key(q_chunk[:1], w.scale).expand(128, H, D).contiguous()
    steps = 20
    g = torch.Generator(device=dev).manual_seed(6)
    dvals = [torch.randn(S, H, D, generator=g, device=dev).to(w.q.dtype) for _ in range(steps)]
    cvals = [torch.randn(128, H, D, generator=g, device=dev).to(w.q.dtype) for _ in range(steps)]
    douts = [torch.empty(S, H, D, dtype=torch.float32, device=dev) for _ in range(steps)]
    pouts = [torch.empty(128, H, D, dtype=torch.float32, device=dev) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        pa.pa_reshape_and_cache(torch.cat([k_dec, k_chunk]), torch.cat([dvals[i], cvals[i]]), w.k_pool, w.v_pool,
                                slots, err)
        pa.pa_mixed_step(douts[i], w.q, tables, ctx, mx, ws, pouts[i], q_chunk, cu, cb, ctab, 128, w.k_pool,
                         w.v_pool, w.scale, err)
    assert pa.pa_get_error(err) == 0
    for i in range(steps):
        assert torch.allclose(douts[i], dvals[i].float(), atol=2e-3, rtol=0), i
        assert torch.allclose(pouts[i][0], cvals[i][0].float(), atol=2e-3, rtol=0), i
