"""pa_mixed_step: decode and chunked prefill of one mixed batch run
concurrently on one stream (the prefill's grid capped to a share of the
SMs, the decode launched behind it as a programmatic dependent).  Its
outputs must be bit-identical to pa_decode and pa_prefill_chunk called one
after the other, for any prefill SM share and with either part empty, and
match the oracle; the stream ordering it promises is exercised by queueing
the inputs' scatter and the outputs' readers on a non-default stream without
any host synchronisation in between."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
import pa_workloads as W
from tests.gpu_common import assert_attn_close, bits_equal, oracle_slots

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_35_gb300 as pa

    torch.cuda.set_device(0)
    return pa


class Step:
    """Device tensors of one mixed step (scatter inputs, decode and prefill)."""

    def __init__(self, pa, m):
        dev = torch.device("cuda")
        w = m.decode
        self.m, self.w = m, w
        S = w.num_seqs
        seq_idx = np.concatenate([np.full(int(n), c) for c, n in enumerate(m.chunk_lens.tolist())])
        pos = np.concatenate([np.arange(c0, c0 + n) for c0, n in zip(m.ctx_before.tolist(), m.chunk_lens.tolist())])
        self.seq_idx, self.pos = seq_idx, pos
        d_slots = pa.pa_slot_mapping(w.block_tables, np.arange(S), w.new_pos, w.block_size)
        c_slots = pa.pa_slot_mapping(m.chunk_tables, seq_idx, pos, w.block_size)
        self.slots = torch.from_numpy(np.concatenate([d_slots, c_slots])).to(dev)
        self.k_new = torch.cat([w.k_new, m.chunk_k]).to(dev)
        self.v_new = torch.cat([w.v_new, m.chunk_v]).to(dev)
        self.mx = int(w.context_lens.max())
        self.tables, self.ctx = w.block_tables.to(dev), w.context_lens.to(dev)
        self.T = int(m.chunk_lens.sum())
        self.cu = torch.cat([torch.zeros(1, dtype=torch.int32), m.chunk_lens.cumsum(0).to(torch.int32)]).to(dev)
        self.cb, self.ctab = m.ctx_before.to(dev), m.chunk_tables.to(dev)
        self.mq = int(m.chunk_lens.max())
        self.ws = pa.decode_workspace(S, w.num_heads, w.head_dim, self.mx)

    def outputs(self):
        w = self.w
        dev = torch.device("cuda")
        return (torch.full((w.num_seqs, w.num_heads, w.head_dim), float("nan"), dtype=torch.bfloat16, device=dev),
                torch.full((self.T, w.num_heads, w.head_dim), float("nan"), dtype=torch.bfloat16, device=dev))

    def separate(self, pa, err):
        w, m = self.w, self.m
        dout, pout = self.outputs()
        pa.pa_decode(dout, w.q, w.k_pool, w.v_pool, self.tables, self.ctx, self.mx, w.scale, self.ws, err)
        pa.pa_prefill_chunk(pout, m.chunk_q, self.cu, self.cb, w.k_pool, w.v_pool, self.ctab, self.mq, w.scale, err)
        return dout, pout

    def mixed(self, pa, err, prefill_sms=0, stream=None):
        w, m = self.w, self.m
        dout, pout = self.outputs()
        pa.pa_mixed_step(dout, w.q, self.tables, self.ctx, self.mx, self.ws, pout, m.chunk_q, self.cu, self.cb,
                         self.ctab, self.mq, w.k_pool, w.v_pool, w.scale, err, prefill_sms=prefill_sms,
                         stream=stream)
        return dout, pout


def test_mixed_step_is_bit_identical_to_separate_calls(pa):
    m = W.mixed_prefill(device="cuda")
    st = Step(pa, m)
    err = pa.new_error_flag()
    w = m.decode
    pa.pa_reshape_and_cache(st.k_new, st.v_new, w.k_pool, w.v_pool, st.slots, err)
    ref_d, ref_p = st.separate(pa, err)
    assert pa.pa_get_error(err) == 0
    for sms in (0, 1, 24, 76, 10000):  # auto share, one SM, a few, half, more than the GPU has
        d, p = st.mixed(pa, err, prefill_sms=sms)
        assert pa.pa_get_error(err) == 0
        assert torch.equal(d.view(torch.int16), ref_d.view(torch.int16)), sms
        assert torch.equal(p.view(torch.int16), ref_p.view(torch.int16)), sms


def test_mixed_step_budget512_matches_oracle(pa):
    """The 512-token step (32 decode tokens + a 480-token chunk at context
    1440), issued on non-default streams with the scatter queued right before
    it and the outputs copied right after it on the caller's stream."""
    m = W.budget512_step(device="cuda")
    w = m.decode
    host = {k: getattr(w, k).cpu() for k in ("k_pool", "v_pool", "q", "k_new", "v_new")}
    chunk_k, chunk_v, chunk_q = m.chunk_k.cpu(), m.chunk_v.cpu(), m.chunk_q.cpu()
    st = Step(pa, m)
    err = pa.new_error_flag()
    main = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(main):
        pa.pa_reshape_and_cache(st.k_new, st.v_new, w.k_pool, w.v_pool, st.slots, err, stream=main)
        d, p = st.mixed(pa, err, stream=main)
        d_host = d.to("cpu", non_blocking=False)
        p_host = p.to("cpu", non_blocking=False)
    assert pa.pa_get_error(err, main) == 0

    S = w.num_seqs
    kb, vb = oracle.pool_bits(host["k_pool"]), oracle.pool_bits(host["v_pool"])
    o_slots = np.concatenate([oracle_slots(w.block_tables, range(S), w.new_pos, w.block_size),
                              oracle_slots(m.chunk_tables, st.seq_idx, st.pos, w.block_size)])
    oracle.reshape_and_cache(torch.cat([host["k_new"], chunk_k]), torch.cat([host["v_new"], chunk_v]), kb, vb,
                             o_slots, w.block_size)
    assert bits_equal(w.k_pool, kb) and bits_equal(w.v_pool, vb)
    dref = oracle.decode(host["q"], kb, vb, w.block_tables, w.context_lens, w.block_size, w.scale, "bf16")
    assert_attn_close(d_host, dref, "bf16", "budget-512 step: decode part")
    # every row of the 480-query chunk
    cu = torch.cat([torch.zeros(1, dtype=torch.int32), m.chunk_lens.cpu().cumsum(0).to(torch.int32)])
    pref = oracle.prefill(chunk_q, cu, m.ctx_before.cpu(), kb, vb, m.chunk_tables, w.block_size, w.scale, "bf16")
    assert_attn_close(p_host, pref, "bf16", "budget-512 step: prefill part")


def test_mixed_step_refuses_bad_arguments_before_launching(pa):
    """A bad argument of either part: nothing may run, not even the other part."""
    m = W.mixed_prefill(device="cuda", num_decode=4, chunk_len=64, ctx_before=(100,))
    st = Step(pa, m)
    err = pa.new_error_flag()
    w = m.decode
    d, p = st.outputs()
    small = torch.empty(16, dtype=torch.uint8, device="cuda")  # decode workspace too small
    with pytest.raises(pa.PAError) as e:
        pa.pa_mixed_step(d, w.q, st.tables, st.ctx, st.mx, small, p, m.chunk_q, st.cu, st.cb, st.ctab, st.mq,
                         w.k_pool, w.v_pool, w.scale, err)
    assert e.value.status == pa.PA_ERR_WORKSPACE
    with pytest.raises(pa.PAError) as e:  # a negative chunk-length bound
        pa.pa_mixed_step(d, w.q, st.tables, st.ctx, st.mx, st.ws, p, m.chunk_q, st.cu, st.cb, st.ctab, -1,
                         w.k_pool, w.v_pool, w.scale, err)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.isnan(p.float()).all() and torch.isnan(d.float()).all()
    assert pa.pa_get_error(err) == 0


def test_mixed_step_with_one_part_empty(pa):
    """No chunks: it is pa_decode; no sequences: it is pa_prefill_chunk."""
    m = W.mixed_prefill(device="cuda", num_decode=6, chunk_len=200, ctx_before=(300,))
    st = Step(pa, m)
    w = m.decode
    dev = torch.device("cuda")
    err = pa.new_error_flag()
    pa.pa_reshape_and_cache(st.k_new, st.v_new, w.k_pool, w.v_pool, st.slots, err)
    ref_d, ref_p = st.separate(pa, err)
    H, D = w.num_heads, w.head_dim
    d, _ = st.outputs()
    no_q = torch.empty(0, H, D, dtype=w.q.dtype, device=dev)
    no_out = torch.empty(0, H, D, dtype=torch.bfloat16, device=dev)
    zero_cu = torch.zeros(1, dtype=torch.int32, device=dev)
    no_cb = torch.empty(0, dtype=torch.int32, device=dev)
    pa.pa_mixed_step(d, w.q, st.tables, st.ctx, st.mx, st.ws, no_out, no_q, zero_cu, no_cb, st.ctab, 0,
                     w.k_pool, w.v_pool, w.scale, err)
    _, p = st.outputs()
    no_tables = torch.empty(0, w.max_blocks_per_seq, dtype=torch.int32, device=dev)
    no_ctx = torch.empty(0, dtype=torch.int32, device=dev)
    pa.pa_mixed_step(no_out, no_q, no_tables, no_ctx, 0, st.ws, p, m.chunk_q, st.cu, st.cb, st.ctab, st.mq,
                     w.k_pool, w.v_pool, w.scale, err)
    assert pa.pa_get_error(err) == 0
    assert torch.equal(d.view(torch.int16), ref_d.view(torch.int16))
    assert torch.equal(p.view(torch.int16), ref_p.view(torch.int16))


def test_mixed_step_head_dim_64(pa):
    m = W.mixed_prefill(device="cuda", num_decode=8, chunk_len=200, ctx_before=(300, 1000), D=64)
    st = Step(pa, m)
    w = m.decode
    err = pa.new_error_flag()
    pa.pa_reshape_and_cache(st.k_new, st.v_new, w.k_pool, w.v_pool, st.slots, err)
    ref_d, ref_p = st.separate(pa, err)
    d, p = st.mixed(pa, err)
    assert pa.pa_get_error(err) == 0
    assert torch.equal(d.view(torch.int16), ref_d.view(torch.int16))
    assert torch.equal(p.view(torch.int16), ref_p.view(torch.int16))
