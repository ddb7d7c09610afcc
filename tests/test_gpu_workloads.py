"""GPU parity on the full-size workloads, in the launch configuration the
benchmark times:

* LLaMA-13B-shaped decode: 64 sequences x 40 heads x 128, block 16,
  contexts uniform in [128, 2048], fp16 (every (sequence, head) checked);
* long-context decode: 256 sequences x 32 heads, bf16, log-normal contexts
  up to 16384 (every sequence checked against the oracle);
* parallel sampling with a shared 1000-token prompt: host allocator,
  copy-on-write pairs, block copy, scatter and decode, replayed on the oracle
  side with its own allocator model;
* mixed chunked prefill: 32 decode sequences plus two 512-token chunks at
  contexts 1024 and 3072, page size 256, bf16 (every decode sequence and
  every chunk row checked).

The oracle's pools always come from its own scatter (and, for parallel
sampling, its own copies) of host copies of the inputs; the GPU's pools
must equal them bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import pa_workloads as W
from oracle.alloc_model import BlockAllocatorModel
from tests.gpu_common import assert_attn_close, bits_equal, oracle_slots

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_35_gb300 as pa

    torch.cuda.set_device(0)
    return pa


def decode_step(pa, w, out_dtype=torch.float16):
    """One decode step as the benchmark runs it: write each sequence's newest
    token (position ctx-1), then attend over ctx tokens."""
    dev = torch.device("cuda")
    slots = pa.pa_slot_mapping(w.block_tables, np.arange(w.num_seqs), w.new_pos, w.block_size)
    err = pa.new_error_flag()
    pa.pa_reshape_and_cache(w.k_new, w.v_new, w.k_pool, w.v_pool, torch.from_numpy(slots).to(dev), err)
    mx = int(w.context_lens.max())
    out = torch.empty(w.num_seqs, w.num_heads, w.head_dim, dtype=out_dtype, device=dev)
    ws = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, mx)
    pa.pa_decode(out, w.q, w.k_pool, w.v_pool, w.block_tables.to(dev), w.context_lens.to(dev), mx, w.scale, ws, err)
    assert pa.pa_get_error(err) == 0
    return out


def _host_copy(w):
    """CPU copies of the workload's tensors (before the step runs)."""
    return {k: getattr(w, k).cpu() for k in ("k_pool", "v_pool", "q", "k_new", "v_new")}


def test_llama13b_decode_full(pa):
    w = W.llama13b_decode(device="cuda")
    host = _host_copy(w)
    out = decode_step(pa, w)
    kb, vb = oracle.pool_bits(host["k_pool"]), oracle.pool_bits(host["v_pool"])
    oracle.reshape_and_cache(host["k_new"], host["v_new"], kb, vb,
                             oracle_slots(w.block_tables, range(w.num_seqs), w.new_pos, w.block_size), w.block_size)
    assert bits_equal(w.k_pool, kb) and bits_equal(w.v_pool, vb)
    ref = oracle.decode(host["q"], kb, vb, w.block_tables, w.context_lens, w.block_size, w.scale, "f16")
    assert_attn_close(out, ref, "f16", "llama13b decode")


def test_long_context_decode_full(pa):
    """All 256 sequences of the long-context batch (log-normal contexts up
    to 16384, split-KV partitions merged in-kernel) against the oracle."""
    w = W.long_context_decode(device="cuda")
    host = _host_copy(w)
    out = decode_step(pa, w, out_dtype=torch.bfloat16)
    assert torch.isfinite(out.float()).all()
    kb, vb = oracle.pool_bits(host["k_pool"]), oracle.pool_bits(host["v_pool"])
    oracle.reshape_and_cache(host["k_new"], host["v_new"], kb, vb,
                             oracle_slots(w.block_tables, range(w.num_seqs), w.new_pos, w.block_size), w.block_size)
    assert bits_equal(w.k_pool, kb) and bits_equal(w.v_pool, vb)
    ref = oracle.decode(host["q"], kb, vb, w.block_tables, w.context_lens, w.block_size, w.scale, "bf16")
    assert_attn_close(out, ref, "bf16", "long-context decode")


def test_shared_prefix_parallel_sampling(pa):
    sc = W.shared_prefix()
    dev = torch.device("cuda")
    P, N, L, B = sc.num_prompts, sc.samples, sc.prompt_len, sc.block_size
    H, D = sc.num_heads, sc.head_dim
    n = P * N
    seq = [[p * N + j for j in range(N)] for p in range(P)]

    # ---- GPU side: the library's allocator + kernels
    alloc = pa.BlockAllocator(sc.num_blocks, B)
    for p in range(P):
        alloc.add_seq(seq[p][0])
    prompt_slots = np.stack([alloc.append_slots([seq[p][0] for p in range(P)])[0] for _ in range(L)], axis=1)
    for p in range(P):
        for j in range(1, N):
            alloc.fork(seq[p][0], seq[p][j])
    kp, vp = sc.pool_init_k.to(dev), sc.pool_init_v.to(dev)
    err = pa.new_error_flag()
    pa.pa_reshape_and_cache(sc.prompt_k.reshape(P * L, H, D).to(dev), sc.prompt_v.reshape(P * L, H, D).to(dev), kp, vp,
                            torch.from_numpy(prompt_slots.reshape(-1)).to(dev), err)
    suffix = sc.suffix_lens.tolist()
    suffix_slots = np.full((n, max(suffix)), -1, dtype=np.int64)
    all_pairs = []
    for r in range(max(suffix)):
        active = [s for s in range(n) if suffix[s] > r]
        slots, pairs = alloc.append_slots(active)
        suffix_slots[active, r] = slots
        if len(pairs):
            all_pairs.append(pairs)
            pa.pa_copy_blocks(kp, vp, torch.from_numpy(pairs).to(dev), err)
    pairs_gpu = np.concatenate(all_pairs)
    assert len(pairs_gpu) == 7 * P  # the 8th sample of each prompt writes in place
    ms = sc.suffix_k.shape[1]
    pa.pa_reshape_and_cache(sc.suffix_k.reshape(n * ms, H, D).to(dev), sc.suffix_v.reshape(n * ms, H, D).to(dev),
                            kp, vp, torch.from_numpy(suffix_slots.reshape(-1)).to(dev), err)
    mb = max(len(alloc.block_table(s)[0]) for s in range(n))
    tables, lens = alloc.block_tables(range(n), mb)
    out = torch.empty(n, H, D, dtype=torch.float16, device=dev)
    mx = int(lens.max())
    ws = pa.decode_workspace(n, H, D, mx)
    pa.pa_decode(out, sc.q.to(dev), kp, vp, torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev), mx,
                 sc.scale, ws, err)
    assert pa.pa_get_error(err) == 0

    # ---- oracle side: its own allocator model, scatter, copy and attention
    model = BlockAllocatorModel(sc.num_blocks, B)
    for p in range(P):
        model.add_seq(seq[p][0])
    o_prompt = np.stack([model.append_slots([seq[p][0] for p in range(P)])[0] for _ in range(L)], axis=1)
    for p in range(P):
        for j in range(1, N):
            model.fork(seq[p][0], seq[p][j])
    kb, vb = oracle.pool_bits(sc.pool_init_k), oracle.pool_bits(sc.pool_init_v)
    oracle.reshape_and_cache(sc.prompt_k.reshape(P * L, H, D), sc.prompt_v.reshape(P * L, H, D), kb, vb,
                             o_prompt.reshape(-1), B)
    o_suffix = np.full((n, max(suffix)), -1, dtype=np.int64)
    o_pairs = []
    for r in range(max(suffix)):
        active = [s for s in range(n) if suffix[s] > r]
        slots, pairs = model.append_slots(active)
        o_suffix[active, r] = slots
        if pairs:
            o_pairs += pairs
            oracle.copy_blocks(kb, vb, pairs, B)
    oracle.reshape_and_cache(sc.suffix_k.reshape(n * ms, H, D), sc.suffix_v.reshape(n * ms, H, D), kb, vb,
                             o_suffix.reshape(-1), B)
    o_tables = np.full((n, mb), -1, dtype=np.int32)
    for s in range(n):
        o_tables[s, :len(model.table(s))] = model.table(s)
    o_lens = np.array([model.length(s) for s in range(n)], dtype=np.int32)

    # indexing and copies are bit-exact
    assert np.array_equal(prompt_slots, o_prompt)
    assert np.array_equal(suffix_slots, o_suffix)
    assert [tuple(x) for x in pairs_gpu.tolist()] == o_pairs
    assert np.array_equal(tables, o_tables) and np.array_equal(lens, o_lens)
    assert bits_equal(kp, kb) and bits_equal(vp, vb)
    ref = oracle.decode(sc.q, kb, vb, o_tables, o_lens, B, sc.scale, "f16")
    assert_attn_close(out, ref, "f16", "shared-prefix decode")


def test_mixed_chunked_prefill_full(pa):
    m = W.mixed_prefill(device="cuda")
    w = m.decode
    dev = torch.device("cuda")
    host = _host_copy(w)
    chunk_k, chunk_v, chunk_q = m.chunk_k.cpu(), m.chunk_v.cpu(), m.chunk_q.cpu()
    S, C = w.num_seqs, len(m.chunk_lens)
    seq_idx = np.concatenate([np.full(int(n), c) for c, n in enumerate(m.chunk_lens.tolist())])
    pos = np.concatenate([np.arange(c0, c0 + n) for c0, n in zip(m.ctx_before.tolist(), m.chunk_lens.tolist())])
    # one scatter of 32 decode tokens + 1024 chunk tokens
    d_slots = pa.pa_slot_mapping(w.block_tables, np.arange(S), w.new_pos, w.block_size)
    c_slots = pa.pa_slot_mapping(m.chunk_tables, seq_idx, pos, w.block_size)
    err = pa.new_error_flag()
    pa.pa_reshape_and_cache(torch.cat([w.k_new, m.chunk_k]), torch.cat([w.v_new, m.chunk_v]), w.k_pool, w.v_pool,
                            torch.from_numpy(np.concatenate([d_slots, c_slots])).to(dev), err)
    mx = int(w.context_lens.max())
    dout = torch.empty(S, w.num_heads, w.head_dim, dtype=torch.bfloat16, device=dev)
    ws = pa.decode_workspace(S, w.num_heads, w.head_dim, mx)
    pa.pa_decode(dout, w.q, w.k_pool, w.v_pool, w.block_tables.to(dev), w.context_lens.to(dev), mx, w.scale, ws, err)
    T = int(m.chunk_lens.sum())
    pout = torch.empty(T, w.num_heads, w.head_dim, dtype=torch.bfloat16, device=dev)
    cu = torch.cat([torch.zeros(1, dtype=torch.int32), m.chunk_lens.cumsum(0).to(torch.int32)])
    pa.pa_prefill_chunk(pout, m.chunk_q, cu.to(dev), m.ctx_before.to(dev), w.k_pool, w.v_pool, m.chunk_tables.to(dev),
                        int(m.chunk_lens.max()), w.scale, err)
    assert pa.pa_get_error(err) == 0

    kb, vb = oracle.pool_bits(host["k_pool"]), oracle.pool_bits(host["v_pool"])
    o_slots = np.concatenate([oracle_slots(w.block_tables, range(S), w.new_pos, w.block_size),
                              oracle_slots(m.chunk_tables, seq_idx, pos, w.block_size)])
    oracle.reshape_and_cache(torch.cat([host["k_new"], chunk_k]), torch.cat([host["v_new"], chunk_v]), kb, vb, o_slots,
                             w.block_size)
    assert bits_equal(w.k_pool, kb) and bits_equal(w.v_pool, vb)
    dref = oracle.decode(host["q"], kb, vb, w.block_tables, w.context_lens, w.block_size, w.scale, "bf16")
    assert_attn_close(dout, dref, "bf16", "mixed: decode part")
    # every row of both chunks
    pref = oracle.prefill(chunk_q, cu, m.ctx_before.cpu(), kb, vb, m.chunk_tables, w.block_size, w.scale, "bf16")
    assert_attn_close(pout, pref, "bf16", "mixed: prefill part")
