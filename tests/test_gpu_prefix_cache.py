"""Prefix caching end to end: request B's prompt repeats the first 80 tokens
of request A's.  With the allocator's prefix cache, B takes over A's five
completed blocks and only its 30 new tokens are scattered and prefilled
(ctx_before = 80).  The rows must equal, bit for bit, those of the same
request prefilled in full without the cache, and match the oracle.  The
oracle side replays both requests through the allocator model and its own
scalar scatter, starting from zeroed pools: the tables must agree with the
C++ allocator's and the GPU's pools with the oracle's, bit for bit."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import pa_workloads as W
from oracle.alloc_model import BlockAllocatorModel
from tests.gpu_common import assert_attn_close

pytestmark = pytest.mark.gpu

H, D, B, NB = 4, 128, 16, 64


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_35_gb300 as pa

    torch.cuda.set_device(0)
    return pa


def _prefill(pa, alloc, seq, prompt, k_all, v_all, q_all, kp, vp, err, reuse=True):
    """Register `prompt` for `seq`, scatter the K/V of the tokens it does not
    reuse, prefill them; returns (rows' output, reused tokens, table)."""
    dev = torch.device("cuda")
    n0 = alloc.add_seq_prefix(seq, prompt) if reuse else (alloc.add_seq(seq) or 0)
    new = list(range(n0, len(prompt)))
    slots = []
    for p in new:
        s, pairs = alloc.append_tokens([seq], [prompt[p]]) if reuse else alloc.append_slots([seq])
        assert len(pairs) == 0
        slots.append(int(s[0]))
    slots = torch.tensor(slots, dtype=torch.int64, device=dev)
    pa.pa_reshape_and_cache(k_all[new].contiguous(), v_all[new].contiguous(), kp, vp, slots, err)
    tbl, ln = alloc.block_table(seq)
    assert ln == len(prompt)
    table = torch.full((1, 16), -1, dtype=torch.int32)
    table[0, : len(tbl)] = torch.tensor(tbl, dtype=torch.int32)
    out = torch.empty(len(new), H, D, dtype=torch.float32, device=dev)
    cu = torch.tensor([0, len(new)], dtype=torch.int32, device=dev)
    cb = torch.tensor([n0], dtype=torch.int32, device=dev)
    pa.pa_prefill_chunk(out, q_all[new].contiguous(), cu, cb, kp, vp, table.to(dev), len(new), 1 / np.sqrt(D), err)
    assert pa.pa_get_error(err) == 0
    return out, n0, table


def test_second_request_reuses_the_cached_prefix(pa):
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(3)
    prompt_a = torch.randint(0, 1000, (100,), generator=g).tolist()
    prompt_b = prompt_a[:80] + torch.randint(1000, 2000, (30,), generator=g).tolist()
    # K/V/q per position: identical for the positions whose prefix is identical
    kv_a = [W.normal((100, H, D), 100 + i, torch.bfloat16) for i in range(3)]
    kv_b = [torch.cat([kv_a[i][:80], W.normal((30, H, D), 200 + i, torch.bfloat16)]) for i in range(3)]
    ka, va, qa = (t.to(dev) for t in kv_a)
    kb, vb, qb = (t.to(dev) for t in kv_b)
    err = pa.new_error_flag()

    kp = torch.zeros(NB, H, B, D, dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    alloc = pa.BlockAllocator(NB, B, prefix_cache=True)
    _prefill(pa, alloc, 0, prompt_a, ka, va, qa, kp, vp, err)
    out_b, reused, table_b = _prefill(pa, alloc, 1, prompt_b, kb, vb, qb, kp, vp, err)
    assert reused == 80
    assert table_b[0, :5].tolist() == alloc.block_table(0)[0][:5]  # A's first five blocks

    # the same request without the cache, in a pool of its own
    kp2, vp2 = torch.zeros_like(kp), torch.zeros_like(vp)
    plain = pa.BlockAllocator(NB, B)
    full, n0, table_full = _prefill(pa, plain, 1, prompt_b, kb, vb, qb, kp2, vp2, err, reuse=False)
    assert n0 == 0
    assert torch.equal(out_b, full[80:])

    # oracle: both requests replayed through the allocator model and the
    # oracle's scatter into zeroed pools of its own
    model = BlockAllocatorModel(NB, B, prefix_cache=True)
    kbits = np.zeros((NB, H, B, D), dtype=np.uint16)
    vbits = np.zeros_like(kbits)
    for seq, prompt, (k_all, v_all, _) in ((0, prompt_a, kv_a), (1, prompt_b, kv_b)):
        n0 = model.add_seq_prefix(seq, prompt)
        new = list(range(n0, len(prompt)))
        slots = []
        for p in new:
            sl, pairs = model.append_slots([seq], [prompt[p]])
            assert pairs == []
            slots.append(sl[0])
        oracle.reshape_and_cache(k_all[new], v_all[new], kbits, vbits, np.array(slots, dtype=np.int64), B)
    model_table = torch.full((1, 16), -1, dtype=torch.int32)
    model_table[0, : len(model.table(1))] = torch.tensor(model.table(1), dtype=torch.int32)
    assert torch.equal(model_table, table_b)
    assert np.array_equal(oracle.pool_bits(kp.cpu()), kbits) and np.array_equal(oracle.pool_bits(vp.cpu()), vbits)
    ref = oracle.prefill(kv_b[2][80:], torch.tensor([0, 30], dtype=torch.int32), torch.tensor([80], dtype=torch.int32),
                         kbits, vbits, model_table, B, 1 / np.sqrt(D), "bf16")
    assert_attn_close(out_b, ref, "f32", "prefix-cached prefill")
