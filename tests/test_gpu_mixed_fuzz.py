"""Seeded randomized mixed steps: decode sequences and prefill chunks of one
pool (random heads, head_dim 64 / 128, block sizes that are multiples of 16,
dtypes, output dtypes, context mixes with the page-boundary edge cases,
ragged chunks at random contexts, random prefill SM shares).  For each case
pa_mixed_step must give, bit for bit, what pa_decode and pa_prefill_chunk
give one after the other, and both parts must match the oracle, whose pools
are built by its own scatter of the step's new tokens (the continuous
batching page's "Chunked prefill": decode tokens and prefill chunks in one
step)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import pa_workloads as W
from tests.gpu_common import TORCH_OUT, assert_attn_close, bits_equal, oracle_slots

pytestmark = pytest.mark.gpu

N_CASES = 40


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_35_gb300 as pa

    torch.cuda.set_device(0)
    return pa


def _case(rng, case):
    D = int(rng.choice([64, 128]))
    B = int(rng.choice([16, 32, 48, 128, 256]))
    H = int(rng.integers(1, 5))
    dtype = str(rng.choice(["f16", "bf16"]))
    S = int(rng.integers(1, 9))
    C = int(rng.integers(1, 4))
    edge = [0, 1, B - 1, B, B + 1, 2 * B, 511, 512, 513]
    dctx = [int(rng.choice(edge)) if rng.random() < 0.4 else int(rng.integers(1, 1300)) for _ in range(S)]
    lens = [int(rng.choice([1, 127, 128, 129, int(rng.integers(1, 400))])) for _ in range(C)]
    before = [int(rng.choice([0, 1, B, int(rng.integers(0, 700))])) for _ in range(C)]
    ctx = torch.tensor(dctx + [b + n for b, n in zip(before, lens)], dtype=torch.int32)
    # the decode token written this step sits at ctx - 1 (at 0 for an empty
    # context, where it is written but not attended); a chunk's last token at
    # its end
    new_pos = ctx - 1 + (ctx == 0).to(torch.int32)
    w = W._decode_workload(f"mixed_fuzz{case}", ctx, new_pos, H, D, B, dtype, seed=300 + case)
    tables = w.block_tables
    dt = W.DTYPES[dtype]
    T = sum(lens)
    base = 1000 * (300 + case)
    return dict(
        D=D, B=B, H=H, S=S, C=C, dtype=dtype, lens=lens, before=before, w=w,
        dctx=torch.tensor(dctx, dtype=torch.int32), new_pos=new_pos[:S].contiguous(),
        dtables=tables[:S].contiguous(), ctables=tables[S:].contiguous(),
        q=w.q[:S].contiguous(), k_new=w.k_new[:S].contiguous(), v_new=w.v_new[:S].contiguous(),
        chunk_q=W.normal((T, H, D), base + 21, dt), chunk_k=W.normal((T, H, D), base + 22, dt),
        chunk_v=W.normal((T, H, D), base + 23, dt),
    )


@pytest.mark.parametrize("case", range(N_CASES))
def test_mixed_step_random_cases(pa, case):
    rng = np.random.default_rng(3000 + case)
    c = _case(rng, case)
    w, S, H, D, B = c["w"], c["S"], c["H"], c["D"], c["B"]
    lens, before = c["lens"], c["before"]
    dec_out_dtype = str(rng.choice(["f32", c["dtype"]]))
    pf_out_dtype = str(rng.choice(["f32", c["dtype"]]))
    share = int(rng.choice([0, 1, int(rng.integers(2, 120))]))
    dev = torch.device("cuda")

    seq_idx = np.concatenate([np.full(n, i) for i, n in enumerate(lens)])
    pos = np.concatenate([np.arange(b, b + n) for b, n in zip(before, lens)])
    d_slots = pa.pa_slot_mapping(c["dtables"], np.arange(S), c["new_pos"], B)
    c_slots = pa.pa_slot_mapping(c["ctables"], seq_idx, pos, B)
    slots = torch.from_numpy(np.concatenate([d_slots, c_slots])).to(dev)
    k_new = torch.cat([c["k_new"], c["chunk_k"]])
    v_new = torch.cat([c["v_new"], c["chunk_v"]])
    kp, vp = w.k_pool.to(dev), w.v_pool.to(dev)
    err = pa.new_error_flag()
    pa.pa_reshape_and_cache(k_new.to(dev), v_new.to(dev), kp, vp, slots, err)

    q, cq = c["q"].to(dev), c["chunk_q"].to(dev)
    dt, ct, ctx = c["dtables"].to(dev), c["ctables"].to(dev), c["dctx"].to(dev)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    cb = torch.tensor(before, dtype=torch.int32)
    mx = max(1, int(c["dctx"].max()))
    ws = pa.decode_workspace(S, H, D, mx)
    T = sum(lens)

    def outs():
        return (torch.full((S, H, D), float("nan"), dtype=TORCH_OUT[dec_out_dtype], device=dev),
                torch.full((T, H, D), float("nan"), dtype=TORCH_OUT[pf_out_dtype], device=dev))

    d, p = outs()
    pa.pa_mixed_step(d, q, dt, ctx, mx, ws, p, cq, cu.to(dev), cb.to(dev), ct, max(lens), kp, vp, w.scale, err,
                     prefill_sms=share)
    d_ref, p_ref = outs()
    pa.pa_decode(d_ref, q, kp, vp, dt, ctx, mx, w.scale, ws, err)
    pa.pa_prefill_chunk(p_ref, cq, cu.to(dev), cb.to(dev), kp, vp, ct, max(lens), w.scale, err)
    assert pa.pa_get_error(err) == 0
    what = (f"case {case}: S={S} C={c['C']} H={H} D={D} B={B} {c['dtype']} share={share} ctx={c['dctx'].tolist()} "
            f"lens={lens} before={before}")
    assert torch.equal(d.view(torch.uint8), d_ref.view(torch.uint8)), what
    assert torch.equal(p.view(torch.uint8), p_ref.view(torch.uint8)), what

    kb, vb = oracle.pool_bits(w.k_pool), oracle.pool_bits(w.v_pool)
    o_slots = np.concatenate([oracle_slots(c["dtables"], range(S), c["new_pos"], B),
                              oracle_slots(c["ctables"], seq_idx, pos, B)])
    oracle.reshape_and_cache(k_new, v_new, kb, vb, o_slots, B)
    assert bits_equal(kp, kb) and bits_equal(vp, vb), what
    dref = oracle.decode(c["q"], kb, vb, c["dtables"], c["dctx"], B, w.scale, c["dtype"])
    assert_attn_close(d, dref, dec_out_dtype, what + " (decode)")
    pref = oracle.prefill(c["chunk_q"], cu, cb, kb, vb, c["ctables"], B, w.scale, c["dtype"])
    assert_attn_close(p, pref, pf_out_dtype, what + " (prefill)")
