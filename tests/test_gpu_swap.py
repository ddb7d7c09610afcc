"""pa_swap_blocks: whole-block moves between the GPU pool and a pinned host
pool (swap-out of a preempted request, swap-in on resume), checked bit for
bit against the oracle's block swap; plus a preempt / resume round trip
through the decode kernel."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import pa_workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_35_gb300 as pa

    torch.cuda.set_device(0)
    return pa


def _pools(NB, H, B, D, dtype, seed, device):
    k = W.normal((NB, H, B, D), seed, dtype, device)
    v = W.normal((NB, H, B, D), seed + 1, dtype, device)
    if device == "cpu":
        k, v = k.pin_memory(), v.pin_memory()
    return k, v


def _pairs(n, src_nb, dst_nb, seed):
    g = torch.Generator().manual_seed(seed)
    src = torch.randperm(src_nb, generator=g)[:n]
    dst = torch.randperm(dst_nb, generator=g)[:n]
    return torch.stack([src, dst], 1).to(torch.int32)


@pytest.mark.parametrize("B,dtype", [(16, torch.float16), (256, torch.bfloat16), (32, torch.float16)])
def test_swap_out_then_in_is_bit_exact(pa, B, dtype):
    H, D = 8, 128
    NB_gpu, NB_cpu = 48, 40
    gk, gv = _pools(NB_gpu, H, B, D, dtype, 11, "cuda")
    ck, cv = _pools(NB_cpu, H, B, D, dtype, 21, "cpu")
    o_gk, o_gv, o_ck, o_cv = (oracle.pool_bits(t.cpu()) for t in (gk, gv, ck, cv))
    err = pa.new_error_flag()
    out_pairs = _pairs(30, NB_gpu, NB_cpu, 1)
    pa.pa_swap_blocks(gk, gv, ck, cv, out_pairs.cuda(), err)  # swap-out: GPU -> pinned host
    assert pa.pa_get_error(err) == 0
    assert oracle.swap_blocks(o_gk, o_gv, o_ck, o_cv, out_pairs.numpy()) == 0
    assert np.array_equal(oracle.pool_bits(ck), o_ck) and np.array_equal(oracle.pool_bits(cv), o_cv)
    in_pairs = _pairs(25, NB_cpu, NB_gpu, 2)
    pa.pa_swap_blocks(ck, cv, gk, gv, in_pairs.cuda(), err)  # swap-in: pinned host -> GPU
    assert pa.pa_get_error(err) == 0
    assert oracle.swap_blocks(o_ck, o_cv, o_gk, o_gv, in_pairs.numpy()) == 0
    assert np.array_equal(oracle.pool_bits(gk.cpu()), o_gk) and np.array_equal(oracle.pool_bits(gv.cpu()), o_gv)


def test_swap_between_two_device_pools_and_two_host_pools(pa):
    H, B, D = 4, 16, 64
    err = pa.new_error_flag()
    for dev in ("cuda", "cpu"):
        ak, av = _pools(10, H, B, D, torch.float16, 31, dev)
        bk, bv = _pools(7, H, B, D, torch.float16, 41, dev)
        o = [oracle.pool_bits(t.cpu()) for t in (ak, av, bk, bv)]
        pairs = torch.tensor([[9, 0], [0, 6], [4, 3]], dtype=torch.int32)
        pa.pa_swap_blocks(ak, av, bk, bv, pairs.cuda(), err)
        assert pa.pa_get_error(err) == 0
        oracle.swap_blocks(*o, pairs.numpy())
        assert np.array_equal(oracle.pool_bits(bk.cpu()), o[2]) and np.array_equal(oracle.pool_bits(bv.cpu()), o[3])


def test_swap_flags_and_skips_bad_ids_and_checks_sizes(pa):
    H, B, D = 2, 16, 64
    gk, gv = _pools(6, H, B, D, torch.bfloat16, 51, "cuda")
    ck, cv = _pools(4, H, B, D, torch.bfloat16, 61, "cpu")
    o = [oracle.pool_bits(t.cpu()) for t in (gk, gv, ck, cv)]
    pairs = torch.tensor([[1, 0], [6, 1], [2, -1], [3, 4], [5, 3]], dtype=torch.int32)
    err = pa.new_error_flag()
    pa.pa_swap_blocks(gk, gv, ck, cv, pairs.cuda(), err)
    assert pa.pa_get_error(err) == pa.PA_FLAG_BAD_BLOCK
    assert oracle.swap_blocks(*o, pairs.numpy()) == 3
    assert np.array_equal(oracle.pool_bits(ck), o[2]) and np.array_equal(oracle.pool_bits(cv), o[3])
    # no pairs: nothing happens; more pairs than one launch takes: refused on the host
    pa.pa_swap_blocks(gk, gv, ck, cv, torch.empty(0, 2, dtype=torch.int32, device="cuda"), err)
    too_many = torch.zeros(65536, 2, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_swap_blocks(gk, gv, ck, cv, too_many, err)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    with pytest.raises(ValueError):  # a host pool that is not pinned
        pa.pa_swap_blocks(gk, gv, ck.clone(), cv.clone(), pairs.cuda(), err)
    assert pa.pa_get_error(err) == 0


def test_preempt_and_resume_gives_the_same_decode(pa):
    """A batch is decoded; half of its sequences are swapped out (their blocks
    freed and overwritten by other data), then swapped back in to other
    physical blocks with their tables remapped: the decode output is
    unchanged, bit for bit."""
    w = W.small_decode(ctx=(17, 300, 700, 1029, 64, 255), H=4, D=128, dtype="bf16", device="cuda")
    dev = torch.device("cuda")
    S, H, D, B = w.num_seqs, w.num_heads, w.head_dim, w.block_size
    tables, ctx = w.block_tables.clone(), w.context_lens
    mx = int(ctx.max())
    err = pa.new_error_flag()
    ws = pa.decode_workspace(S, H, D, mx)

    def decode(tab):
        out = torch.empty(S, H, D, dtype=torch.float32, device=dev)
        pa.pa_decode(out, w.q, w.k_pool, w.v_pool, tab.to(dev), ctx.to(dev), mx, w.scale, ws, err)
        assert pa.pa_get_error(err) == 0
        return out

    before = decode(tables)
    victims = [1, 3, 5]
    used = [int(b) for s in victims for b in tables[s, : -(-int(ctx[s]) // B)]]
    host_k = torch.empty(len(used), H, B, D, dtype=w.k_pool.dtype).pin_memory()
    host_v = torch.empty_like(host_k).pin_memory()
    out_pairs = torch.tensor([[b, i] for i, b in enumerate(used)], dtype=torch.int32, device=dev)
    pa.pa_swap_blocks(w.k_pool, w.v_pool, host_k, host_v, out_pairs, err)
    # the freed blocks get other requests' data
    junk = torch.tensor(used, device=dev)
    w.k_pool[junk] = torch.randn(len(used), H, B, D, device=dev).to(w.k_pool.dtype)
    w.v_pool[junk] = torch.randn(len(used), H, B, D, device=dev).to(w.v_pool.dtype)
    # resume into blocks that nobody uses: the pool's spare blocks, then the freed ones reversed
    taken = set(int(b) for b in tables[tables >= 0])
    spare = [b for b in range(w.num_blocks) if b not in taken] + used[::-1]
    new_ids = spare[: len(used)]
    in_pairs = torch.tensor([[i, b] for i, b in enumerate(new_ids)], dtype=torch.int32, device=dev)
    pa.pa_swap_blocks(host_k, host_v, w.k_pool, w.v_pool, in_pairs, err)
    remap = dict(zip(used, new_ids))
    new_tables = tables.clone()
    for s in victims:
        n = -(-int(ctx[s]) // B)
        new_tables[s, :n] = torch.tensor([remap[int(b)] for b in tables[s, :n]], dtype=torch.int32)
    after = decode(new_tables)
    assert torch.equal(before, after)
