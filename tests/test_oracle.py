"""Pins of the CPU oracle against what the pages and mathematics fix.

Every pin here checks the oracle against something other than itself: a
value worked by hand from the pages' formulas (tests/golden), a library
routine on the textbook special case, a closed form, an invariance the
method promises, or the second (numpy) restatement.  The mutation tests at
the end plant plausible mistakes in a copy of the numpy oracle and check
that the pins catch them.
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import reference_np as rnp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _f64(t, dtype):
    return rnp.bits_to_f64(oracle._bits(t), dtype).reshape(tuple(t.shape))


def _place(contig, tables, block_size, num_blocks, fill):
    """Put contiguous per-sequence rows [S][n][H][D] into a [NB][H][B][D]
    pool: 1-based token j goes to block floor((j-1)/B), slot (j-1) mod B of
    the sequence's table (paper-summary page, section 4)."""
    S, n, H, D = contig.shape
    pool = fill.clone()
    for s in range(S):
        for j in range(1, n + 1):
            blk = int(tables[s, (j - 1) // block_size])
            pool[blk, :, (j - 1) % block_size, :] = contig[s, j - 1]
    return pool


def _random_case(S=3, n=45, H=2, D=64, B=16, NB=None, dtype="f16", seed=5):
    dt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    g = torch.Generator().manual_seed(seed)
    nblk = -(-n // B)
    NB = NB or S * nblk + 7
    perm = torch.randperm(NB, generator=g)
    tables = perm[: S * nblk].reshape(S, nblk).to(torch.int32)
    K = torch.randn(S, n, H, D, generator=g).to(dt)
    V = torch.randn(S, n, H, D, generator=g).to(dt)
    q = torch.randn(S, H, D, generator=g).to(dt)
    garbage = torch.randn(NB, H, B, D, generator=g).to(dt)
    kp = _place(K, tables, B, NB, garbage)
    vp = _place(V, tables, B, NB, garbage.flip(0))
    return q, K, V, kp, vp, tables


def _torch_attention(q, K, V, scale):
    """Textbook softmax attention on contiguous float64 data (library path)."""
    x = scale * torch.einsum("d,nd->n", q, K)
    return torch.softmax(x, dim=0) @ V


# -- data decoding --------------------------------------------------------

def test_f16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    L = oracle.lib()
    got = np.array([L.oracle_f16_to_double(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_bf16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    L = oracle.lib()
    got = np.array([L.oracle_bf16_to_double(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    np_got = rnp.bits_to_f64(bits, "bf16")
    assert np.array_equal(np_got[fin], ref[fin])


# -- values the pages fix ---------------------------------------------------

def test_block_mapping_golden():
    for B, j, blk, slot in _golden_rows("block_mapping.txt"):
        B, j, blk, slot = int(B), int(j), int(blk), int(slot)
        table = np.arange(1000, 1000 + j // B + 2)
        phys, s = rnp.token_location(table, j - 1, B)
        assert (phys, s) == (int(table[blk]), slot)
        assert oracle.slot_of(table, j - 1, B) == int(table[blk]) * B + slot


def test_closed_form_two_tokens():
    rows = {}
    for r in _golden_rows("attention_closed_form.txt"):
        rows.setdefault(r[0], []).append([float(x) for x in r[1:]])
    q = torch.tensor(rows["q"][0])
    K = torch.tensor(rows["k"])
    V = torch.tensor(rows["v"])
    expect = np.array(rows["o"][0])
    D, B = 4, 16
    # numpy restatement on contiguous data
    got_np = rnp.attend(q.numpy().astype(np.float64), K.numpy().astype(np.float64),
                        V.numpy().astype(np.float64), 1 / math.sqrt(D))
    assert np.allclose(got_np, expect, atol=1e-15, rtol=0)
    # C oracle through a paged pool: sequence in physical block 3 of 5
    kp = torch.zeros(5, 1, B, D, dtype=torch.float16)
    vp = torch.zeros(5, 1, B, D, dtype=torch.float16)
    kp[3, 0, :2] = K.half()
    vp[3, 0, :2] = V.half()
    out = oracle.decode(q.half().reshape(1, 1, D), kp, vp, torch.tensor([[3]], dtype=torch.int32),
                        torch.tensor([2], dtype=torch.int32), B, 1 / math.sqrt(D), "f16")
    assert np.allclose(out[0, 0], expect, atol=1e-15, rtol=0)
    assert abs(expect[0] - math.e / (math.e + 1)) < 1e-15


# -- special cases with closed forms ------------------------------------------

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_context_one_returns_v0(dtype):
    q, K, V, kp, vp, tables = _random_case(dtype=dtype)
    ctx = torch.ones(3, dtype=torch.int32)
    out = oracle.decode(q, kp, vp, tables, ctx, 16, 0.125, dtype)
    assert np.array_equal(out, _f64(V[:, 0], dtype))
    out_np = rnp.decode(_f64(q, dtype), _f64(kp, dtype), _f64(vp, dtype), tables.numpy(), ctx.numpy(), 16, 0.125)
    assert np.array_equal(out_np, _f64(V[:, 0], dtype))


def test_constant_keys_give_mean_of_values():
    q, K, V, kp, vp, tables = _random_case(n=45)
    same = K[:, :1].expand_as(K).contiguous()
    kp2 = _place(same, tables, 16, kp.shape[0], kp)
    ctx = torch.tensor([45, 17, 3], dtype=torch.int32)
    out = oracle.decode(q, kp2, vp, tables, ctx, 16, 0.125, "f16")
    Vf = _f64(V, "f16")
    for s, n in enumerate(ctx.tolist()):
        assert np.allclose(out[s], Vf[s, :n].mean(axis=0), atol=1e-13, rtol=0)


def test_one_hot_key_sweep_locates_every_position():
    """k_j = alpha*q for one j makes every other weight vanish below 1e-40:
    the output is V's row j.  Sweeping j over every position checks where
    the oracle finds each token."""
    q, K, V, kp, vp, tables = _random_case(S=2, n=45, H=2, D=64)
    Vf = _f64(V, "f16")
    for j in range(45):
        K2 = K.clone()
        K2[:, j] = (12.0 * q.float()).half()
        kp2 = _place(K2, tables, 16, kp.shape[0], kp)
        out = oracle.decode(q, kp2, vp, tables, torch.tensor([45, 45], dtype=torch.int32), 16, 0.125, "f16")
        assert np.allclose(out, Vf[:, j], atol=1e-30, rtol=1e-14), j


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_paged_equals_contiguous_attention(dtype):
    """Section 4 / blog 'Attention計算の修正': the paged computation gives
    the same result as attention over contiguous K, V (checked against
    torch's softmax on the contiguous data)."""
    q, K, V, kp, vp, tables = _random_case(S=3, n=61, H=2, D=64, dtype=dtype, seed=11)
    ctx = torch.tensor([61, 33, 16], dtype=torch.int32)
    out = oracle.decode(q, kp, vp, tables, ctx, 16, 0.125, dtype)
    for s, n in enumerate(ctx.tolist()):
        for h in range(2):
            ref = _torch_attention(q[s, h].double(), K[s, :n, h].double(), V[s, :n, h].double(), 0.125)
            assert np.allclose(out[s, h], ref.numpy(), atol=1e-13, rtol=0)


def test_weights_sum_to_one():
    g = torch.Generator().manual_seed(3)
    for n in (1, 2, 17, 300):
        q = torch.randn(64, generator=g, dtype=torch.float64).numpy()
        K = torch.randn(n, 64, generator=g, dtype=torch.float64).numpy()
        w = rnp.softmax_weights(q, K, 0.125)
        assert abs(w.sum() - 1.0) < 1e-13 and (w >= 0).all()


# -- invariances ------------------------------------------------------------

def test_block_permutation_invariance_is_bitwise():
    q, K, V, kp, vp, tables = _random_case(S=3, n=61, H=2, D=64, seed=4)
    ctx = torch.tensor([61, 60, 29], dtype=torch.int32)
    base = oracle.decode(q, kp, vp, tables, ctx, 16, 0.125, "f16")
    NB = kp.shape[0]
    perm = torch.randperm(NB, generator=torch.Generator().manual_seed(9))
    kp2 = torch.empty_like(kp)
    vp2 = torch.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    tables2 = perm[tables.long()].to(torch.int32)
    out = oracle.decode(q, kp2, vp2, tables2, ctx, 16, 0.125, "f16")
    assert np.array_equal(base, out)


def test_split_kv_combine_identity():
    g = torch.Generator().manual_seed(7)
    for n, cuts in ((100, [13, 64]), (2048, [512, 1024, 1536]), (17, [16])):
        q = torch.randn(128, generator=g, dtype=torch.float64).numpy()
        K = 2 * torch.randn(n, 128, generator=g, dtype=torch.float64).numpy()
        V = torch.randn(n, 128, generator=g, dtype=torch.float64).numpy()
        full = rnp.attend(q, K, V, 1 / math.sqrt(128))
        edges = [0] + cuts + [n]
        parts = [rnp.partition_stats(q, K[a:b], V[a:b], 1 / math.sqrt(128)) for a, b in zip(edges, edges[1:])]
        assert np.allclose(rnp.lse_combine(parts), full, atol=1e-12, rtol=0)


# -- the two restatements agree ---------------------------------------------

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_c_and_numpy_oracles_agree_on_decode(dtype):
    import pa_workloads as W
    w = W.tiny_decode() if dtype == "f16" else W.small_decode(ctx=(1, 16, 17, 45, 100), H=2, D=64, dtype="bf16")
    out_c = oracle.decode(w.q, w.k_pool, w.v_pool, w.block_tables, w.context_lens, w.block_size, w.scale, w.dtype)
    out_np = rnp.decode(_f64(w.q, dtype), _f64(w.k_pool, dtype), _f64(w.v_pool, dtype), w.block_tables.numpy(),
                        w.context_lens.numpy(), w.block_size, w.scale)
    assert np.allclose(out_c, out_np, atol=1e-13, rtol=0)


def test_c_and_numpy_oracles_agree_on_prefill():
    import pa_workloads as W
    m = W.small_prefill(chunk_lens=(20, 9), ctx_before=(37, 16), H=2, D=64, B=16)
    w = m.decode
    cu = torch.cat([torch.zeros(1, dtype=torch.int32), m.chunk_lens.cumsum(0).to(torch.int32)])
    out_c = oracle.prefill(m.chunk_q, cu, m.ctx_before, w.k_pool, w.v_pool, m.chunk_tables, w.block_size,
                           w.scale, w.dtype)
    out_np = rnp.prefill(_f64(m.chunk_q, "bf16"), cu.numpy(), m.ctx_before.numpy(), _f64(w.k_pool, "bf16"),
                         _f64(w.v_pool, "bf16"), m.chunk_tables.numpy(), w.block_size, w.scale)
    assert np.allclose(out_c, out_np, atol=1e-13, rtol=0)


def test_prefill_row_equals_decode_at_its_position():
    import pa_workloads as W
    m = W.small_prefill(chunk_lens=(20, 9), ctx_before=(37, 16), H=2, D=64, B=16)
    w = m.decode
    cu = torch.cat([torch.zeros(1, dtype=torch.int32), m.chunk_lens.cumsum(0).to(torch.int32)])
    out = oracle.prefill(m.chunk_q, cu, m.ctx_before, w.k_pool, w.v_pool, m.chunk_tables, w.block_size, w.scale,
                         "bf16")
    for c in range(2):
        for i in range(int(m.chunk_lens[c])):
            r = int(cu[c]) + i
            n = int(m.ctx_before[c]) + i + 1
            d = oracle.decode(m.chunk_q[r:r + 1], w.k_pool, w.v_pool, m.chunk_tables[c:c + 1],
                              torch.tensor([n], dtype=torch.int32), w.block_size, w.scale, "bf16")
            assert np.array_equal(out[r], d[0])


def test_prefill_first_row_sees_only_the_context():
    """Causality: row i of a chunk at c0 attends exactly c0+i+1 tokens, so
    changing K at positions >= c0+2 leaves rows 0 and 1 unchanged."""
    import pa_workloads as W
    m = W.small_prefill(chunk_lens=(8,), ctx_before=(21,), H=1, D=64, B=16)
    w = m.decode
    cu = torch.tensor([0, 8], dtype=torch.int32)
    a = oracle.prefill(m.chunk_q, cu, m.ctx_before, w.k_pool, w.v_pool, m.chunk_tables, 16, w.scale, "bf16")
    kp = w.k_pool.clone()
    blk = int(m.chunk_tables[0, 23 // 16])
    kp[blk, :, 23 % 16:] = 7.0   # positions 23..31 only
    b = oracle.prefill(m.chunk_q, cu, m.ctx_before, kp, w.v_pool, m.chunk_tables, 16, w.scale, "bf16")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert not np.array_equal(a[2], b[2])


def test_empty_context_gives_zero_row():
    q, K, V, kp, vp, tables = _random_case()
    ctx = torch.tensor([0, 5, 0], dtype=torch.int32)
    out = oracle.decode(q, kp, vp, tables, ctx, 16, 0.125, "f16")
    assert not out[0].any() and not out[2].any() and out[1].any()


# -- scatter and copy ---------------------------------------------------------

def test_reshape_and_cache_places_tokens_and_skips_padding():
    g = torch.Generator().manual_seed(2)
    NB, H, B, D = 6, 3, 16, 64
    kp = torch.randn(NB, H, B, D, generator=g).half()
    vp = torch.randn(NB, H, B, D, generator=g).half()
    kn = torch.randn(5, H, D, generator=g).half()
    vn = torch.randn(5, H, D, generator=g).half()
    slots = torch.tensor([0, 17, -1, 95, 40], dtype=torch.int64)
    kb, vb = oracle.pool_bits(kp), oracle.pool_bits(vp)
    oracle.reshape_and_cache(kn, vn, kb, vb, slots, B)
    expect_k, expect_v = kp.clone(), vp.clone()
    for t, s in enumerate(slots.tolist()):
        if s >= 0:
            expect_k[s // B, :, s % B] = kn[t]
            expect_v[s // B, :, s % B] = vn[t]
    assert np.array_equal(kb, oracle.pool_bits(expect_k))
    assert np.array_equal(vb, oracle.pool_bits(expect_v))
    with pytest.raises(RuntimeError):
        oracle.reshape_and_cache(kn[:1], vn[:1], kb, vb, torch.tensor([NB * B]), B)


def test_copy_blocks_is_whole_block_bitwise():
    g = torch.Generator().manual_seed(3)
    NB, H, B, D = 8, 2, 16, 64
    kp = torch.randn(NB, H, B, D, generator=g).bfloat16()
    vp = torch.randn(NB, H, B, D, generator=g).bfloat16()
    kb, vb = oracle.pool_bits(kp), oracle.pool_bits(vp)
    oracle.copy_blocks(kb, vb, [(1, 5), (2, 7)], B)
    for b in range(NB):
        src = {5: 1, 7: 2}.get(b, b)
        assert np.array_equal(kb[b], oracle.pool_bits(kp[src])), b
        assert np.array_equal(vb[b], oracle.pool_bits(vp[src])), b
    with pytest.raises(RuntimeError):
        oracle.copy_blocks(kb, vb, [(0, NB)], B)


def test_swap_blocks_moves_whole_blocks_between_pools():
    """Swap-out to a second (host) pool and swap-in to other blocks: each
    block is filled with its own id, so where every block's contents went is
    checked by value, including the pools' untouched blocks and a skipped
    pair with an id outside its pool."""
    NB_gpu, NB_cpu, H, B, D = 6, 4, 2, 16, 8
    ids = lambda n, off: np.repeat(np.arange(off, off + n, dtype=np.uint16), H * B * D).reshape(n, H, B, D)
    gk, gv = ids(NB_gpu, 0), ids(NB_gpu, 100)
    ck, cv = ids(NB_cpu, 50), ids(NB_cpu, 150)
    skipped = oracle.swap_blocks(gk, gv, ck, cv, [(4, 0), (1, 3), (2, NB_cpu)])  # out: gpu 4 -> cpu 0, 1 -> 3
    assert skipped == 1
    assert [int(ck[b, 0, 0, 0]) for b in range(NB_cpu)] == [4, 51, 52, 1]
    assert [int(cv[b, 1, 15, 7]) for b in range(NB_cpu)] == [104, 151, 152, 101]
    assert (gk == ids(NB_gpu, 0)).all() and (gv == ids(NB_gpu, 100)).all()  # the source is left as it was
    skipped = oracle.swap_blocks(ck, cv, gk, gv, [(0, 5), (3, 2), (-1, 0)])  # in: cpu 0 -> gpu 5, cpu 3 -> gpu 2
    assert skipped == 1
    assert [int(gk[b, 1, 3, 2]) for b in range(NB_gpu)] == [0, 1, 1, 3, 4, 4]
    assert [int(gv[b, 0, 0, 0]) for b in range(NB_gpu)] == [100, 101, 101, 103, 104, 104]
    for pool in (gk, gv, ck, cv):  # whole blocks: every element of a block holds one value
        assert (pool == pool[:, :1, :1, :1]).all()


# -- planted mistakes: the pins must catch them --------------------------------

def _paged_vs_contiguous_error(decode_fn):
    q, K, V, kp, vp, tables = _random_case(S=2, n=61, H=2, D=64, seed=13)
    ctx = np.array([61, 40])
    f = lambda t: _f64(t, "f16")
    out = decode_fn(f(q), f(kp), f(vp), tables.numpy(), ctx, 16, 0.125)
    err = 0.0
    for s, n in enumerate(ctx.tolist()):
        for h in range(2):
            ref = _torch_attention(q[s, h].double(), K[s, :n, h].double(), V[s, :n, h].double(), 0.125)
            err = max(err, float(np.abs(out[s, h] - ref.numpy()).max()))
    return err


def _closed_form_error(attend_fn):
    rows = {}
    for r in _golden_rows("attention_closed_form.txt"):
        rows.setdefault(r[0], []).append([float(x) for x in r[1:]])
    got = attend_fn(np.array(rows["q"][0]), np.array(rows["k"]), np.array(rows["v"]), 0.5)
    return float(np.abs(got - np.array(rows["o"][0])).max())


def test_pins_pass_on_the_oracle():
    assert _paged_vs_contiguous_error(rnp.decode) < 1e-13
    assert _closed_form_error(rnp.attend) < 1e-15


@pytest.mark.parametrize("mutant", ["block_off_by_one", "slot_block_swapped", "slot_from_next_token"])
def test_pins_catch_planted_indexing_mistakes(monkeypatch, mutant):
    bad = {
        "block_off_by_one": lambda row, p, B: (int(row[min((p + 1) // B, len(row) - 1)]), p % B),
        "slot_block_swapped": lambda row, p, B: (int(row[p % B % len(row)]), p // B),
        "slot_from_next_token": lambda row, p, B: (int(row[p // B]), (p + 1) % B),
    }[mutant]
    monkeypatch.setattr(rnp, "token_location", bad)
    assert _paged_vs_contiguous_error(rnp.decode) > 1e-3


@pytest.mark.parametrize("mutant", ["no_scale", "transposed_weights", "no_normalisation"])
def test_pins_catch_planted_arithmetic_mistakes(monkeypatch, mutant):
    def no_scale(q, K, scale):
        x = K @ q
        e = np.exp(x - x.max())
        return e / e.sum()

    def transposed(q, K, scale):
        x = scale * (K @ q)
        e = np.exp(x - x.max())
        return (e / e.sum())[::-1].copy()

    def unnormalised(q, K, scale):
        x = scale * (K @ q)
        return np.exp(x - x.max())

    bad = {"no_scale": no_scale, "transposed_weights": transposed, "no_normalisation": unnormalised}[mutant]
    monkeypatch.setattr(rnp, "softmax_weights", bad)
    assert _closed_form_error(rnp.attend) > 1e-3 or _paged_vs_contiguous_error(rnp.decode) > 1e-3
