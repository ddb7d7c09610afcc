"""A second, independent restatement of the oracle in numpy (float64).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the CUDA library or its binding.

It follows the same definitions as ``pa_oracle.c`` (section 4 equation of
"Efficient Memory Management for Large Language Model Serving with
PagedAttention"; the block-concatenated attention of the blog page's
"Attention計算の修正" section; the chunked-prefill description of the
continuous-batching page) but is written independently, with numpy array
operations instead of scalar loops, so that the two cross-check each other
on small inputs.  It also restates the split-KV combine that online softmax
makes exact, so that the identity can be checked in float64.
"""
from __future__ import annotations

import numpy as np


def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of raw fp16 / bf16 bit patterns (uint16 array)."""
    bits = np.ascontiguousarray(bits).view(np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def token_location(table_row: np.ndarray, pos: int, block_size: int):
    """0-based position -> (physical block, slot): logical block pos // B
    through the block table, slot pos % B (section 4 block mapping)."""
    return int(table_row[pos // block_size]), pos % block_size


def gather_sequence(pool: np.ndarray, table_row: np.ndarray, n: int, head: int, block_size: int):
    """Reassemble the first n tokens of one sequence for one head from a
    [NB][H][B][D] pool: returns an [n][D] array (logical order)."""
    rows = []
    for p in range(n):
        blk, slot = token_location(table_row, p, block_size)
        if blk < 0 or blk >= pool.shape[0]:
            raise IndexError(f"position {p} maps to block {blk}")
        rows.append(pool[blk, head, slot, :])
    return np.stack(rows) if rows else np.zeros((0, pool.shape[-1]))


def softmax_weights(q: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """A_j = exp(scale q.k_j) / sum_j' exp(scale q.k_j') over the rows of K."""
    x = scale * (K @ q)
    x = x - x.max()
    e = np.exp(x)
    return e / e.sum()


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    if K.shape[0] == 0:
        return np.zeros(V.shape[-1])
    return softmax_weights(q, K, scale) @ V


def decode(q, k_pool, v_pool, tables, context_lens, block_size, scale):
    """out[s, h] = attention of q[s, h] over the first context_lens[s]
    tokens of sequence s (float64 inputs, float64 output)."""
    S, H, D = q.shape
    out = np.zeros((S, H, D))
    for s in range(S):
        n = int(context_lens[s])
        for h in range(H):
            K = gather_sequence(k_pool, tables[s], n, h, block_size)
            V = gather_sequence(v_pool, tables[s], n, h, block_size)
            out[s, h] = attend(q[s, h], K, V, scale)
    return out


def prefill(q, cu_q_lens, ctx_before, k_pool, v_pool, tables, block_size, scale):
    """Chunk c's row i (position ctx_before[c]+i) attends positions
    0..ctx_before[c]+i of sequence c."""
    T, H, D = q.shape
    out = np.zeros((T, H, D))
    for c in range(len(ctx_before)):
        c0 = int(ctx_before[c])
        for i in range(int(cu_q_lens[c + 1] - cu_q_lens[c])):
            r = int(cu_q_lens[c]) + i
            n = c0 + i + 1
            for h in range(H):
                K = gather_sequence(k_pool, tables[c], n, h, block_size)
                V = gather_sequence(v_pool, tables[c], n, h, block_size)
                out[r, h] = attend(q[r, h], K, V, scale)
    return out


def reshape_and_cache(k_new, v_new, k_pool, v_pool, slot_mapping, block_size):
    """In place: token t's K/V rows go to slot slot_mapping[t] (skip if < 0)."""
    NB = k_pool.shape[0]
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        if slot >= NB * block_size:
            raise IndexError(f"slot {slot} beyond pool")
        k_pool[slot // block_size, :, slot % block_size, :] = k_new[t]
        v_pool[slot // block_size, :, slot % block_size, :] = v_new[t]


def copy_blocks(k_pool, v_pool, pairs):
    """In place, in order: block dst := block src (all heads, all slots)."""
    for src, dst in np.asarray(pairs).reshape(-1, 2).tolist():
        k_pool[dst] = k_pool[src]
        v_pool[dst] = v_pool[src]


def partition_stats(q, K, V, scale):
    """(m, l, o) of one split-KV partition: m = max score, l = sum
    exp(score - m), o = sum exp(score - m) v / l."""
    x = scale * (K @ q)
    m = x.max()
    e = np.exp(x - m)
    l = e.sum()
    return m, l, (e @ V) / l


def lse_combine(parts):
    """Combine partitions (m_p, l_p, o_p): M = max m_p,
    o = sum_p exp(m_p - M) l_p o_p / sum_p exp(m_p - M) l_p."""
    M = max(m for m, _, _ in parts)
    w = np.array([np.exp(m - M) * l for m, l, _ in parts])
    O = sum(wi * o for wi, (_, _, o) in zip(w, parts))
    return O / w.sum()
