"""Shared helpers of the GPU parity tests: tolerance and oracle plumbing."""
from __future__ import annotations

import numpy as np
import torch

import oracle

ATTN_ATOL = 2e-3  # max-abs error of attention against the fp64 oracle


def half_ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Half a unit in the last place of |x| in fp16 / bf16 (normal range)."""
    mant = {"f16": 10, "bf16": 7}[dtype]
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -14)))
    return 0.5 * 2.0 ** (e - mant)


def attn_error_excess(got: np.ndarray, ref: np.ndarray, out_dtype: str) -> float:
    """Largest amount by which |got - ref| exceeds the gate: 2e-3 for fp32
    output, 2e-3 + half an output ulp for fp16/bf16 output (the rounding of
    an exact result alone can exceed 2e-3 in bf16).  <= 0 means within."""
    diff = np.abs(got - ref)
    if out_dtype == "f32":
        return float((diff - ATTN_ATOL).max()) if diff.size else -1.0
    mag = np.maximum(np.abs(ref), np.abs(got))
    return float((diff - ATTN_ATOL - half_ulp(mag, out_dtype)).max()) if diff.size else -1.0


def assert_attn_close(got: torch.Tensor, ref: np.ndarray, out_dtype: str, what: str = ""):
    g = got.detach().cpu().double().numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    ex = attn_error_excess(g, ref, out_dtype)
    assert ex <= 0, f"{what}: max |err| = {np.abs(g - ref).max():.3e} exceeds the gate by {ex:.3e}"


TORCH_OUT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def oracle_slots(tables: torch.Tensor, seq_idx, pos, block_size: int) -> np.ndarray:
    t = tables.cpu().numpy()
    return np.array([oracle.slot_of(t[s], int(p), block_size) for s, p in zip(seq_idx, pos)], dtype=np.int64)


def bits_equal(a: torch.Tensor, b: np.ndarray) -> bool:
    return np.array_equal(oracle.pool_bits(a.cpu()), b)
