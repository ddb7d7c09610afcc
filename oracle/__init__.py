"""CPU oracle for the paged KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference leg of ``bench.py`` may import this package.
The CUDA library and its Python binding never import it, and it imports
nothing from them.

Contents:
  * ``pa_oracle.c``     -- plain fp64 C: reassembly + attention (decode and
                           causal chunked prefill), slot scatter, block copy,
                           block swap between two pools.
                           Built into ``liboracle.so`` by ``build()``.
  * ``reference_np.py`` -- an independent numpy restatement of the same
                           definitions, plus the split-KV combine identity.
  * ``alloc_model.py``  -- the block manager's semantics (free list, reference
                           counts, copy-on-write) as a Python model.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liboracle.so")
SRC_PATH = os.path.join(HERE, "pa_oracle.c")

_DT = {"f16": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile pa_oracle.c with gcc (-O2, no fast-math, OpenMP if available)."""
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= os.path.getmtime(SRC_PATH):
        return LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", SRC_PATH, "-o", LIB_PATH, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    return LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        i = ctypes.c_int
        L.oracle_decode.argtypes = [P, P, P, P, P, i, P, i, i, i, i, i, ctypes.c_double, i]
        L.oracle_prefill.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, i, ctypes.c_double, i]
        L.oracle_reshape_and_cache.argtypes = [P, P, P, P, P, i, i, i, i, i]
        L.oracle_copy_blocks.argtypes = [P, P, P, i, i, i, i, i]
        L.oracle_swap_blocks.argtypes = [P, P, i, P, P, i, P, i, i, i, i]
        L.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_f16_to_double.restype = ctypes.c_double
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = ctypes.c_double
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_set_num_threads.argtypes = [i]
        L.oracle_set_num_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> int:
    """Threads of the oracle's OpenMP loops from now on; returns the count in effect."""
    return int(lib().oracle_set_num_threads(int(n)))


def _bits(t) -> np.ndarray:
    """Raw 16-bit patterns of a CPU torch fp16/bf16 tensor (or uint16 array)."""
    if isinstance(t, np.ndarray):
        return np.ascontiguousarray(t.view(np.uint16))
    import torch
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(a) -> np.ndarray:
    if not isinstance(a, np.ndarray):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with status {rc}")


def decode(q, k_pool, v_pool, block_tables, context_lens, block_size, scale, dtype) -> np.ndarray:
    """fp64 decode attention; tensors may be torch (CPU) or numpy bit arrays."""
    qb, kb, vb = _bits(q), _bits(k_pool), _bits(v_pool)
    S, H, D = q.shape
    NB = k_pool.shape[0]
    tb, cl = _i32(block_tables), _i32(context_lens)
    out = np.zeros((S, H, D), dtype=np.float64)
    rc = lib().oracle_decode(_ptr(out), _ptr(qb), _ptr(kb), _ptr(vb), _ptr(tb), tb.shape[1], _ptr(cl),
                             S, H, D, block_size, NB, float(scale), _DT[dtype])
    _check(rc, "decode")
    return out


def prefill(q, cu_q_lens, ctx_before, k_pool, v_pool, block_tables, block_size, scale, dtype) -> np.ndarray:
    qb, kb, vb = _bits(q), _bits(k_pool), _bits(v_pool)
    T, H, D = q.shape
    NB = k_pool.shape[0]
    cu, cb, tb = _i32(cu_q_lens), _i32(ctx_before), _i32(block_tables)
    out = np.zeros((T, H, D), dtype=np.float64)
    rc = lib().oracle_prefill(_ptr(out), _ptr(qb), _ptr(cu), _ptr(cb), _ptr(kb), _ptr(vb), _ptr(tb), tb.shape[1],
                              len(cb), H, D, block_size, NB, float(scale), _DT[dtype])
    _check(rc, "prefill")
    return out


def reshape_and_cache(k_new, v_new, k_bits: np.ndarray, v_bits: np.ndarray, slot_mapping, block_size):
    """In place on uint16 pool arrays [NB][H][B][D]."""
    kn, vn = _bits(k_new), _bits(v_new)
    T, H, D = k_new.shape
    sm = slot_mapping if isinstance(slot_mapping, np.ndarray) else slot_mapping.detach().cpu().numpy()
    sm = np.ascontiguousarray(sm, dtype=np.int64)
    rc = lib().oracle_reshape_and_cache(_ptr(kn), _ptr(vn), _ptr(k_bits), _ptr(v_bits), _ptr(sm), T, H, D,
                                        block_size, k_bits.shape[0])
    _check(rc, "reshape_and_cache")


def copy_blocks(k_bits: np.ndarray, v_bits: np.ndarray, pairs, block_size):
    pr = _i32(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    NB, H, B, D = k_bits.shape
    rc = lib().oracle_copy_blocks(_ptr(k_bits), _ptr(v_bits), _ptr(pr), pr.shape[0], H, D, B, NB)
    _check(rc, "copy_blocks")


def swap_blocks(src_k: np.ndarray, src_v: np.ndarray, dst_k: np.ndarray, dst_v: np.ndarray, pairs) -> int:
    """dst block d := src block s for each (s, d) in pairs (uint16 pool bits,
    [blocks][H][B][D]); pairs with an id outside its pool are skipped.
    Returns the number of skipped pairs."""
    pr = _i32(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    NBs, H, B, D = src_k.shape
    for a in (src_k, src_v, dst_k, dst_v):
        if a.dtype != np.uint16 or not a.flags["C_CONTIGUOUS"] or tuple(a.shape[1:]) != (H, B, D):
            raise ValueError("pools must be C-contiguous uint16 [blocks][H][B][D]")
    return int(lib().oracle_swap_blocks(_ptr(src_k), _ptr(src_v), NBs, _ptr(dst_k), _ptr(dst_v), dst_k.shape[0],
                                        _ptr(pr), pr.shape[0], H, D, B))


def slot_of(table_row, pos: int, block_size: int) -> int:
    """Slot index of 0-based position ``pos``: table[pos // B] * B + pos % B."""
    return int(table_row[pos // block_size]) * block_size + pos % block_size


def pool_bits(t) -> np.ndarray:
    """Writable uint16 copy of a pool tensor's bits."""
    return _bits(t).copy()
