"""Python binding of libpa (paged KV-cache attention for GB300, sm_103a).

Argument marshalling only: every function here checks shapes and dtypes,
takes raw device pointers from torch tensors and the current CUDA stream,
and calls the C ABI declared in ``include/pa.h``.  All computation runs in
the library's CUDA kernels (or, for the block allocator, its host C++).
There is no fallback: if ``libpa.so`` has not been built, every call raises.

Names match the C entry points: ``pa_reshape_and_cache``, ``pa_copy_blocks``,
``pa_swap_blocks``, ``pa_decode``, ``pa_decode_static_scratch``,
``pa_prefill_chunk``, ``pa_mixed_step``, ``pa_check_decode_inputs``,
``pa_check_prefill_inputs``, ``pa_get_error``, ``pa_slot_mapping``; the
``pa_decode_graphs_*`` graph cache is wrapped by :class:`DecodeGraphs` and the
``pa_alloc_*`` allocator (with its optional prefix cache) by
:class:`BlockAllocator`.  ``memsim`` is a host-only memory-waste simulator
built on the allocator.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpa.so")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_NO_FREE_BLOCKS = 3
PA_ERR_REFCOUNT = 4
PA_ERR_BAD_INDEX = 5
PA_ERR_CUDA = 6
PA_ERR_TIMEOUT = 7
PA_ERR_WORKSPACE = 8

PA_F16, PA_BF16, PA_F32 = 0, 1, 2
PA_ALLOC_PREFIX_CACHE = 1

PA_FLAG_BAD_BLOCK = 1
PA_FLAG_BAD_SLOT = 2
PA_FLAG_BAD_LENGTH = 4
PA_FLAG_TIMEOUT = 8
PA_FLAG_BAD_GROUP = 16

_TORCH_TO_PA = {torch.float16: PA_F16, torch.bfloat16: PA_BF16, torch.float32: PA_F32}

# Every function the header declares, with its ctypes signature.
_P, _I, _L, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "pa_version": ([], _I),
    "pa_status_string": ([_I], ctypes.c_char_p),
    "pa_device_sm_count": ([], _I),
    "pa_reshape_and_cache": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "pa_copy_blocks": ([_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "pa_decode_partition_size": ([_I, _I, _I], _I),
    "pa_decode_workspace_bytes": ([_I, _I, _I, _I, _I], _Z),
    "pa_decode": ([_P, _I, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _Z, _I, _P, _P], _I),
    "pa_decode_static_scratch": ([_P, _I, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _P], _I),
    "pa_decode_grouped_workspace_bytes": ([_I, _I, _I, _I, _I], _Z),
    "pa_decode_grouped": ([_P, _I, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _P, _I, _P, _Z, _I,
                           _P, _P], _I),
    "pa_prefill_chunk": ([_P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _P], _I),
    "pa_mixed_step": ([_P, _I, _P, _P, _I, _P, _I, _I, _P, _Z, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _I,
                       _I, _I, _F, _I, _I, _P, _P], _I),
    "pa_swap_blocks": ([_P, _P, _I, _P, _P, _I, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "pa_decode_graphs_workspace_bytes": ([_I, _I, _I, _I, _I, _I], _Z),
    "pa_decode_graphs_create": ([_P, _I, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _Z, _I, _I, _P,
                                 _P], _I),
    "pa_decode_graphs_run": ([_P, _I, _I, _P], _I),
    "pa_decode_graphs_count": ([_P], _I),
    "pa_decode_graphs_destroy": ([_P], None),
    "pa_check_decode_inputs": ([_P, _I, _P, _I, _I, _I, _I, _P, _P], _I),
    "pa_check_prefill_inputs": ([_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "pa_selftest_wait_timeout": ([_P, _P, _P, _P], _I),
    "pa_get_error": ([_P, _P, _P], _I),
    "pa_slot_mapping": ([_P, _I, _I, _I, _P, _P, _I, _P], _I),
    "pa_alloc_create": ([_I, _I, _P], _I),
    "pa_alloc_destroy": ([_P], None),
    "pa_alloc_add_seq": ([_P, _I], _I),
    "pa_alloc_fork": ([_P, _I, _I], _I),
    "pa_alloc_append_slots": ([_P, _P, _I, _P, _P, _P], _I),
    "pa_alloc_free_seq": ([_P, _I], _I),
    "pa_alloc_block_table": ([_P, _I, _P, _I, _P, _P], _I),
    "pa_alloc_block_tables": ([_P, _P, _I, _I, _P, _P], _I),
    "pa_alloc_num_free": ([_P], _I),
    "pa_alloc_ref": ([_P, _I], _I),
    "pa_alloc_num_seqs": ([_P], _I),
    "pa_alloc_create_ex": ([_I, _I, _I, _P], _I),
    "pa_alloc_add_seq_prefix": ([_P, _I, _P, _I, _P], _I),
    "pa_alloc_append_tokens": ([_P, _P, _P, _I, _P, _P, _P], _I),
    "pa_alloc_prefix_stats": ([_P, _P, _P], _I),
    "pa_alloc_prefix_groups": ([_P, _P, _I, _I, _P, _P, _P], _I),
}


class PAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C-ABI library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -c \"import __graft_entry__ as g; g.build()\"`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().pa_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != PA_OK:
        raise PAError(status, what)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str, dtype=None, ndim=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, has {t.dim()}")
    return t.data_ptr()


def _kv_code(t: torch.Tensor) -> int:
    if t.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError(f"K/V/q must be float16 or bfloat16, got {t.dtype}")
    return _TORCH_TO_PA[t.dtype]


def new_error_flag(device=None) -> torch.Tensor:
    """A zeroed device int32 for the kernels' error bits."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


# ---- GPU entry points ---------------------------------------------------------------

def pa_reshape_and_cache(k_new, v_new, k_pool, v_pool, slot_mapping, err_flag, stream=None):
    """Scatter k_new/v_new [T][H][D] into pools [NB][H][B][D] at slot_mapping[T] (int64)."""
    NB, H, B, D = k_pool.shape
    T = k_new.shape[0]
    if tuple(k_new.shape) != (T, H, D) or tuple(v_new.shape) != (T, H, D) or v_pool.shape != k_pool.shape:
        raise ValueError("shape mismatch")
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [num_tokens]")
    dt = _kv_code(k_pool)
    st = lib().pa_reshape_and_cache(
        _dev(k_new, "k_new", k_pool.dtype), _dev(v_new, "v_new", k_pool.dtype), _dev(k_pool, "k_pool"),
        _dev(v_pool, "v_pool", k_pool.dtype), _dev(slot_mapping, "slot_mapping", torch.int64), T, H, D, B, NB, dt,
        _dev(err_flag, "err_flag", torch.int32), _stream(stream))
    _check(st, "pa_reshape_and_cache")


def pa_copy_blocks(k_pool, v_pool, pairs, err_flag, stream=None):
    """Copy whole blocks: pairs int32 [n][2] of (src, dst)."""
    NB, H, B, D = k_pool.shape
    n = pairs.shape[0] if pairs.numel() else 0
    if n and tuple(pairs.shape) != (n, 2):
        raise ValueError("pairs must be [n][2]")
    st = lib().pa_copy_blocks(
        _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool", k_pool.dtype),
        _dev(pairs, "pairs", torch.int32) if n else None, n, H, D, B, NB, _kv_code(k_pool),
        _dev(err_flag, "err_flag", torch.int32), _stream(stream))
    _check(st, "pa_copy_blocks")


def _pool_ptr(t: torch.Tensor, name: str, dtype=None) -> int:
    """Address of a pool that lives on the GPU or in pinned host memory."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a tensor")
    if t.is_cuda:
        return _dev(t, name, dtype)
    if not t.is_pinned():
        raise ValueError(f"{name} must be a CUDA tensor or a pinned host tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    return t.data_ptr()


def pa_swap_blocks(src_k, src_v, dst_k, dst_v, pairs, err_flag, stream=None):
    """Copy whole blocks from pool src to pool dst: pairs int32 [n][2] of
    (src block, dst block) on the GPU.  Either pool may be a pinned host
    tensor ([blocks][H][B][D], same per-block shape and dtype)."""
    NBs, H, B, D = src_k.shape
    NBd = dst_k.shape[0]
    if src_v.shape != src_k.shape or dst_v.shape != dst_k.shape or tuple(dst_k.shape[1:]) != (H, B, D):
        raise ValueError("pool shape mismatch")
    n = pairs.shape[0] if pairs.numel() else 0
    if n and tuple(pairs.shape) != (n, 2):
        raise ValueError("pairs must be [n][2]")
    st = lib().pa_swap_blocks(
        _pool_ptr(src_k, "src_k"), _pool_ptr(src_v, "src_v", src_k.dtype), NBs, _pool_ptr(dst_k, "dst_k", src_k.dtype),
        _pool_ptr(dst_v, "dst_v", src_k.dtype), NBd, _dev(pairs, "pairs", torch.int32) if n else None, n, H, D, B,
        _kv_code(src_k), _dev(err_flag, "err_flag", torch.int32), _stream(stream))
    _check(st, "pa_swap_blocks")


def pa_decode_partition_size(num_seqs: int, num_heads: int, max_context_len: int) -> int:
    return int(lib().pa_decode_partition_size(num_seqs, num_heads, max_context_len))


def pa_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, partition_size=0) -> int:
    return int(lib().pa_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, partition_size))


def decode_workspace(num_seqs, num_heads, head_dim, max_context_len, partition_size=0, device=None):
    """A uint8 device tensor big enough for pa_decode with these sizes."""
    n = pa_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, partition_size)
    if n == 0:
        raise ValueError("bad sizes for the decode workspace")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def pa_decode(out, q, k_pool, v_pool, block_tables, context_lens, max_context_len, scale, workspace, err_flag,
              partition_size=0, stream=None):
    """out[S][H][D] = paged decode attention of q[S][H][D]."""
    NB, H, B, D = k_pool.shape
    S = q.shape[0]
    if tuple(q.shape) != (S, H, D) or tuple(out.shape) != (S, H, D) or v_pool.shape != k_pool.shape:
        raise ValueError("shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] < S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [>=S][MB], context_lens [S]")
    st = lib().pa_decode(
        _dev(out, "out", (torch.float16, torch.bfloat16, torch.float32)), _TORCH_TO_PA[out.dtype],
        _dev(q, "q", k_pool.dtype), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool", k_pool.dtype),
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), int(max_context_len), S, H, D, B, NB, float(scale),
        _kv_code(k_pool), _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        int(partition_size), _dev(err_flag, "err_flag", torch.int32), _stream(stream))
    _check(st, "pa_decode")


def pa_decode_grouped_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, partition_size=0) -> int:
    return int(lib().pa_decode_grouped_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len,
                                                       partition_size))


def decode_grouped_workspace(num_seqs, num_heads, head_dim, max_context_len, partition_size=0, device=None):
    """A uint8 device tensor big enough for pa_decode_grouped with these sizes."""
    n = pa_decode_grouped_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, partition_size)
    if n == 0:
        raise ValueError("bad sizes for the grouped decode workspace")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def pa_decode_grouped(out, q, k_pool, v_pool, block_tables, context_lens, max_context_len, scale, group_start,
                      group_prefix, workspace, err_flag, partition_size=0, stream=None):
    """pa_decode with each group's shared prefix read once for the group:
    sequences group_start[g] .. group_start[g+1]-1 share their first
    group_prefix[g] tokens (device int32 [G+1] and [G]; see pa.h)."""
    NB, H, B, D = k_pool.shape
    S = q.shape[0]
    if tuple(q.shape) != (S, H, D) or tuple(out.shape) != (S, H, D) or v_pool.shape != k_pool.shape:
        raise ValueError("shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] < S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [>=S][MB], context_lens [S]")
    G = group_prefix.numel()
    if group_start.numel() != G + 1:
        raise ValueError("group_start must hold num_groups + 1 entries")
    st = lib().pa_decode_grouped(
        _dev(out, "out", (torch.float16, torch.bfloat16, torch.float32)), _TORCH_TO_PA[out.dtype],
        _dev(q, "q", k_pool.dtype), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool", k_pool.dtype),
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), int(max_context_len), S, H, D, B, NB, float(scale),
        _kv_code(k_pool), _dev(group_start, "group_start", torch.int32), _dev(group_prefix, "group_prefix", torch.int32),
        G, _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(), int(partition_size),
        _dev(err_flag, "err_flag", torch.int32), _stream(stream))
    _check(st, "pa_decode_grouped")


def pa_decode_static_scratch(out, q, k_pool, v_pool, block_tables, context_lens, max_context_len, scale, err_flag,
                             partition_size=0, stream=None):
    """pa_decode with the library's fixed device scratch instead of a caller
    workspace, for callers that cannot allocate device memory (see pa.h)."""
    NB, H, B, D = k_pool.shape
    S = q.shape[0]
    if tuple(q.shape) != (S, H, D) or tuple(out.shape) != (S, H, D) or v_pool.shape != k_pool.shape:
        raise ValueError("shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] < S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [>=S][MB], context_lens [S]")
    st = lib().pa_decode_static_scratch(
        _dev(out, "out", (torch.float16, torch.bfloat16, torch.float32)), _TORCH_TO_PA[out.dtype],
        _dev(q, "q", k_pool.dtype), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool", k_pool.dtype),
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), int(max_context_len), S, H, D, B, NB, float(scale),
        _kv_code(k_pool), int(partition_size), _dev(err_flag, "err_flag", torch.int32), _stream(stream))
    _check(st, "pa_decode_static_scratch")


def pa_prefill_chunk(out, q, cu_q_lens, ctx_before, k_pool, v_pool, block_tables, max_q_len, scale, err_flag,
                     stream=None):
    """Causal attention of prefill chunks: q, out [total][H][D]."""
    NB, H, B, D = k_pool.shape
    T = q.shape[0]
    C = ctx_before.shape[0]
    if tuple(q.shape) != (T, H, D) or tuple(out.shape) != (T, H, D) or cu_q_lens.shape != (C + 1,):
        raise ValueError("shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] < C:
        raise ValueError("block_tables must be [>=C][MB]")
    st = lib().pa_prefill_chunk(
        _dev(out, "out", (torch.float16, torch.bfloat16, torch.float32)), _TORCH_TO_PA[out.dtype],
        _dev(q, "q", k_pool.dtype), _dev(cu_q_lens, "cu_q_lens", torch.int32),
        _dev(ctx_before, "ctx_before", torch.int32), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool", k_pool.dtype),
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1], C, T, int(max_q_len), H, D, B, NB,
        float(scale), _kv_code(k_pool), _dev(err_flag, "err_flag", torch.int32), _stream(stream))
    _check(st, "pa_prefill_chunk")


def pa_mixed_step(dec_out, dec_q, dec_block_tables, context_lens, max_context_len, workspace, pf_out, pf_q,
                  cu_q_lens, ctx_before, pf_block_tables, max_q_len, k_pool, v_pool, scale, err_flag,
                  prefill_sms=0, stream=None):
    """Decode of dec_q [S][H][D] and prefill of the chunks in pf_q [total][H][D]
    over the same pools, running concurrently on `stream` (the prefill on at
    most prefill_sms SMs, 0 = the default share)."""
    NB, H, B, D = k_pool.shape
    S = dec_q.shape[0]
    T = pf_q.shape[0]
    C = ctx_before.shape[0]
    if tuple(dec_q.shape) != (S, H, D) or tuple(dec_out.shape) != (S, H, D) or v_pool.shape != k_pool.shape:
        raise ValueError("decode shape mismatch")
    if dec_block_tables.dim() != 2 or dec_block_tables.shape[0] < S or context_lens.shape != (S,):
        raise ValueError("dec_block_tables must be [>=S][MB], context_lens [S]")
    if tuple(pf_q.shape) != (T, H, D) or tuple(pf_out.shape) != (T, H, D) or cu_q_lens.shape != (C + 1,):
        raise ValueError("prefill shape mismatch")
    if pf_block_tables.dim() != 2 or pf_block_tables.shape[0] < C:
        raise ValueError("pf_block_tables must be [>=C][MB]")
    st = lib().pa_mixed_step(
        _dev(dec_out, "dec_out", (torch.float16, torch.bfloat16, torch.float32)), _TORCH_TO_PA[dec_out.dtype],
        _dev(dec_q, "dec_q", k_pool.dtype), _dev(dec_block_tables, "dec_block_tables", torch.int32),
        dec_block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32), int(max_context_len), S,
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _dev(pf_out, "pf_out", (torch.float16, torch.bfloat16, torch.float32)), _TORCH_TO_PA[pf_out.dtype],
        _dev(pf_q, "pf_q", k_pool.dtype), _dev(cu_q_lens, "cu_q_lens", torch.int32),
        _dev(ctx_before, "ctx_before", torch.int32), _dev(pf_block_tables, "pf_block_tables", torch.int32),
        pf_block_tables.shape[1], C, T, int(max_q_len), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool", k_pool.dtype),
        H, D, B, NB, float(scale), _kv_code(k_pool), int(prefill_sms), _dev(err_flag, "err_flag", torch.int32),
        _stream(stream))
    _check(st, "pa_mixed_step")


def pa_check_decode_inputs(block_tables, context_lens, max_context_len, block_size, num_blocks, stream=None):
    """Host-side check of a decode's tables and lengths (synchronises the
    stream).  Returns None, or (sequence, logical block) of the first bad
    entry (logical block -1: a bad length)."""
    S = context_lens.shape[0]
    bad = np.zeros(2, dtype=np.int64)
    st = lib().pa_check_decode_inputs(_dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
                                      _dev(context_lens, "context_lens", torch.int32), S, int(max_context_len),
                                      int(block_size), int(num_blocks), _stream(stream), bad.ctypes.data)
    if st == PA_ERR_BAD_INDEX:
        return int(bad[0]), int(bad[1])
    _check(st, "pa_check_decode_inputs")
    return None


def pa_check_prefill_inputs(cu_q_lens, ctx_before, block_tables, total_q, max_q_len, block_size, num_blocks,
                            stream=None):
    """Host-side check of a prefill's chunk bounds and tables (synchronises
    the stream).  Returns None, or (chunk, logical block) of the first bad
    entry (logical block -1: a bad length; (-1, -1): bad cu_q_lens ends)."""
    C = ctx_before.shape[0]
    bad = np.zeros(2, dtype=np.int64)
    st = lib().pa_check_prefill_inputs(_dev(cu_q_lens, "cu_q_lens", torch.int32),
                                       _dev(ctx_before, "ctx_before", torch.int32),
                                       _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1], C,
                                       int(total_q), int(max_q_len), int(block_size), int(num_blocks),
                                       _stream(stream), bad.ctypes.data)
    if st == PA_ERR_BAD_INDEX:
        return int(bad[0]), int(bad[1])
    _check(st, "pa_check_prefill_inputs")
    return None


def pa_get_error(err_flag, stream=None) -> int:
    """Synchronise, read and clear the device error flag; returns its bits."""
    bits = ctypes.c_int32(0)
    st = lib().pa_get_error(_dev(err_flag, "err_flag", torch.int32), ctypes.addressof(bits), _stream(stream))
    if st not in (PA_OK, PA_ERR_BAD_INDEX, PA_ERR_TIMEOUT):
        raise PAError(st, "pa_get_error")
    return int(bits.value)


# ---- host entry points --------------------------------------------------------------

def _host_i32(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def pa_slot_mapping(block_tables, seq_idx, pos, block_size: int) -> np.ndarray:
    """Host slots of (sequence row, position) pairs through host block tables."""
    tb = _host_i32(block_tables)
    si = _host_i32(seq_idx)
    ps = _host_i32(pos)
    out = np.zeros(si.shape[0], dtype=np.int64)
    st = lib().pa_slot_mapping(tb.ctypes.data, tb.shape[0], tb.shape[1], block_size, si.ctypes.data, ps.ctypes.data,
                               si.shape[0], out.ctypes.data)
    _check(st, "pa_slot_mapping")
    return out


class DecodeGraphs:
    """pa_decode recorded once per padded (sequence count, KV length) shape
    and replayed (see pa.h).  Owns the static device buffers the graphs use:
    write the step's rows into .q, .tables and .context_lens, then run()."""

    def __init__(self, k_pool, v_pool, max_seqs, max_context_len, max_blocks_per_seq, scale, err_flag,
                 seq_interval=8, kv_interval=256, out_dtype=None):
        NB, H, B, D = k_pool.shape
        dev = k_pool.device
        s_max = -(-max_seqs // seq_interval) * seq_interval
        self.k_pool, self.v_pool, self.err_flag = k_pool, v_pool, err_flag
        self.q = torch.zeros(s_max, H, D, dtype=k_pool.dtype, device=dev)
        self.out = torch.zeros(s_max, H, D, dtype=out_dtype or k_pool.dtype, device=dev)
        self.tables = torch.full((s_max, max_blocks_per_seq), -1, dtype=torch.int32, device=dev)
        self.context_lens = torch.zeros(s_max, dtype=torch.int32, device=dev)
        n = int(lib().pa_decode_graphs_workspace_bytes(max_seqs, H, D, max_context_len, seq_interval, kv_interval))
        if n == 0:
            raise ValueError("bad sizes for decode graphs")
        self.workspace = torch.empty(n, dtype=torch.uint8, device=dev)
        h = ctypes.c_void_p()
        st = lib().pa_decode_graphs_create(
            _dev(self.out, "out"), _TORCH_TO_PA[self.out.dtype], _dev(self.q, "q"), _dev(k_pool, "k_pool"),
            _dev(v_pool, "v_pool", k_pool.dtype), _dev(self.tables, "tables"), max_blocks_per_seq,
            _dev(self.context_lens, "context_lens"), max_seqs, max_context_len, H, D, B, NB, float(scale),
            _kv_code(k_pool), _dev(self.workspace, "workspace"), n, seq_interval, kv_interval,
            _dev(err_flag, "err_flag", torch.int32), ctypes.byref(h))
        _check(st, "pa_decode_graphs_create")
        self._h = h

    def run(self, num_seqs: int, max_context_len: int, stream=None):
        _check(lib().pa_decode_graphs_run(self._h, int(num_seqs), int(max_context_len), _stream(stream)),
               "pa_decode_graphs_run")

    @property
    def count(self) -> int:
        return int(lib().pa_decode_graphs_count(self._h))

    def close(self):
        if getattr(self, "_h", None):
            lib().pa_decode_graphs_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class BlockAllocator:
    """Host block manager (free list, reference counts, copy-on-write)."""

    def __init__(self, num_blocks: int, block_size: int, prefix_cache: bool = False):
        self.block_size = block_size
        self.num_blocks = num_blocks
        h = ctypes.c_void_p()
        flags = PA_ALLOC_PREFIX_CACHE if prefix_cache else 0
        _check(lib().pa_alloc_create_ex(num_blocks, block_size, flags, ctypes.byref(h)), "pa_alloc_create_ex")
        self._h = h

    def close(self):
        if self._h:
            lib().pa_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_seq(self, seq_id: int):
        _check(lib().pa_alloc_add_seq(self._h, seq_id), "pa_alloc_add_seq")

    def fork(self, parent: int, child: int):
        _check(lib().pa_alloc_fork(self._h, parent, child), "pa_alloc_fork")

    def append_slots(self, seq_ids):
        """One token per listed sequence -> (slots int64 [n], pairs int32 [k][2])."""
        ids = _host_i32(list(seq_ids))
        n = ids.shape[0]
        slots = np.zeros(n, dtype=np.int64)
        pairs = np.zeros((max(n, 1), 2), dtype=np.int32)
        npairs = ctypes.c_int(0)
        _check(lib().pa_alloc_append_slots(self._h, ids.ctypes.data, n, slots.ctypes.data, pairs.ctypes.data,
                                           ctypes.byref(npairs)), "pa_alloc_append_slots")
        return slots, pairs[: npairs.value].copy()

    def add_seq_prefix(self, seq_id: int, tokens) -> int:
        """New sequence with prompt ``tokens``; returns how many leading tokens
        it reuses from cached blocks (their K/V need no prefill)."""
        ids = _host_i32(list(tokens))
        reused = ctypes.c_int(0)
        _check(lib().pa_alloc_add_seq_prefix(self._h, seq_id, ids.ctypes.data if ids.size else None, ids.shape[0],
                                             ctypes.byref(reused)), "pa_alloc_add_seq_prefix")
        return reused.value

    def append_tokens(self, seq_ids, token_ids):
        """append_slots with the appended tokens' ids (for the prefix cache)."""
        ids = _host_i32(list(seq_ids))
        toks = _host_i32(list(token_ids))
        n = ids.shape[0]
        if toks.shape[0] != n:
            raise ValueError("one token id per sequence")
        slots = np.zeros(n, dtype=np.int64)
        pairs = np.zeros((max(n, 1), 2), dtype=np.int32)
        npairs = ctypes.c_int(0)
        _check(lib().pa_alloc_append_tokens(self._h, ids.ctypes.data, toks.ctypes.data, n, slots.ctypes.data,
                                            pairs.ctypes.data, ctypes.byref(npairs)), "pa_alloc_append_tokens")
        return slots, pairs[: npairs.value].copy()

    def prefix_stats(self):
        """(blocks holding a cache entry, of which free)."""
        c, f = ctypes.c_int(0), ctypes.c_int(0)
        _check(lib().pa_alloc_prefix_stats(self._h, ctypes.byref(c), ctypes.byref(f)), "pa_alloc_prefix_stats")
        return c.value, f.value

    def free_seq(self, seq_id: int):
        _check(lib().pa_alloc_free_seq(self._h, seq_id), "pa_alloc_free_seq")

    def block_table(self, seq_id: int):
        nb, ln = ctypes.c_int(0), ctypes.c_int(0)
        lib().pa_alloc_block_table(self._h, seq_id, None, 0, ctypes.byref(nb), ctypes.byref(ln))
        out = np.zeros(max(nb.value, 1), dtype=np.int32)
        _check(lib().pa_alloc_block_table(self._h, seq_id, out.ctypes.data, out.shape[0], ctypes.byref(nb),
                                          ctypes.byref(ln)), "pa_alloc_block_table")
        return out[: nb.value].tolist(), ln.value

    def block_tables(self, seq_ids, max_blocks_per_seq: int):
        """(tables int32 [n][max_blocks_per_seq] padded with -1, lengths int32 [n])."""
        ids = _host_i32(list(seq_ids))
        n = ids.shape[0]
        tables = np.zeros((n, max_blocks_per_seq), dtype=np.int32)
        lens = np.zeros(n, dtype=np.int32)
        _check(lib().pa_alloc_block_tables(self._h, ids.ctypes.data, n, max_blocks_per_seq, tables.ctypes.data,
                                           lens.ctypes.data), "pa_alloc_block_tables")
        return tables, lens

    def prefix_groups(self, seq_ids, max_group: int = 8):
        """(group_start int32 [G+1], group_prefix int32 [G]) for pa_decode_grouped
        over the batch seq_ids, in that order (see pa_alloc_prefix_groups)."""
        ids = _host_i32(list(seq_ids))
        n = ids.shape[0]
        start = np.zeros(n + 1, dtype=np.int32)
        prefix = np.zeros(max(n, 1), dtype=np.int32)
        g = ctypes.c_int(0)
        _check(lib().pa_alloc_prefix_groups(self._h, ids.ctypes.data, n, int(max_group), start.ctypes.data,
                                            prefix.ctypes.data, ctypes.byref(g)), "pa_alloc_prefix_groups")
        return start[: g.value + 1].copy(), prefix[: g.value].copy()

    def num_free(self) -> int:
        return int(lib().pa_alloc_num_free(self._h))

    def ref(self, block_id: int) -> int:
        return int(lib().pa_alloc_ref(self._h, block_id))

    def num_seqs(self) -> int:
        return int(lib().pa_alloc_num_seqs(self._h))
