"""pa_decode_static_scratch: paged decode for callers that cannot allocate.

Some users of this library cannot allocate device memory themselves: a
plugin that a host framework hands only its input and output buffers (the
framework owns every byte of device memory), or code on a latency-critical
path where cudaMalloc / cudaFree would synchronise the device.  For them the
library offers pa_decode_static_scratch, which runs the same decode as
pa_decode but keeps its scratch in a fixed device array inside the library.

These tests call it through the C ABI and check its output against
pa_decode with a caller-allocated workspace, on two different calls in a
row (the array keeps whatever the previous call left in it).  Both run the
same deterministic kernels on the same inputs, so the outputs must be equal
bit for bit; each call is also checked against the fp64 oracle within the
attention tolerance of the other parity tests.  A request larger than the
fixed array must be refused without a launch.  This file is collected last
so that a failure here comes after every other test.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import oracle
import pa_workloads as W
from tests.gpu_common import assert_attn_close

pytestmark = pytest.mark.gpu

OUT_NAME = {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32"}


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_35_gb300 as pa

    torch.cuda.set_device(0)
    return pa


def _code(pa, t):
    return {torch.float16: pa.PA_F16, torch.bfloat16: pa.PA_BF16, torch.float32: pa.PA_F32}[t.dtype]


def _static_call(pa, out, q, kp, vp, tables, ctx, mx, scale, err, partition_size=0):
    """The entry point called directly through the C ABI (ctypes)."""
    NB, H, B, D = kp.shape
    S = q.shape[0]
    return pa.lib().pa_decode_static_scratch(
        out.data_ptr(), _code(pa, out), q.data_ptr(), kp.data_ptr(), vp.data_ptr(), tables.data_ptr(),
        tables.shape[1], ctx.data_ptr(), mx, S, H, D, B, NB, ctypes.c_float(scale), _code(pa, kp), partition_size,
        err.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _compare_one(pa, w, partition_size, out_dtype):
    dev = torch.device("cuda")
    kp, vp, q = w.k_pool.to(dev), w.v_pool.to(dev), w.q.to(dev)
    tables, ctx = w.block_tables.to(dev), w.context_lens.to(dev)
    mx = int(w.context_lens.max())
    S, H, D = w.num_seqs, w.num_heads, w.head_dim
    err = pa.new_error_flag()
    ref = torch.empty(S, H, D, dtype=out_dtype, device=dev)
    ws = pa.decode_workspace(S, H, D, mx, partition_size)
    pa.pa_decode(ref, q, kp, vp, tables, ctx, mx, w.scale, ws, err, partition_size=partition_size)
    assert pa.pa_get_error(err) == 0
    got = torch.full((S, H, D), float("nan"), dtype=out_dtype, device=dev)
    st = _static_call(pa, got, q, kp, vp, tables, ctx, mx, w.scale, err, partition_size)
    assert st == pa.PA_OK, pa.status_string(st)
    assert pa.pa_get_error(err) == 0
    assert torch.equal(got.view(torch.uint8), ref.view(torch.uint8))
    # and the fp64 oracle over the same pools
    kb, vb = oracle.pool_bits(kp.cpu()), oracle.pool_bits(vp.cpu())
    expect = oracle.decode(w.q.cpu(), kb, vb, w.block_tables, w.context_lens, w.block_size, w.scale, w.dtype)
    assert_attn_close(got, expect, OUT_NAME[out_dtype], "static-scratch decode")


def test_static_scratch_matches_pa_decode_on_two_calls_in_a_row(pa):
    # first call: the LLaMA-13B-shaped batch (64 x 40 heads, contexts to 2048)
    _compare_one(pa, W.llama13b_decode(device="cuda"), 0, torch.float16)
    # second call, right after, with other sizes, dtypes and many partitions:
    # whatever the first call left in the shared array must not leak in
    _compare_one(pa, W.small_decode(ctx=(1, 17, 300, 1029, 2100), H=3, D=64, dtype="bf16"), 16, torch.float32)


def test_static_scratch_refuses_requests_beyond_its_size(pa):
    S, H, D, mx = 256, 32, 128, 16384
    assert pa.pa_decode_workspace_bytes(S, H, D, mx) > pa.lib().pa_decode_workspace_bytes(1, 1, 64, 1, 0)
    need = pa.pa_decode_workspace_bytes(S, H, D, mx)
    assert need > 16 * 1024 * 1024
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: the call must refuse before any launch
    st = pa.lib().pa_decode_static_scratch(fake, pa.PA_BF16, fake, fake, fake, fake, 1024, fake, mx, S, H, D, 16,
                                           100000, ctypes.c_float(0.088), pa.PA_BF16, 0, fake, None)
    assert st == pa.PA_ERR_WORKSPACE
