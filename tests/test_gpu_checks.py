"""Host-side input validation (pa_check_decode_inputs /
pa_check_prefill_inputs) and the PA_DEBUG mode that runs it before every
decode and prefill launch."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest
import torch

import pa_workloads as W

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_35_gb300 as pa

    torch.cuda.set_device(0)
    return pa


def test_decode_input_check_finds_the_first_bad_entry(pa):
    w = W.small_decode(ctx=(1, 17, 300, 40), H=2, D=64)
    B, NB, mx = w.block_size, w.num_blocks, int(w.context_lens.max())
    tables, ctx = w.block_tables.clone(), w.context_lens.clone()
    dev = torch.device("cuda")
    assert pa.pa_check_decode_inputs(tables.to(dev), ctx.to(dev), mx, B, NB) is None
    # an entry past a sequence's blocks is never read: not an error
    t2 = tables.clone()
    t2[0, -1] = 10 ** 6
    assert pa.pa_check_decode_inputs(t2.to(dev), ctx.to(dev), mx, B, NB) is None
    t2[2, 5] = -7  # sequence 2 (300 tokens) reads blocks 0..18
    t2[3, 1] = NB  # sequence 3 (40 tokens) reads blocks 0..2
    assert pa.pa_check_decode_inputs(t2.to(dev), ctx.to(dev), mx, B, NB) == (2, 5)
    c2 = ctx.clone()
    c2[1] = tables.shape[1] * B + 1  # longer than its table row
    assert pa.pa_check_decode_inputs(tables.to(dev), c2.to(dev), 10 ** 6, B, NB) == (1, -1)
    c2[1] = mx + 1  # past max_context_len
    assert pa.pa_check_decode_inputs(tables.to(dev), c2.to(dev), mx, B, NB) == (1, -1)


def test_prefill_input_check_finds_the_first_bad_entry(pa):
    m = W.small_prefill(chunk_lens=(130, 77), ctx_before=(200, 37), H=2, B=16)
    dev = torch.device("cuda")
    cu = torch.tensor([0, 130, 207], dtype=torch.int32, device=dev)
    cb = m.ctx_before.to(dev)
    tb = m.chunk_tables.clone()
    NB = m.decode.num_blocks
    assert pa.pa_check_prefill_inputs(cu, cb, tb.to(dev), 207, 130, 16, NB) is None
    tb[1, 4] = -1  # chunk 1 covers positions 0..113: blocks 0..7
    assert pa.pa_check_prefill_inputs(cu, cb, tb.to(dev), 207, 130, 16, NB) == (1, 4)
    assert pa.pa_check_prefill_inputs(cu, cb, m.chunk_tables.to(dev), 206, 130, 16, NB) == (-1, -1)
    assert pa.pa_check_prefill_inputs(cu, cb, m.chunk_tables.to(dev), 207, 100, 16, NB) == (0, -1)


SCRIPT = r"""
import torch, pa_workloads as W
import paged_kv_cache_35_gb300 as pa
w = W.small_decode(ctx=(33, 300), H=2, D=64)
dev = torch.device("cuda")
t = w.block_tables.clone(); t[1, 3] = -4
out = torch.zeros(2, 2, 64, dtype=torch.float16, device=dev)
err = pa.new_error_flag()
ws = pa.decode_workspace(2, 2, 64, 300)
try:
    pa.pa_decode(out, w.q.to(dev), w.k_pool.to(dev), w.v_pool.to(dev), t.to(dev), w.context_lens.to(dev), 300,
                 w.scale, ws, err)
    print("launched", pa.pa_get_error(err))
except pa.PAError as e:
    print("refused", e.status, pa.pa_get_error(err))
"""


def _run(env_value):
    env = dict(os.environ)
    env.pop("PA_DEBUG", None)
    if env_value is not None:
        env["PA_DEBUG"] = env_value
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    return r.stdout.strip().splitlines()[-1], r.stderr


def test_pa_debug_refuses_bad_tables_before_any_launch(pa):
    import paged_kv_cache_35_gb300 as pa_mod

    line, err_text = _run("1")
    assert line == f"refused {pa_mod.PA_ERR_BAD_INDEX} 0", line  # nothing ran: the device flag is clear
    assert "sequence 1, logical block 3" in err_text
    line, _ = _run(None)  # without PA_DEBUG the kernel runs, skips the bad chunk and flags it
    assert line == f"launched {pa_mod.PA_FLAG_BAD_BLOCK}", line


def test_a_wait_that_runs_out_flags_timeout_and_the_context_stays_usable(pa):
    """A kernel waits, with the library's bounded wait, on an mbarrier that
    nothing arrives at: after the limit it sets PA_FLAG_TIMEOUT, lets its
    own bulk copy land and exits; then an ordinary decode runs correctly."""
    import ctypes

    dev = torch.device("cuda")
    src = torch.arange(1024, dtype=torch.int32, device=dev)  # 4 KiB
    err = pa.new_error_flag()
    result = torch.full((3,), -2, dtype=torch.int32, device=dev)
    st = pa.lib().pa_selftest_wait_timeout(src.data_ptr(), err.data_ptr(), result.data_ptr(),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == pa.PA_OK
    assert pa.pa_get_error(err) == pa.PA_FLAG_TIMEOUT
    assert result.tolist() == [0, 1, 1023]
    w = W.small_decode(ctx=(5, 300), H=2, D=64)
    out = torch.empty(2, 2, 64, dtype=torch.float32, device=dev)
    ws = pa.decode_workspace(2, 2, 64, 300)
    pa.pa_decode(out, w.q.to(dev), w.k_pool.to(dev), w.v_pool.to(dev), w.block_tables.to(dev),
                 w.context_lens.to(dev), 300, w.scale, ws, err)
    assert pa.pa_get_error(err) == 0
    assert torch.isfinite(out).all()


THREADS_SCRIPT = r"""
import threading
import torch
import paged_kv_cache_35_gb300 as pa
import pa_workloads as W

dev = torch.device("cuda")
torch.cuda.set_device(0)
w = W.small_decode(ctx=(1, 17, 300, 1029), H=2, dtype="bf16")
m = W.small_prefill(chunk_lens=(130, 77), ctx_before=(200, 37), H=3)
S, H, D, mx = w.num_seqs, w.num_heads, w.head_dim, int(w.context_lens.max())
kp, vp, tb, cl, q = (t.to(dev) for t in (w.k_pool, w.v_pool, w.block_tables, w.context_lens, w.q))
mk, mv, mt = m.decode.k_pool.to(dev), m.decode.v_pool.to(dev), m.chunk_tables.to(dev)
cu = torch.cat([torch.zeros(1, dtype=torch.int32), m.chunk_lens.cumsum(0).to(torch.int32)]).to(dev)
cb, mq = m.ctx_before.to(dev), m.chunk_q.to(dev)
T = int(m.chunk_lens.sum())
n = 4
streams = [torch.cuda.Stream() for _ in range(n)]
outs = [torch.empty(S, H, D, dtype=torch.float32, device=dev) for _ in range(n)]
pouts = [torch.empty(T, 3, D, dtype=torch.float32, device=dev) for _ in range(n)]
wss = [pa.decode_workspace(S, H, D, mx) for _ in range(n)]
errs = [pa.new_error_flag() for _ in range(n)]
torch.cuda.synchronize()
start = threading.Barrier(n)
status = [None] * n

def work(i):
    try:
        start.wait()
        # the first decode and prefill calls of this process, from n threads at once
        pa.pa_decode(outs[i], q, kp, vp, tb, cl, mx, w.scale, wss[i], errs[i], stream=streams[i])
        pa.pa_prefill_chunk(pouts[i], mq, cu, cb, mk, mv, mt, int(m.chunk_lens.max()), m.decode.scale, errs[i],
                            stream=streams[i])
        status[i] = "ok"
    except Exception as e:  # reported below
        status[i] = repr(e)

ths = [threading.Thread(target=work, args=(i,)) for i in range(n)]
for t in ths:
    t.start()
for t in ths:
    t.join()
torch.cuda.synchronize()
assert status == ["ok"] * n, status
assert all(pa.pa_get_error(e) == 0 for e in errs)
for i in range(1, n):
    assert torch.equal(outs[i], outs[0]) and torch.equal(pouts[i], pouts[0]), i
assert torch.isfinite(outs[0]).all() and torch.isfinite(pouts[0]).all()
print("threads ok")
"""


def test_first_calls_from_several_host_threads_at_once(pa):
    """The per-device kernel settings are filled on first use; four host
    threads making their first decode and prefill calls at the same time, on
    their own streams, must all launch and agree bit for bit (run in a fresh
    process so that these really are the first calls)."""
    r = subprocess.run([sys.executable, "-c", THREADS_SCRIPT], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip().splitlines()[-1] == "threads ok"
