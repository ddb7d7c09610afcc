"""Host-side logic of bench.py (no GPU): byte accounting pinned to the
pages' figures, the multi-rank timing reduction over gloo, and the clock
record parsing."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    vals = {}
    with open(os.path.join(GOLDEN, "kv_bytes_per_token.txt"), encoding="utf-8") as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return vals


def test_kv_bytes_per_token_matches_the_pages():
    g = _golden()
    per_token = bench.kv_bytes_per_token(int(g["layers"]), int(g["heads"]), int(g["head_dim"]),
                                         int(g["bytes_per_element"]))
    assert per_token == int(g["bytes_per_token"])
    # one layer of the decode byte count, times the layer count, is the same figure
    one_layer = bench.decode_bytes([1], int(g["heads"]), int(g["head_dim"]), 16, int(g["bytes_per_element"]))
    kv_part = one_layer - 2 * int(g["heads"]) * int(g["head_dim"]) * 2 - 4 - 4
    assert kv_part * int(g["layers"]) == per_token
    request = per_token * int(g["request_tokens"])
    assert abs(request / 2 ** 30 - g["request_gb_approx"]) < 0.05


def test_decode_and_scatter_bytes_by_hand():
    # two sequences of 17 and 32 tokens, 2 heads x 64, fp16, block 16
    b = bench.decode_bytes([17, 32], 2, 64, 16, 2)
    kv = 2 * (17 + 32) * 2 * 64 * 2
    qo = 2 * 2 * 2 * 64 * 2
    tables = 4 * (2 + 2)
    assert b == kv + qo + tables + 8
    assert bench.scatter_bytes(3, 2, 64, 2) == 4 * 3 * 2 * 64 * 2 + 24


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    r, w, local = bench.dist_setup()
    bench.dist_barrier(w)
    got = bench.dist_max(10.0 + 5.0 * r, w)
    q.put((r, w, local, got))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_replicas_reduce_the_max_time_over_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == world for r in res)
    assert all(r[3] == 15.0 for r in res)


def test_clock_summary_flags_throttle_reasons():
    cs = bench.ClockSampler(0)
    cs.samples = [
        (1.0, ["0", "2070", "2070", "400.1", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]),
        (2.0, ["0", "1900", "2070", "1390.0", "0x4", "Not Active", "Not Active", "Not Active", "Active"]),
        (5.0, ["0", "1000", "2070", "100.0", "0x0", "Active", "Not Active", "Not Active", "Not Active"]),
    ]
    s = cs.summary(0.5, 3.0)
    assert s["samples"] == 2 and s["sm_mhz"] == 1985.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    s = cs.summary(10.0, 11.0)  # no sample inside: falls back to the whole run
    assert s["samples"] == 3 and "hw_slowdown" in s["reasons"]


def test_grouped_decode_bytes():
    """Without shared prefixes the grouped call reads what pa_decode reads
    (plus the group arrays); a group of n members sharing p tokens reads
    those tokens' K/V and table entries once instead of n times."""
    import bench

    ctx, H, D, B, elt = [40, 700, 1029, 16], 3, 128, 16, 2
    plain = bench.decode_bytes(ctx, H, D, B, elt)
    assert bench.grouped_decode_bytes(ctx, [0, 4], [0], H, D, B, elt) == plain + 4 * 3
    ctx = [1000 + 5, 1000 + 200, 1000 + 77]
    shared = 992
    got = bench.grouped_decode_bytes(ctx, [0, 3], [shared], H, D, B, elt)
    saved_kv = 2 * shared * H * D * elt * (3 - 1)
    saved_tables = 4 * (shared // B) * (3 - 1)
    assert got == bench.decode_bytes(ctx, H, D, B, elt) - saved_kv - saved_tables + 4 * 3
