#!/usr/bin/env python
"""Benchmark of the paged decode hot path on one GB300 (or N replicas).

Workload (the configuration the headline metric is quoted on): a
LLaMA-13B-shaped single layer -- 64 sequences, 40 heads x 128, block size 16,
context lengths uniform in [128, 2048] (seed 1), fp16 K/V/q ~ N(0, 1), pool
sized to the blocks in use + 10 %, block placement a seeded random
permutation.  Synthetic data; no model weights are involved.

One step = the whole decode hot path over the batch:
  pa_reshape_and_cache  (each sequence's newest token -> its slot)
  pa_decode             (planning kernel + persistent split-KV decode kernel
                         with the fused log-sum-exp merge)
The slot mapping and the block tables come from the host before timing (the
host allocator is never inside the timed region).

Printed: one JSON line (rank 0).  `value` = algorithmic HBM bytes of the step
/ step time (GB/s), over all ranks; `seq_steps_per_s` beside it.  K/V bytes
per step (1.4 GB) are >10x the 129 MB L2, so no L2 flush between steps.

`--impl reference` times the CPU oracle (fp64, plain C, OpenMP) on the same
workload instead, on the host cores, rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention: achieved HBM GB/s (% of GB300 peak) and seq-steps/sec"
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + write) per pa_decode call on the LLaMA-13B-shaped
# workload, from an ncu capture of one launch (dram__bytes_read.sum +
# dram__bytes_write.sum); valid only for the decode kernel source whose
# sha256 prefix is given (otherwise reported as null).
TRAFFIC = {"bytes_per_launch": 1488554240, "kernel_sha256_prefix": "60ec91adda895f35"}
# The group kernel (pa_decode_grouped) on the parallel-sampling workload: DRAM bytes of one launch.
GROUP_TRAFFIC = {"bytes_per_launch": 348372736, "kernel_sha256_prefix": "60ec91adda895f35"}


# DRAM bytes (read + write) per pa_prefill_chunk call on the four-prompt
# prefill workloads, from ncu captures of one launch each; valid only for the
# prefill kernel source whose sha256 prefix is given.
PREFILL_TRAFFIC = {"kernel_sha256_prefix": "4962eb099e81b390",
                   "bf16": {"bytes_per_launch": 341745664}, "f16": {"bytes_per_launch": 341157120}}


def kernel_sha(files=("pa_decode.cu", "pa_common.cuh")) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_cache_35_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured bf16 dense (burst)"
    except Exception:
        return 1900.0, "fallback bf16 dense"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def decode_bytes(ctx_lens, H, D, B, elt) -> int:
    """Algorithmic bytes of one pa_decode call: K and V of every context
    token, q and out rows, the table entries covering the contexts, and the
    context lengths."""
    kv = 2 * sum(int(c) for c in ctx_lens) * H * D * elt
    qo = 2 * len(ctx_lens) * H * D * elt
    tables = 4 * sum(-(-int(c) // B) for c in ctx_lens)
    return kv + qo + tables + 4 * len(ctx_lens)


def grouped_decode_bytes(ctx_lens, starts, prefixes, H, D, B, elt) -> int:
    """Algorithmic bytes of one pa_decode_grouped call: each group's shared
    prefix K and V once per group, every sequence's own K and V, q and out
    rows, the table entries read (the prefix's once per group), the context
    lengths and the group arrays."""
    ctx = [int(c) for c in ctx_lens]
    pre = [0] * len(ctx)
    for g, p in enumerate(prefixes):
        for s in range(int(starts[g]), int(starts[g + 1])):
            pre[s] = int(p)
    kv = 2 * (sum(int(p) for p in prefixes) + sum(c - q for c, q in zip(ctx, pre))) * H * D * elt
    qo = 2 * len(ctx) * H * D * elt
    tables = 4 * (sum(-(-int(p) // B) for p in prefixes) + sum(-(-c // B) - q // B for c, q in zip(ctx, pre)))
    return kv + qo + tables + 4 * len(ctx) + 4 * (2 * len(prefixes) + 1)


def scatter_bytes(T, H, D, elt) -> int:
    """pa_reshape_and_cache: read k_new, v_new, write their slots, read slots."""
    return 4 * T * H * D * elt + 8 * T


def kv_bytes_per_token(layers, heads, head_dim, elt) -> int:
    """K and V bytes one token occupies in a model of `layers` layers."""
    return 2 * layers * heads * head_dim * elt


# ---- clocks ---------------------------------------------------------------------------------
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class NvmlPoller:
    """Reads the SM clock and the clock-event reasons of one GPU through NVML
    (ctypes on the driver's libnvidia-ml, read-only calls) every `period_s`
    in a thread, so that a timed region shorter than nvidia-smi's sampling
    period still gets samples of its own."""

    SW_POWER_CAP, HW_SLOWDOWN, SW_THERMAL, HW_THERMAL, HW_POWER_BRAKE = 0x4, 0x8, 0x20, 0x40, 0x80

    def __init__(self, pci_bus_id, index: int, period_s: float = 0.002):
        import ctypes

        self.samples = []
        self.period = period_s
        self.ok = False
        self._stop = threading.Event()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            rc = -1
            if pci_bus_id:
                rc = nv.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(h))
            if rc != 0:
                rc = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h))
            if rc != 0:
                return
            self.reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 else None
            self.nv, self.h, self.ctypes = nv, h, ctypes
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def start(self):
        if self.ok:
            threading.Thread(target=self._run, daemon=True).start()

    def _run(self):
        ct = self.ctypes
        clk, rsn = ct.c_uint(), ct.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk)) == 0 and \
                    self.reasons_fn(self.h, ct.byref(rsn)) == 0:
                self.samples.append((time.time(), float(clk.value), int(rsn.value)))
            time.sleep(self.period)

    def stop(self):
        self._stop.set()

    def summary(self, t0, t1):
        inside = [(c, r) for t, c, r in self.samples if t0 <= t <= t1]
        window = "timed region (NVML poll every 2 ms)"
        if not inside:  # a region shorter than the poll period: the samples just before and after it
            before = [(c, r) for t, c, r in self.samples if t < t0][-1:]
            after = [(c, r) for t, c, r in self.samples if t > t1][:1]
            inside = before + after
            window = "the NVML samples just before and after the timed region (shorter than the 2 ms poll)"
        if not inside:
            return None
        names = {self.SW_POWER_CAP: "sw_power_cap", self.HW_SLOWDOWN: "hw_slowdown",
                 self.SW_THERMAL: "sw_thermal_slowdown", self.HW_THERMAL: "hw_thermal_slowdown",
                 self.HW_POWER_BRAKE: "hw_power_brake_slowdown"}
        reasons = sorted({n for c, r in inside for bit, n in names.items() if r & bit})
        mhz = [c for c, _ in inside]
        return {"sm_mhz": statistics.median(mhz), "sm_mhz_min": min(mhz), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(inside), "window": window}


def _pci_bus_id(gpu_index: int):
    try:
        import torch

        p = torch.cuda.get_device_properties(gpu_index)
        return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi's clock line every 100 ms (the recipe's fields) and an NVML
    poll every 2 ms, over the same GPU (found by its PCI bus id)."""

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.bus = _pci_bus_id(gpu_index)
        self.nvml = NvmlPoller(self.bus, gpu_index)

    def start(self):
        self.nvml.start()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.bus or self.gpu}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()
        # nvidia-smi takes a moment to print its first line: wait for it (and
        # for the first NVML sample) before the caller's warm-up, so that even
        # a timed region of a fraction of a millisecond has samples around it
        t_end = time.time() + 2.0
        while time.time() < t_end and (not self.samples or (self.nvml.ok and not self.nvml.samples)):
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        self.nvml.stop()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        fast = self.nvml.summary(t0, t1)
        if not self.samples:
            res = {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        else:
            inside = [s for t, s in self.samples if t0 <= t <= t1]
            window = "timed region"
            if not inside:
                inside = [s for _, s in self.samples]
                window = "whole run (timed region shorter than the sampling period)"
            sm = [float(s[1]) for s in inside if s[1].replace(".", "").isdigit()]
            mx = [float(s[2]) for s in inside if s[2].replace(".", "").isdigit()]
            reasons = set()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for s in inside:
                for n, v in zip(names, s[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
            pw = [float(s[3]) for s in inside if s[3].replace(".", "").isdigit()]
            res = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                   "reasons": sorted(reasons), "power_w_max": max(pw) if pw else None, "samples": len(inside),
                   "window": window}
        if fast is not None:
            # the 2 ms poll covers the timed region itself: it sets the headline clock figures
            res["nvidia_smi"] = {k: res[k] for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "window")
                                 if k in res}
            res.update({"sm_mhz": fast["sm_mhz"], "sm_mhz_min": fast["sm_mhz_min"],
                        "sm_max_mhz": fast["sm_max_mhz"] or res.get("sm_max_mhz"),
                        "reasons": sorted(set(fast["reasons"]) | set(res.get("reasons", [])) - {"nvidia-smi unavailable"}),
                        "samples": fast["samples"], "window": fast["window"]})
        return res


# ---- distributed plumbing ------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    return rank, world, local


def dist_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ---- workloads ----------------------------------------------------------------------------------------
WORKLOAD_TEXT = {
    "llama13b": "llama13b_decode_b64: 64 seqs x 40 heads x 128, block 16, ctx U[128,2048], fp16",
    "long_context": "long_context_decode_b256: 256 seqs x 32 heads x 128, block 16, ctx log-normal "
                    "(median 1024, sigma 1, clipped 16..16384), bf16",
    "tiny": "tiny_paged_decode: 4 seqs x 4 heads x 64, block 16, ctx {1,16,17,45}, 32-block pool, fp16",
    "shared_prefix": "parallel_sampling_shared_prefix: 8 prompts x 8 samples, prompt 1000, suffix U[1,256], "
                     "40 heads x 128, block 16, fp16, copy-on-write through the host allocator",
    "mixed": "mixed_chunked_prefill: 32 decode seqs (ctx U[256,4096]) + 2 chunks x 512 queries at ctx 1024/3072, "
             "40 heads x 128, page 256, bf16",
    "budget512": "budget512_step: 512-token budget = 32 decode seqs (ctx U[256,4096]) + one 480-query chunk at "
                 "ctx 1440, 40 heads x 128, page 256, bf16",
}
MIXED = ("mixed", "budget512")
WORKLOAD_TEXT["memsim"] = ("host-only memory simulator: seeded long-tailed and short request traces, KV capacity "
                           "32768 tokens, reservation baselines (first fit) vs paged blocks of 16")
WORKLOAD_TEXT["batch_sweep"] = ("decode latency vs batch size 1..256, contexts of 1024, 40 heads x 128, fp16: "
                                "16-token pages at random places vs one contiguous 1024-token block per sequence")
WORKLOAD_TEXT["prefill"] = ("prefill of 4 prompts x 2048 tokens at context 0, 40 heads x 128, page 256, bf16: "
                            "the prompts' K/V scattered into the pool, then causal paged attention on the tensor "
                            "cores (one pa_prefill_chunk call)")
WORKLOAD_TEXT["prefill_f16"] = ("prefill of 4 prompts x 2048 tokens at context 0, 40 heads x 128, page 256, fp16: "
                                "the prompts' K/V scattered into the pool, then causal paged attention on the "
                                "tensor cores (one pa_prefill_chunk call)")
PREFILL_METRIC = "chunked prefill: causal paged attention TFLOP/s (4 * head_dim * heads per admissible key)"
WORKLOAD_TEXT["prefix_cache"] = ("prefix caching: 16 requests = a shared 1024-token system prompt + 256 tokens of "
                                 "their own, 40 heads x 128, block 16, bf16; suffix prefill over cached blocks vs "
                                 "whole-prompt prefill")
WORKLOAD_TEXT["swap"] = ("block swap: K/V of 8 requests x 2048 tokens, 40 heads x 128, fp16, block sizes 16..256, "
                         "GPU pool (blocks scattered) <-> pinned host pool")


def workload_config(name, w):
    return {"workload": WORKLOAD_TEXT[name], "num_seqs": w.num_seqs, "num_heads": w.num_heads,
            "head_dim": w.head_dim, "block_size": w.block_size, "pool_blocks": w.num_blocks, "kv_dtype": w.dtype,
            "placement": "seeded random permutation of the pool" if name != "shared_prefix" else
            "host allocator (free list from the end, copy-on-write)",
            "step": ("pa_reshape_and_cache (decode tokens + chunk tokens) + pa_mixed_step (chunked prefill on a "
                     "capped grid with the decode launched behind it as a programmatic dependent, concurrently)"
                     if name in MIXED else
                     "pa_reshape_and_cache (1 new token/seq) + pa_decode over ctx"),
            "l2": "no flush: K/V read per step >> 129 MB L2" if name in ("llama13b", "long_context") + MIXED else
                  "working set partly L2-resident (reported as such)"}


def shared_prefix_decode_workload(pa, W, dev):
    """The parallel-sampling state built through the library: prompts written,
    forked 8 ways, first suffix token of each sample copy-on-writes the
    shared partial block, suffixes written.  Returned as a decode workload
    whose step rewrites each sample's newest token and attends over it."""
    import numpy as np
    import torch

    sc = W.shared_prefix(device=dev)
    P, N, L, B, H, D = sc.num_prompts, sc.samples, sc.prompt_len, sc.block_size, sc.num_heads, sc.head_dim
    n = P * N
    alloc = pa.BlockAllocator(sc.num_blocks, B)
    for p in range(P):
        alloc.add_seq(p * N)
    pslots = np.stack([alloc.append_slots([p * N for p in range(P)])[0] for _ in range(L)], axis=1)
    for p in range(P):
        for j in range(1, N):
            alloc.fork(p * N, p * N + j)
    kp, vp = sc.pool_init_k, sc.pool_init_v
    err = pa.new_error_flag(dev)
    pa.pa_reshape_and_cache(sc.prompt_k.reshape(P * L, H, D), sc.prompt_v.reshape(P * L, H, D), kp, vp,
                            torch.from_numpy(pslots.reshape(-1)).to(dev), err)
    suffix = sc.suffix_lens.tolist()
    ms = sc.suffix_k.shape[1]
    sslots = np.full((n, ms), -1, dtype=np.int64)
    for r in range(max(suffix)):
        active = [s for s in range(n) if suffix[s] > r]
        slots, pairs = alloc.append_slots(active)
        sslots[active, r] = slots
        if len(pairs):
            pa.pa_copy_blocks(kp, vp, torch.from_numpy(pairs).to(dev), err)
    pa.pa_reshape_and_cache(sc.suffix_k.reshape(n * ms, H, D), sc.suffix_v.reshape(n * ms, H, D), kp, vp,
                            torch.from_numpy(sslots.reshape(-1)).to(dev), err)
    if pa.pa_get_error(err):
        raise RuntimeError("device error while building the shared-prefix state")
    mb = max(len(alloc.block_table(s)[0]) for s in range(n))
    tables, lens = alloc.block_tables(range(n), mb)
    lens_t = torch.from_numpy(lens)
    unique_blocks = sc.num_blocks - alloc.num_free()
    group_start, group_prefix = alloc.prefix_groups(range(n))
    w = W.DecodeWorkload(
        name="shared_prefix", num_heads=H, head_dim=D, block_size=B, num_blocks=sc.num_blocks, dtype="f16",
        context_lens=lens_t, new_pos=(lens_t - 1).to(torch.int32), block_tables=torch.from_numpy(tables),
        max_blocks_per_seq=mb, q=sc.q, k_new=W.normal((n, H, D), 31, torch.float16, dev),
        v_new=W.normal((n, H, D), 32, torch.float16, dev), k_pool=kp, v_pool=vp, scale=sc.scale,
        extra={"unique_kv_bytes": 2 * unique_blocks * H * B * D * 2,
               "group_start": torch.from_numpy(group_start), "group_prefix": torch.from_numpy(group_prefix)})
    alloc.close()
    return w


class OracleStep:
    """The CPU oracle's version of one step (slot scatter + decode) on a
    workload, with the inputs converted to bit arrays once, outside any
    timing.  `rows` restricts the step to a subset of the sequences."""

    def __init__(self, w, host, rows=None):
        import numpy as np

        import oracle

        self.oracle = oracle
        self.w = w
        rows = list(range(w.num_seqs)) if rows is None else list(rows)
        self.kb, self.vb = oracle.pool_bits(host["k_pool"]), oracle.pool_bits(host["v_pool"])
        tb = w.block_tables.numpy()
        self.tables = np.ascontiguousarray(tb[rows])
        self.ctx = np.ascontiguousarray(w.context_lens.numpy()[rows])
        self.slots = np.array([oracle.slot_of(tb[s], int(w.new_pos[s]), w.block_size) for s in rows], dtype=np.int64)
        self.q = host["q"][rows].contiguous()
        self.k_new = host["k_new"][rows].contiguous()
        self.v_new = host["v_new"][rows].contiguous()
        self.rows = rows

    def run(self):
        o, w = self.oracle, self.w
        o.reshape_and_cache(self.k_new, self.v_new, self.kb, self.vb, self.slots, w.block_size)
        return o.decode(self.q, self.kb, self.vb, self.tables, self.ctx, w.block_size, w.scale, w.dtype)

    def time(self, budget_s: float, max_reps: int = 1000):
        """Repeat run() until ~budget_s; returns (seconds per run, runs)."""
        reps, t0 = 0, time.perf_counter()
        while True:
            self.run()
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s or reps >= max_reps:
                return el / reps, reps


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: rank 0 only."""
    if rank != 0:
        return
    import torch

    import oracle
    import pa_workloads as W

    oracle.build()
    w = W.llama13b_decode(device="cpu")
    host = {k: getattr(w, k) for k in ("k_pool", "v_pool", "q", "k_new", "v_new")}
    elt = 2
    step_b = decode_bytes(w.context_lens.tolist(), w.num_heads, w.head_dim, w.block_size, elt) + scatter_bytes(
        w.num_seqs, w.num_heads, w.head_dim, elt)
    # warm-up steps (untimed), then K timed steps; each step is the whole
    # workload unless that would exceed ~60 s in total, in which case each
    # step runs on a fixed subset of the sequences.
    full = OracleStep(w, host)
    thr = oracle.num_threads()
    t_one, _ = full.time(0.0, 1)
    frac = min(1.0, 60.0 / max(1e-9, t_one * args.steps))
    nsub = max(1, int(w.num_seqs * frac))
    step = full if nsub == w.num_seqs else OracleStep(w, host, rows=range(nsub))
    for _ in range(max(0, args.warmup - 1)):
        step.run()
    sub_b = decode_bytes(step.ctx.tolist(), w.num_heads, w.head_dim, w.block_size, elt) + scatter_bytes(
        nsub, w.num_heads, w.head_dim, elt)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step.run()
    el = time.perf_counter() - t0
    gbs = sub_b * args.steps / el / 1e9
    sample = (f"{nsub} of {w.num_seqs} sequences x {w.num_heads} heads per step" if nsub < w.num_seqs
              else "whole workload per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config("llama13b", w),
        "parallelism": "none: the CPU oracle on the host cores of rank 0",
        "seq_steps_per_s": nsub * args.steps / el,
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": thr, "kind": "oracle", "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "step_bytes_full_workload": step_b,
    }
    print(json.dumps(line), flush=True)


SPIN_CYCLES = 400_000  # ~0.2 ms at 2 GHz
TIMING_NOTE = ("CUDA events around exactly K steps after a barrier and a synchronize; a ~0.2 ms GPU spin is "
               "queued before the start event so that the host's enqueueing of the first step is not inside "
               "the device-timed region; the clock samplers run from before the warm-up (no idle gap)")


def spin_before_region():
    """Keep the GPU busy while the host enqueues the start event and the
    first steps: without it a short region (the driver's 20 steps) also
    times the first launch's host latency, ~0.5 % per 20 steps."""
    import torch

    spin = getattr(torch.cuda, "_sleep", None)
    if spin is not None:
        spin(SPIN_CYCLES)


def time_calls(fn, stream, dev, n_back: int, n_each: int) -> dict:
    """Device time of one call of `fn` on `stream`: `n_back` calls back to
    back between two events (the mean, which the rooflines use), then
    `n_each` calls each between events of its own (median, min and max; an
    event recorded between two kernels stops the next one's programmatic
    early start, so these run slightly longer than the back-to-back mean)."""
    import torch

    ev = lambda: torch.cuda.Event(enable_timing=True)
    a, b = ev(), ev()
    torch.cuda.synchronize(dev)
    a.record(stream)
    for _ in range(n_back):
        fn()
    b.record(stream)
    torch.cuda.synchronize(dev)
    mean_ms = a.elapsed_time(b) / n_back
    s, e = [ev() for _ in range(n_each)], [ev() for _ in range(n_each)]
    for i in range(n_each):
        s[i].record(stream)
        fn()
        e[i].record(stream)
    torch.cuda.synchronize(dev)
    per = sorted(x.elapsed_time(y) for x, y in zip(s, e))
    return {"mean_ms_back_to_back": mean_ms, "calls_back_to_back": n_back, "median_ms": statistics.median(per),
            "min_ms": per[0], "max_ms": per[-1], "calls_timed_each": n_each}


def call_stats(per_ms) -> dict:
    per = sorted(per_ms)
    return {"mean_ms": statistics.mean(per), "median_ms": statistics.median(per), "min_ms": per[0],
            "max_ms": per[-1], "calls_timed_each": len(per)}


def cpu_baseline_decode(w, budget_s: float, elt: int = 2) -> dict:
    """The oracle (scatter + decode) timed on the host cores with its OpenMP
    loops on every core, and single-threaded on the first sequences (a
    bounded sample of the same workload); the same GB/s unit as the line."""
    import oracle

    H, D, B = w.num_heads, w.head_dim, w.block_size
    host = {k: getattr(w, k).cpu() for k in ("k_pool", "v_pool", "q", "k_new", "v_new")}
    thr = oracle.num_threads()
    full = OracleStep(w, host)
    t_rep, reps = full.time(budget_s)
    res = {"value": (decode_bytes(w.context_lens.tolist(), H, D, B, elt) + scatter_bytes(w.num_seqs, H, D, elt))
           / t_rep / 1e9, "unit": "GB/s", "cores": thr, "kind": "oracle",
           "sample": f"the whole step's scatter + decode on {thr} threads (OpenMP over (sequence, head)), "
                     f"{reps} repetitions, {t_rep * reps:.1f} s wall"}
    nsub = max(1, min(w.num_seqs, 8))
    sub = OracleStep(w, host, rows=range(nsub))
    oracle.set_num_threads(1)
    try:
        t1, r1 = sub.time(budget_s / 2)
    finally:
        oracle.set_num_threads(thr)
    sub_b = decode_bytes(sub.ctx.tolist(), H, D, B, elt) + scatter_bytes(nsub, H, D, elt)
    res["single_thread"] = {"value": sub_b / t1 / 1e9, "unit": "GB/s", "cores": 1,
                            "sample": f"scatter + decode of the first {nsub} of {w.num_seqs} sequences, one "
                                      f"thread, {r1} repetitions, {t1 * r1:.1f} s wall"}
    return res


def measure_decode(args, rank, world, local, name, secondary=False):
    """One decode-path workload: warm-up, K timed steps, then the kernel
    timings for the roofline.  `secondary` (the other configurations of the
    default run) skips the end-to-end pass, the CPU baseline and the graph
    comparison.  Returns the JSON line as a dict."""
    import numpy as np
    import torch

    import paged_kv_cache_35_gb300 as pa
    import pa_workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mixed = None
    if name == "llama13b":
        w = W.llama13b_decode(device=dev)
    elif name == "long_context":
        w = W.long_context_decode(device=dev, num_seqs=args.num_seqs or 256)
    elif name == "tiny":
        w = W.tiny_decode(device=dev)
    elif name == "shared_prefix":
        w = shared_prefix_decode_workload(pa, W, dev)
    else:
        mixed = W.mixed_prefill(device=dev) if name == "mixed" else W.budget512_step(device=dev)
        w = mixed.decode
    S, H, D, B = w.num_seqs, w.num_heads, w.head_dim, w.block_size
    elt = 2
    tdt = torch.float16 if w.dtype == "f16" else torch.bfloat16
    slots = pa.pa_slot_mapping(w.block_tables, np.arange(S), w.new_pos, B)
    k_new, v_new = w.k_new, w.v_new
    if mixed is not None:  # one scatter: the decode tokens and the chunks' tokens
        seq_idx = np.concatenate([np.full(int(n), c) for c, n in enumerate(mixed.chunk_lens.tolist())])
        pos = np.concatenate([np.arange(c0, c0 + n) for c0, n in
                              zip(mixed.ctx_before.tolist(), mixed.chunk_lens.tolist())])
        slots = np.concatenate([slots, pa.pa_slot_mapping(mixed.chunk_tables, seq_idx, pos, B)])
        k_new = torch.cat([w.k_new, mixed.chunk_k])
        v_new = torch.cat([w.v_new, mixed.chunk_v])
        T = int(mixed.chunk_lens.sum())
        pout = torch.empty(T, H, D, dtype=tdt, device=dev)
        cu_d = torch.cat([torch.zeros(1, dtype=torch.int32), mixed.chunk_lens.cumsum(0).to(torch.int32)]).to(dev)
        cb_d, ctab_d = mixed.ctx_before.to(dev), mixed.chunk_tables.to(dev)
        mq = int(mixed.chunk_lens.max())
    slots_d = torch.from_numpy(slots).to(dev)
    tables_d = w.block_tables.to(dev)
    ctx_d = w.context_lens.to(dev)
    mx = int(w.context_lens.max())
    out = torch.empty(S, H, D, dtype=tdt, device=dev)
    ws = pa.decode_workspace(S, H, D, mx, device=dev)
    err = pa.new_error_flag(dev)
    stream = torch.cuda.current_stream(dev)
    # parallel sampling: the step decodes with each shared prompt read once per group
    grouped = "group_start" in w.extra
    if grouped:
        gs_d, gp_d = w.extra["group_start"].to(dev), w.extra["group_prefix"].to(dev)
        ws_g = pa.decode_grouped_workspace(S, H, D, mx, device=dev)

    def decode_plain(q_in=None):
        pa.pa_decode(out, w.q if q_in is None else q_in, w.k_pool, w.v_pool, tables_d, ctx_d, mx, w.scale, ws, err,
                     stream=stream)

    def prefill():
        pa.pa_prefill_chunk(pout, mixed.chunk_q, cu_d, cb_d, w.k_pool, w.v_pool, ctab_d, mq, w.scale, err, stream)

    def decode(q_in=None):
        if grouped:
            pa.pa_decode_grouped(out, w.q if q_in is None else q_in, w.k_pool, w.v_pool, tables_d, ctx_d, mx,
                                 w.scale, gs_d, gp_d, ws_g, err, stream=stream)
        else:
            decode_plain(q_in)

    def mixed_step(q_in=None, tables_in=None, ctx_in=None, cq_in=None, cu_in=None, cb_in=None, ctab_in=None):
        pick = lambda given, resident: resident if given is None else given
        pa.pa_mixed_step(out, pick(q_in, w.q), pick(tables_in, tables_d), pick(ctx_in, ctx_d), mx, ws, pout,
                         pick(cq_in, mixed.chunk_q), pick(cu_in, cu_d), pick(cb_in, cb_d), pick(ctab_in, ctab_d), mq,
                         w.k_pool, w.v_pool, w.scale, err, stream=stream)

    def step():
        pa.pa_reshape_and_cache(k_new, v_new, w.k_pool, w.v_pool, slots_d, err, stream)
        if mixed is not None:
            mixed_step()
        else:
            decode()

    clocks = ClockSampler(local)
    clocks.start()  # before the warm-up: the GPU stays busy up to the timed region
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    flags = pa.pa_get_error(err, stream)
    if flags:
        clocks.stop()
        raise RuntimeError(f"device error flags {flags} during warm-up")

    logical_bytes = decode_bytes(w.context_lens.tolist(), H, D, B, elt)
    dbytes = (grouped_decode_bytes(w.context_lens.tolist(), w.extra["group_start"].tolist(),
                                   w.extra["group_prefix"].tolist(), H, D, B, elt) if grouped else logical_bytes)
    sbytes = scatter_bytes(k_new.shape[0], H, D, elt)
    pflops = pbytes = 0
    if mixed is not None:
        pflops = sum(4 * D * H * sum(c0 + i + 1 for i in range(n))
                     for c0, n in zip(mixed.ctx_before.tolist(), mixed.chunk_lens.tolist()))
        pbytes = sum(2 * (c0 + n) * H * D * elt + 2 * n * H * D * elt
                     for c0, n in zip(mixed.ctx_before.tolist(), mixed.chunk_lens.tolist()))
    step_b = dbytes + sbytes + pbytes

    K = args.steps
    ev = lambda: torch.cuda.Event(enable_timing=True)

    # ---- device-timed region: K steps back to back, nothing between them.
    t_start, t_end = ev(), ev()
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    h0 = time.time()
    spin_before_region()
    t_start.record(stream)
    for _ in range(K):
        step()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    h1 = time.time()
    dist_barrier(world)
    clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    flags = pa.pa_get_error(err, stream)
    if flags:
        raise RuntimeError(f"device error flags {flags} in the timed region")
    max_ms = dist_max(total_ms, world)
    ms_per_step = max_ms / K
    total_s = max_ms / 1e3
    value = step_b * K * world / total_s / 1e9
    seq_steps = S * K * world / total_s

    # ---- kernel timings for the roofline, after the timed region.
    seq_ms = pre_t = None
    if mixed is None:
        # pa_decode alone (planning + decode kernels), back to back: the K/V
        # it reads per call (>= 1.4 GB on the full-size batches) is far larger than L2.
        dec_t = time_calls(decode, stream, dev, max(K, 100), 50)
        dec_ms = dec_t["mean_ms_back_to_back"]
        if grouped:  # the same state decoded sequence by sequence, for comparison
            plain_t = time_calls(decode_plain, stream, dev, max(K, 100), 50)
            decode()  # `out` holds the grouped result again (the end-to-end check compares bits)
    else:
        # Component pass: scatter, decode, prefill one after the other with
        # events around the two attention calls -- inside the concurrent step
        # the decode's events would also span the prefill; the decode between
        # two prefills also flushes the prefill's 105 MB of K/V from L2.
        Kc = max(K, 50)
        dec_s, dec_e = [ev() for _ in range(Kc)], [ev() for _ in range(Kc)]
        pre_s, pre_e = [ev() for _ in range(Kc)], [ev() for _ in range(Kc)]
        c0_, c1_ = ev(), ev()
        torch.cuda.synchronize(dev)
        c0_.record(stream)
        for i in range(Kc):
            pa.pa_reshape_and_cache(k_new, v_new, w.k_pool, w.v_pool, slots_d, err, stream)
            dec_s[i].record(stream)
            decode()
            dec_e[i].record(stream)
            pre_s[i].record(stream)
            prefill()
            pre_e[i].record(stream)
        c1_.record(stream)
        torch.cuda.synchronize(dev)
        dec_t = call_stats([a.elapsed_time(b) for a, b in zip(dec_s, dec_e)])
        pre_t = call_stats([a.elapsed_time(b) for a, b in zip(pre_s, pre_e)])
        seq_ms = c0_.elapsed_time(c1_) / Kc
        dec_ms = dec_t["mean_ms"]
    if pa.pa_get_error(err, stream):
        raise RuntimeError("device error flags in the kernel-timing pass")

    peak, peak_kind = load_peaks()
    dec_note = None
    if dec_ms > ms_per_step:
        # the decode call cannot take longer than the step that contains it
        dec_note = (f"decode call timed at {dec_ms:.4f} ms, longer than the step ({ms_per_step:.4f} ms): the "
                    "roofline uses the step time")
        dec_ms = ms_per_step
    achieved = dbytes / (dec_ms / 1e3) / 1e9
    sha = kernel_sha()
    traffic = (TRAFFIC["bytes_per_launch"] if name == "llama13b" and TRAFFIC["kernel_sha256_prefix"] == sha
               else GROUP_TRAFFIC["bytes_per_launch"] if grouped and GROUP_TRAFFIC["kernel_sha256_prefix"] == sha
               else None)
    launches = 3 + (1 if mixed is not None else 0)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(name, w),
        "parallelism": f"replicas x{world}",
        "timing": TIMING_NOTE,
        "seq_steps_per_s": seq_steps,
        "hbm_frac_of_measured_peak": value / world / peak,
        "hbm_frac_of_nominal_8tbs": value / world / 8000.0,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_kind": f"{peak_kind} copy bandwidth",
                     "kernel": "pa_decode call (planning kernel + persistent decode kernel)",
                     "algorithmic_bytes_per_launch": dbytes, "avg_launch_ms": dec_ms,
                     "calls": dec_t, "kernel_sha256_prefix": sha},
        "gpu_launches": launches * K,
        "clocks": clocks.summary(h0, h1),
    }
    if dec_note:
        line["roofline"]["note"] = dec_note
    if "unique_kv_bytes" in w.extra:
        line["config"]["unique_kv_bytes"] = w.extra["unique_kv_bytes"]
    if grouped:
        line["roofline"]["kernel"] = "pa_decode_grouped call (planning kernel + persistent group kernel)"
        line["roofline"]["note"] = ("bytes as the grouped call reads them: each shared prompt once per group, "
                                    "every sample's own tokens once")
        line["config"]["step"] = ("pa_reshape_and_cache (1 new token/seq) + pa_decode_grouped over ctx (8 groups "
                                  "of 8 samples, prompt blocks shared)")
        line["config"]["groups"] = {"group_start": w.extra["group_start"].tolist(),
                                    "group_prefix": w.extra["group_prefix"].tolist()}
        line["logical"] = {"bytes_per_step": logical_bytes + sbytes,
                           "GBs": (logical_bytes + sbytes) * K * world / total_s / 1e9,
                           "note": "shared prompt blocks counted once per sample that attends over them"}
        line["ungrouped_decode"] = {"kernel": "pa_decode call on the same state", "calls": plain_t,
                                    "avg_launch_ms": plain_t["mean_ms_back_to_back"],
                                    "grouped_speedup": plain_t["mean_ms_back_to_back"] / dec_ms}
    if mixed is not None:
        line["roofline"]["note"] = ("decode kernel timed alone in a component pass after the timed region (inside "
                                    "the concurrent step its events would also span the prefill)")
        line["sequential_ms_per_step"] = seq_ms
        line["concurrent_speedup_vs_sequential"] = seq_ms / ms_per_step
        bf16_peak = load_tensor_peak()
        pre_avg_s = pre_t["mean_ms"] / 1e3
        line["prefill"] = {"bound": "tensor", "achieved": pflops / pre_avg_s / 1e12, "unit": "TFLOP/s",
                           "peak": bf16_peak[0], "frac": pflops / pre_avg_s / 1e12 / bf16_peak[0],
                           "peak_kind": bf16_peak[1], "algorithmic_flops_per_launch": pflops,
                           "avg_launch_ms": pre_t["mean_ms"], "calls": pre_t,
                           "kernel_sha256_prefix": kernel_sha(("pa_prefill.cu", "pa_common.cuh"))}
    if secondary:
        return line

    # ---- end to end through the API: pinned host inputs in, result out, every step.
    # The copies run on their own streams with two sets of device buffers, so
    # step i's inputs arrive while step i-1 computes and step i-1's result
    # returns while step i computes; the timed region spans the first input
    # copy to the last result copy.
    Ke = min(K, 200)
    pin = lambda t: t.detach().cpu().pin_memory()
    host_in = [pin(w.q), pin(k_new), pin(v_new), pin(torch.from_numpy(slots)), pin(w.block_tables),
               pin(w.context_lens)]
    if mixed is not None:
        host_in += [pin(mixed.chunk_q), pin(cu_d), pin(cb_d), pin(ctab_d)]
    outs_dev = [out] + ([pout] if mixed is not None else [])
    host_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs_dev]
    bufs_in = [[torch.empty(h.shape, dtype=h.dtype, device=dev) for h in host_in] for _ in range(2)]
    bufs_out = [[torch.empty_like(o) for o in outs_dev] for _ in range(2)]
    h2d = sum(h.numel() * h.element_size() for h in host_in)
    d2h = sum(h.numel() * h.element_size() for h in host_out)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    drained = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):  # recorded once so the first waits have something to wait for
        done[b].record(stream)
        drained[b].record(stream)

    def e2e_step(i):
        b = i % 2
        d_in, d_out = bufs_in[b], bufs_out[b]
        with torch.cuda.stream(s_in):
            s_in.wait_event(done[b])  # step i-2 has finished reading these buffers
            for d, h in zip(d_in, host_in):
                d.copy_(h, non_blocking=True)
            ready[b].record(s_in)
        stream.wait_event(ready[b])
        stream.wait_event(drained[b])  # step i-2's result has left these buffers
        d_q, d_k, d_v, d_slots, d_tables, d_ctx = d_in[:6]
        pa.pa_reshape_and_cache(d_k, d_v, w.k_pool, w.v_pool, d_slots, err, stream)
        if mixed is not None:
            d_cq, d_cu, d_cb, d_ctab = d_in[6:]
            pa.pa_mixed_step(d_out[0], d_q, d_tables, d_ctx, mx, ws, d_out[1], d_cq, d_cu, d_cb, d_ctab, mq,
                             w.k_pool, w.v_pool, w.scale, err, stream=stream)
        elif grouped:
            pa.pa_decode_grouped(d_out[0], d_q, w.k_pool, w.v_pool, d_tables, d_ctx, mx, w.scale, gs_d, gp_d, ws_g,
                                 err, stream=stream)
        else:
            pa.pa_decode(d_out[0], d_q, w.k_pool, w.v_pool, d_tables, d_ctx, mx, w.scale, ws, err, stream=stream)
        done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[b])
            for h, d in zip(host_out, d_out):
                h.copy_(d, non_blocking=True)
            drained[b].record(s_out)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    dist_barrier(world)
    e0, e1 = ev(), ev()
    spin_before_region()
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(Ke):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    e2e_ms = dist_max(e0.elapsed_time(e1), world)
    e2e_value = step_b * Ke * world / (e2e_ms / 1e3) / 1e9
    if not torch.equal(host_out[0].view(torch.int16), out.cpu().view(torch.int16)):
        raise RuntimeError("the end-to-end result differs from the device-timed step's")
    line["e2e"] = {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                   "ms_per_step": e2e_ms / Ke, "steps": Ke,
                   "overlap": "copies on their own streams, double-buffered, overlapping the previous step"}
    if name == "tiny":
        line["graph_replay"] = graph_replay_comparison(pa, w, dev, stream)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode(w, args.cpu_budget, elt)
    return line


# Configurations the default run also times after the headline (same
# --steps / --warmup), each nested under "other_configs" in the same line.
OTHER_CONFIGS = ("tiny", "shared_prefix", "long_context", "mixed", "budget512", "prefill", "swap")


def secondary_summary(line: dict) -> dict:
    keep = ("metric", "value", "unit", "ms_per_step", "steps", "warmup", "dtype", "config", "roofline", "clocks",
            "seq_steps_per_s", "prefill", "sequential_ms_per_step", "concurrent_speedup_vs_sequential",
            "gpu_launches", "copy_blocks_roofline", "sweep_by_block_size", "logical", "ungrouped_decode")
    return {k: line[k] for k in keep if k in line}


def run_ours(args, rank, world, local):
    import torch

    import __graft_entry__

    __graft_entry__.build()
    line = measure_decode(args, rank, world, local, args.workload)
    if args.workload == "llama13b" and not args.no_other_configs:
        others = {}
        for name in OTHER_CONFIGS:
            torch.cuda.empty_cache()
            if name == "prefill":
                sub = measure_prefill(args, rank, world, local, name, secondary=True)
            elif name == "swap":
                sub = measure_swap(args, rank, world, local)
            else:
                sub = measure_decode(args, rank, world, local, name, secondary=True)
            others[name] = secondary_summary(sub)
        line["other_configs"] = others
        line["gpu_launches_other_configs"] = sum(o["gpu_launches"] for o in others.values())
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_prefill(args, rank, world, local):
    import __graft_entry__

    __graft_entry__.build()
    line = measure_prefill(args, rank, world, local, args.workload)
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure_prefill(args, rank, world, local, name, secondary=False):
    """One prefill step = four 2048-token prompts' K/V scattered into their
    pages, then one pa_prefill_chunk over the four prompts (context 0).  value: algorithmic
    TFLOP/s of the step; roofline: the prefill kernel alone (calls back to
    back after the timed region; K/V and queries, 252 MB, exceed L2), against
    the measured dense tensor peak (fp16 and bf16 run at the same rate); e2e:
    pinned host inputs in and the output out every step, copies pipelined;
    cpu_baseline: the oracle on four 16-row sub-chunks spread over the first
    prompt (a sub-chunk starting at row a has context a, so its rows are
    exactly those rows of the prompt).  `secondary` skips the end-to-end pass
    and the CPU baseline.  Returns the JSON line as a dict."""
    import numpy as np
    import torch

    import paged_kv_cache_35_gb300 as pa
    import pa_workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dtype = "f16" if name == "prefill_f16" else "bf16"
    NP, L = 4, 2048  # prompts, tokens per prompt
    T = NP * L
    m = W.small_prefill(device=dev, chunk_lens=(L,) * NP, ctx_before=(0,) * NP, H=40, B=256, dtype=dtype)
    w = m.decode
    H, D, B = w.num_heads, w.head_dim, w.block_size
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    slots = pa.pa_slot_mapping(m.chunk_tables, np.repeat(np.arange(NP), L), np.tile(np.arange(L), NP), B)
    slots_d = torch.from_numpy(slots).to(dev)
    cu_d = torch.arange(0, T + 1, L, dtype=torch.int32, device=dev)
    cb_d = torch.zeros(NP, dtype=torch.int32, device=dev)
    tab_d = m.chunk_tables.to(dev)
    out = torch.empty(T, H, D, dtype=tdt, device=dev)
    err = pa.new_error_flag(dev)
    stream = torch.cuda.current_stream(dev)

    def prefill(o=None, q=None, cu=None, cb=None, tab=None):
        pick = lambda given, resident: resident if given is None else given
        pa.pa_prefill_chunk(pick(o, out), pick(q, m.chunk_q), pick(cu, cu_d), pick(cb, cb_d), w.k_pool, w.v_pool,
                            pick(tab, tab_d), L, w.scale, err, stream)

    def step():
        pa.pa_reshape_and_cache(m.chunk_k, m.chunk_v, w.k_pool, w.v_pool, slots_d, err, stream)
        prefill()

    clocks = ClockSampler(local)
    clocks.start()  # before the warm-up: the GPU stays busy up to the timed region
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    flags = pa.pa_get_error(err, stream)
    if flags:
        clocks.stop()
        raise RuntimeError(f"device error flags {flags} during warm-up")
    flops = NP * 4 * D * H * L * (L + 1) // 2

    K = args.steps
    ev = lambda: torch.cuda.Event(enable_timing=True)
    t_start, t_end = ev(), ev()
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    h0 = time.time()
    spin_before_region()
    t_start.record(stream)
    for _ in range(K):
        step()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    h1 = time.time()
    dist_barrier(world)
    clocks.stop()
    flags = pa.pa_get_error(err, stream)
    if flags:
        raise RuntimeError(f"device error flags {flags} in the timed region")
    max_ms = dist_max(t_start.elapsed_time(t_end), world)
    ms_per_step = max_ms / K
    value = flops * K * world / (max_ms / 1e3) / 1e12
    pre_t = time_calls(prefill, stream, dev, max(K, 100), 50)
    pre_ms = pre_t["mean_ms_back_to_back"]
    pre_note = None
    if pre_ms > ms_per_step:
        pre_note = (f"prefill call timed at {pre_ms:.4f} ms, longer than the step ({ms_per_step:.4f} ms): the "
                    "roofline uses the step time")
        pre_ms = ms_per_step
    if pa.pa_get_error(err, stream):
        raise RuntimeError("device error flags in the kernel-timing pass")
    peak, peak_kind = load_tensor_peak()
    pf_sha = kernel_sha(("pa_prefill.cu", "pa_common.cuh"))
    pf_traffic = (PREFILL_TRAFFIC[dtype]["bytes_per_launch"] if PREFILL_TRAFFIC["kernel_sha256_prefix"] == pf_sha
                  else None)
    achieved = flops / (pre_ms / 1e3) / 1e12
    line = {
        "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype, "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[name], "prompts": NP, "tokens_per_prompt": L, "context_before": 0,
                   "num_heads": H, "head_dim": D, "block_size": B, "kv_dtype": dtype,
                   "l2": "no flush: inputs larger than L2 (per step the scatter reads 168 MB of new K/V and "
                         "writes it to the pool, the prefill reads it and 84 MB of queries and writes 84 MB)"},
        "parallelism": f"replicas x{world}",
        "timing": TIMING_NOTE,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": pf_traffic, "peak_kind": peak_kind,
                     "kernel": "prefill_kernel (pa_prefill_chunk)", "algorithmic_flops_per_launch": flops,
                     "avg_launch_ms": pre_ms, "calls": pre_t,
                     "kernel_sha256_prefix": pf_sha,
                     "traffic_source": "ncu DRAM bytes (read + write) of one launch of this workload"},
        "gpu_launches": 2 * K,
        "clocks": clocks.summary(h0, h1),
    }
    if pre_note:
        line["roofline"]["note"] = pre_note
    if secondary:
        return line

    # ---- end to end: pinned host inputs (q, the prompt's K/V, slots, table,
    # offsets) in and the output out every step, double-buffered on their own streams
    Ke = min(K, 200)
    pin = lambda t: t.detach().cpu().pin_memory()
    host_in = [pin(m.chunk_q), pin(m.chunk_k), pin(m.chunk_v), pin(torch.from_numpy(slots)), pin(m.chunk_tables),
               pin(cu_d), pin(cb_d)]
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    bufs_in = [[torch.empty(h.shape, dtype=h.dtype, device=dev) for h in host_in] for _ in range(2)]
    bufs_out = [torch.empty_like(out) for _ in range(2)]
    h2d = sum(h.numel() * h.element_size() for h in host_in)
    d2h = host_out.numel() * host_out.element_size()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    drained = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):
        done[b].record(stream)
        drained[b].record(stream)

    def e2e_step(i):
        b = i % 2
        d_in, d_out = bufs_in[b], bufs_out[b]
        with torch.cuda.stream(s_in):
            s_in.wait_event(done[b])
            for d, h in zip(d_in, host_in):
                d.copy_(h, non_blocking=True)
            ready[b].record(s_in)
        stream.wait_event(ready[b])
        stream.wait_event(drained[b])
        d_q, d_k, d_v, d_slots, d_tab, d_cu, d_cb = d_in
        pa.pa_reshape_and_cache(d_k, d_v, w.k_pool, w.v_pool, d_slots, err, stream)
        prefill(d_out, d_q, d_cu, d_cb, d_tab)
        done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[b])
            host_out.copy_(d_out, non_blocking=True)
            drained[b].record(s_out)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    dist_barrier(world)
    e0, e1 = ev(), ev()
    spin_before_region()
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(Ke):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    e2e_ms = dist_max(e0.elapsed_time(e1), world)
    if not torch.equal(host_out.view(torch.int16), out.cpu().view(torch.int16)):
        raise RuntimeError("the end-to-end result differs from the device-timed step's")
    if pa.pa_get_error(err, stream):
        raise RuntimeError("device error flags in the end-to-end pass")

    line["e2e"] = {"value": flops * Ke * world / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / Ke, "steps": Ke,
                   "overlap": "copies on their own streams, double-buffered, overlapping the previous step"}
    if rank == 0 and not args.no_cpu_baseline:
        import oracle

        kb, vb = oracle.pool_bits(w.k_pool.cpu()), oracle.pool_bits(w.v_pool.cpu())
        oracle.reshape_and_cache(m.chunk_k.cpu(), m.chunk_v.cpu(), kb, vb, slots, B)
        starts, n = (0, 672, 1344, 2032), 16
        q_host = m.chunk_q.cpu()
        q_s = torch.cat([q_host[a:a + n] for a in starts])
        cu_s = torch.arange(0, n * len(starts) + 1, n, dtype=torch.int32)
        cb_s = torch.tensor(starts, dtype=torch.int32)
        tab_s = m.chunk_tables.cpu()[:1].expand(len(starts), -1).contiguous()
        s_flops = sum(4 * D * H * (a + i + 1) for a in starts for i in range(n))
        reps, t0 = 0, time.perf_counter()
        while True:
            oracle.prefill(q_s, cu_s, cb_s, kb, vb, tab_s, B, w.scale, dtype)
            reps += 1
            el = time.perf_counter() - t0
            if el >= args.cpu_budget or reps >= 1000:
                break
        line["cpu_baseline"] = {"value": s_flops * reps / el / 1e12, "unit": "TFLOP/s",
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": f"{len(starts)} x {n} query rows (contexts 1..{starts[-1] + n}), "
                                          f"{reps} repetitions, {el:.1f} s wall"}
    return line


def graph_replay_comparison(pa, w, dev, stream, n=2000):
    """The decode step issued as a direct pa_decode call and as a replay of
    its recorded CUDA graph (DecodeGraphs, sequence interval 8, KV interval
    256): steps back to back (host issue cost and device time per step) and
    one step alone (launch to completion)."""
    import torch

    S, H, D = w.num_seqs, w.num_heads, w.head_dim
    mx = int(w.context_lens.max())
    tables, ctx = w.block_tables.to(dev), w.context_lens.to(dev)
    out = torch.empty(S, H, D, dtype=w.q.dtype, device=dev)
    err = pa.new_error_flag(dev)
    ws = pa.decode_workspace(S, H, D, mx, device=dev)
    g = pa.DecodeGraphs(w.k_pool, w.v_pool, max_seqs=S, max_context_len=mx, max_blocks_per_seq=w.max_blocks_per_seq,
                        scale=w.scale, err_flag=err, seq_interval=8, kv_interval=256)
    g.q[:S] = w.q
    g.tables[:S, :w.max_blocks_per_seq] = tables
    g.context_lens[:S] = ctx
    fns = {"direct": lambda: pa.pa_decode(out, w.q, w.k_pool, w.v_pool, tables, ctx, mx, w.scale, ws, err,
                                          stream=stream),
           "graph": lambda: g.run(S, mx, stream)}
    res = {}
    for label, fn in fns.items():
        for _ in range(20):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        t1 = time.perf_counter()
        torch.cuda.synchronize(dev)
        one = []
        for _ in range(50):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            one.append(a.elapsed_time(b) * 1e3)
        res[label] = {"us_per_step_back_to_back": e0.elapsed_time(e1) / n * 1e3,
                      "host_us_per_call": (t1 - t0) / n * 1e6, "us_one_step_alone": statistics.median(one)}
    if pa.pa_get_error(err, stream):
        raise RuntimeError("device error flags in the graph replay comparison")
    res["graphs_recorded"] = g.count
    g.close()
    return res


def run_swap(args, rank, world, local):
    line = measure_swap(args, rank, world, local)
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure_swap(args, rank, world, local):
    """Block swap between the GPU pool and a pinned host pool, by block size:
    the swap side of the pages' swap-versus-recompute comparison.  Each
    replica swaps the K/V of 8 requests x 2048 tokens (40 heads x 128, fp16)
    out to the host pool and back in, through pa_swap_blocks with the blocks
    scattered over a pool twice that size; the link's ceiling is one
    contiguous copy of the same bytes, timed the same way in the same run.
    The same blocks are also copied inside the GPU pool with pa_copy_blocks
    (the copy-on-write copy at batch scale: scattered sources to scattered
    destinations), against a contiguous device copy of the same bytes and
    the measured copy peak.  Returns the JSON line as a dict."""
    import numpy as np
    import torch

    import paged_kv_cache_35_gb300 as pa
    import pa_workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    H, D, tokens = 40, 128, 8 * 2048
    ev = lambda: torch.cuda.Event(enable_timing=True)
    K = max(1, min(args.steps, 50))

    def timed(fn):
        for _ in range(max(3, min(args.warmup, 10))):
            fn()
        torch.cuda.synchronize(dev)
        dist_barrier(world)
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(K):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return dist_max(a.elapsed_time(b) / K, world)

    sweep = []
    err = pa.new_error_flag(dev)
    clocks = ClockSampler(local)
    clocks.start()
    h0 = time.time()
    for B in (16, 32, 64, 128, 256):
        nb = tokens // B
        gk = W.normal((2 * nb, H, B, D), 71, torch.float16, dev)
        gv = W.normal((2 * nb, H, B, D), 72, torch.float16, dev)
        ck = torch.empty(nb, H, B, D, dtype=torch.float16).pin_memory()
        cv = torch.empty_like(ck).pin_memory()
        g = torch.Generator().manual_seed(B)
        scattered = torch.randperm(2 * nb, generator=g)[:nb]
        out_pairs = torch.stack([scattered, torch.arange(nb)], 1).to(torch.int32).to(dev)
        in_pairs = torch.stack([torch.arange(nb), scattered.flip(0)], 1).to(torch.int32).to(dev)
        nbytes = 2 * nb * H * B * D * 2
        t_out = timed(lambda: pa.pa_swap_blocks(gk, gv, ck, cv, out_pairs, err, stream))
        t_in = timed(lambda: pa.pa_swap_blocks(ck, cv, gk, gv, in_pairs, err, stream))
        slab_k, slab_v = gk[:nb], gv[:nb]
        t_cout = timed(lambda: (ck.copy_(slab_k, non_blocking=True), cv.copy_(slab_v, non_blocking=True)))
        t_cin = timed(lambda: (slab_k.copy_(ck, non_blocking=True), slab_v.copy_(cv, non_blocking=True)))
        # copy-on-write copies at batch scale: nb scattered sources to nb other scattered blocks
        perm = torch.randperm(2 * nb, generator=g)
        copy_pairs = torch.stack([perm[:nb], perm[nb:]], 1).to(torch.int32).to(dev)
        t_copy = timed(lambda: pa.pa_copy_blocks(gk, gv, copy_pairs, err, stream))
        dst_k, dst_v = gk[nb:], gv[nb:]
        t_dcopy = timed(lambda: (dst_k.copy_(slab_k), dst_v.copy_(slab_v)))
        if pa.pa_get_error(err, stream):
            raise RuntimeError("device error flags during the swap sweep")
        sweep.append({"block_size": B, "blocks": nb, "bytes": nbytes,
                      "swap_out_ms": t_out, "swap_in_ms": t_in,
                      "swap_out_GBs": nbytes / t_out / 1e6, "swap_in_GBs": nbytes / t_in / 1e6,
                      "contiguous_out_GBs": nbytes / t_cout / 1e6, "contiguous_in_GBs": nbytes / t_cin / 1e6,
                      "copy_blocks_ms": t_copy, "copy_blocks_GBs": 2 * nbytes / t_copy / 1e6,
                      "contiguous_device_copy_GBs": 2 * nbytes / t_dcopy / 1e6})
        del gk, gv, ck, cv
    h1 = time.time()
    clocks.stop()
    head = sweep[0]
    value = 2 * head["bytes"] * world / ((head["swap_out_ms"] + head["swap_in_ms"]) / 1e3) / 1e9
    link = 2 * head["bytes"] / ((head["bytes"] / head["contiguous_out_GBs"] + head["bytes"] / head["contiguous_in_GBs"])
                                / 1e9) / 1e9
    line = {"metric": "paged KV block swap, GPU pool <-> pinned host pool (swap-out + swap-in)", "value": value,
            "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": max(3, min(args.warmup, 10)),
            "ms_per_step": head["swap_out_ms"] + head["swap_in_ms"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT["swap"], "block_size": 16, "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "link", "achieved": value / world, "peak": link, "unit": "GB/s",
                         "frac": value / world / link, "traffic": None,
                         "peak_kind": "measured in this run: one contiguous copy of the same bytes each way"},
            "gpu_launches": 2 * K, "sweep_by_block_size": sweep,
            "clocks": clocks.summary(h0, h1)}
    peak, peak_kind = load_peaks()
    cb = head["copy_blocks_GBs"]
    line["copy_blocks_roofline"] = {
        "bound": "hbm", "achieved": cb, "peak": peak, "unit": "GB/s", "frac": cb / peak, "traffic": None,
        "peak_kind": f"{peak_kind} copy bandwidth", "kernel": "copy_blocks_kernel (pa_copy_blocks)",
        "algorithmic_bytes_per_launch": 2 * head["bytes"], "avg_launch_ms": head["copy_blocks_ms"],
        "note": f"{head['blocks']} pairs of 16-token blocks (40 heads x 128, fp16), K and V read and written; "
                "the contiguous device copy of the same bytes in this run reached "
                f"{head['contiguous_device_copy_GBs']:.0f} GB/s"}
    return line


def run_prefix_cache(args, rank, world, local):
    """Prefix caching on the GPU: 16 requests whose prompts share a
    1024-token system prompt and end in 256 tokens of their own.  With the
    allocator's prefix cache the prompt's 64 blocks are held once (filled by
    an earlier request) and each step prefills only the 16 suffixes over
    them (chunks of 256 queries at context 1024); without it every request
    holds and prefills its whole 1280-token prompt.  Reports both prefill
    times, the blocks held, and checks that the suffix rows agree bit for
    bit."""
    import numpy as np
    import torch

    import paged_kv_cache_35_gb300 as pa
    import pa_workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    n_req, shared, own, H, D, B = 16, 1024, 256, 40, 128, 16
    L = shared + own
    g = torch.Generator().manual_seed(7)
    sys_ids = torch.randint(0, 32000, (shared,), generator=g).tolist()
    prompts = [sys_ids + torch.randint(0, 32000, (own,), generator=g).tolist() for _ in range(n_req + 1)]
    # K/V/q of a position depend on its whole prefix: equal for the shared prompt, drawn per request after it
    kv_sys = [W.normal((shared, H, D), 300 + i, torch.bfloat16) for i in range(3)]
    kv_own = [[W.normal((own, H, D), 1000 * (r + 1) + i, torch.bfloat16) for i in range(3)] for r in range(n_req + 1)]
    full = lambda r, i: torch.cat([kv_sys[i], kv_own[r][i]])
    err = pa.new_error_flag(dev)
    scale = 1.0 / np.sqrt(D)

    def build(cached: bool):
        nb = (n_req + 1) * (L // B) + 8
        alloc = pa.BlockAllocator(nb, B, prefix_cache=cached)
        kp = torch.zeros(nb, H, B, D, dtype=torch.bfloat16, device=dev)
        vp = torch.zeros_like(kp)
        ks, vs, slots, first = [], [], [], []
        for r in range(n_req + 1):  # request 0 fills the cache (when there is one)
            n0 = alloc.add_seq_prefix(r, prompts[r])
            first.append(n0)
            for p_ in range(n0, L):
                slots.append(int(alloc.append_tokens([r], [prompts[r][p_]])[0][0]))
            ks.append(full(r, 0)[n0:])
            vs.append(full(r, 1)[n0:])
        pa.pa_reshape_and_cache(torch.cat(ks).to(dev), torch.cat(vs).to(dev), kp, vp,
                                torch.tensor(slots, dtype=torch.int64, device=dev), err, stream)
        reqs = list(range(1, n_req + 1))
        mb = L // B
        tables, _ = alloc.block_tables(reqs, mb)
        c0 = [first[r] for r in reqs]
        q = torch.cat([full(r, 2)[first[r]:] for r in reqs]).to(dev)
        lens = [L - x for x in c0]
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
        out = torch.empty(q.shape[0], H, D, dtype=torch.bfloat16, device=dev)
        cb = torch.tensor(c0, dtype=torch.int32, device=dev)
        tb = torch.from_numpy(tables).to(dev)
        held = nb - alloc.num_free()
        fn = lambda: pa.pa_prefill_chunk(out, q, cu, cb, kp, vp, tb, max(lens), scale, err, stream)
        flops = sum(4 * D * H * sum(x + i + 1 for i in range(L - x)) for x in c0)
        alloc.close()
        return fn, out, lens, held, flops, c0

    res = {}
    outs = {}
    for cached in (True, False):
        fn, out, lens, held, flops, c0 = build(cached)
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize(dev)
        K = max(5, min(args.steps, 200))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / K
        key = "cached" if cached else "uncached"
        res[key] = {"prefill_us": ms * 1e3, "queries": sum(lens), "context_before": c0[0], "gflop": flops / 1e9,
                    "tflops": flops / (ms / 1e3) / 1e12, "blocks_held": held}
        outs[key] = (out, lens)
    if pa.pa_get_error(err, stream):
        raise RuntimeError("device error flags in the prefix-cache workload")
    # the suffix rows of the uncached prefill must equal the cached prefill's rows
    oc, _ = outs["cached"]
    ou, lu = outs["uncached"]
    rows = torch.cat([torch.arange(sum(lu[:i]) + shared, sum(lu[:i + 1])) for i in range(n_req)]).to(dev)
    same = bool(torch.equal(ou[rows].view(torch.int16), oc.view(torch.int16)))
    if not same:
        raise RuntimeError("cached and uncached prefill rows differ")
    speed = res["uncached"]["prefill_us"] / res["cached"]["prefill_us"]
    line = {"metric": "prefill time with a cached shared prompt, relative to prefilling whole prompts", "value": speed,
            "unit": "x", "n_gpus": world, "steps": K, "warmup": max(3, args.warmup), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT["prefix_cache"], "parallelism": f"replicas x{world}"},
            "cached": res["cached"], "uncached": res["uncached"],
            "memory_saving": 1.0 - res["cached"]["blocks_held"] / res["uncached"]["blocks_held"],
            "suffix_rows_bit_identical": same, "gpu_launches": K}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_batch_sweep(args, rank, world, local):
    """Decode latency against batch size, paged against contiguous: every
    sequence has 1024 tokens, 40 heads x 128, fp16.  "paged": 16-token
    blocks at random places in the pool; "contiguous": one 1024-token block
    per sequence, the sequences' blocks in order (the K/V of a (sequence,
    head) is one contiguous run, as without paging).  Same kernel, same
    arithmetic; the difference is the cost of paging."""
    import statistics

    import torch

    import paged_kv_cache_35_gb300 as pa
    import pa_workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    H, D, ctx_len = 40, 128, 1024
    rows = []
    for S in (1, 2, 4, 8, 16, 32, 64, 128, 256):
        ctx = torch.full((S,), ctx_len, dtype=torch.int32)
        w = W._decode_workload("batch_sweep_paged", ctx, ctx - 1, H, D, 16, "f16", device=dev)
        tables = w.block_tables.to(dev)
        lens = w.context_lens.to(dev)
        # the same K/V, gathered per sequence in logical order: [S][H][ctx_len][D]
        pos = torch.arange(ctx_len, device=dev)
        blk = tables[:, pos // 16].long()  # [S][ctx_len]
        gather = lambda pool: pool[blk, :, (pos % 16).expand(S, ctx_len), :].permute(0, 2, 1, 3).contiguous()
        k_c, v_c = gather(w.k_pool), gather(w.v_pool)
        t_c = torch.arange(S, dtype=torch.int32, device=dev).reshape(S, 1)
        res = {"batch": S}
        outs = {}
        for kind, kp, vp, tb, B in (("paged", w.k_pool, w.v_pool, tables, 16), ("contiguous", k_c, v_c, t_c, ctx_len)):
            out = torch.empty(S, H, D, dtype=torch.float16, device=dev)
            ws = pa.decode_workspace(S, H, D, ctx_len, device=dev)
            err = pa.new_error_flag(dev)
            fn = lambda: pa.pa_decode(out, w.q, kp, vp, tb, lens, ctx_len, w.scale, ws, err, stream=stream)
            for _ in range(10):
                fn()
            torch.cuda.synchronize(dev)
            ts = []
            for _ in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(50):
                    fn()
                b.record(stream)
                torch.cuda.synchronize(dev)
                ts.append(a.elapsed_time(b) / 50 * 1e3)
            if pa.pa_get_error(err, stream):
                raise RuntimeError("device error flags in the batch sweep")
            us = statistics.median(ts)
            res[kind + "_us"] = us
            res[kind + "_GBs"] = decode_bytes([ctx_len] * S, H, D, B, 2) / us / 1e3
            outs[kind] = out
        res["bit_identical"] = bool(torch.equal(outs["paged"].view(torch.int16), outs["contiguous"].view(torch.int16)))
        res["paged_over_contiguous"] = res["paged_us"] / res["contiguous_us"]
        rows.append(res)
        del w, k_c, v_c
    worst = max(r["paged_over_contiguous"] for r in rows)
    line = {"metric": "decode latency, 16-token pages relative to contiguous K/V (worst over batch sizes)",
            "value": worst, "unit": "x", "n_gpus": world, "steps": 250, "warmup": 10, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT["batch_sweep"], "parallelism": f"replicas x{world}"},
            "sweep": rows, "gpu_launches": 2 * 250 * len(rows) * 2}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_memsim(args, rank, world):
    """Host-only: KV memory holding tokens under Orca-Max / Orca-Pow2 /
    Orca-Oracle reservations and under the paged allocator, on two seeded
    synthetic traces, plus parallel-sampling and beam-search block sharing."""
    if rank != 0:
        return
    from paged_kv_cache_35_gb300 import memsim

    t0 = time.perf_counter()
    n_req = max(50, min(args.steps, 600))
    traces = {kind: memsim.synthetic_trace(kind, n_req, seed=1) for kind in ("long_tail", "short")}
    policies = {kind: {p: memsim.simulate(p, tr, 32768).summary() for p in memsim.POLICIES}
                for kind, tr in traces.items()}
    sharing = memsim.sharing_over_trace(traces["long_tail"][:100])
    value = 100.0 * policies["long_tail"]["paged"]["token_fraction"]
    line = {"metric": "KV-cache memory holding tokens, paged blocks (time average)", "value": value, "unit": "%",
            "n_gpus": 0, "steps": n_req, "warmup": 0, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int64", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT["memsim"], "capacity_tokens": 32768, "block_size": 16,
                       "max_len": 2048, "requests_per_trace": n_req},
            "policies": policies, "sharing": sharing, "wall_s": time.perf_counter() - t0}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_TEXT), default="llama13b",
                    help="llama13b (the headline configuration) or another configuration")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of CPU-oracle timing")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--num-seqs", type=int, default=0,
                    help="long_context only: the first N sequences of the same length draw (a smaller case for "
                         "profiling captures); 0 = all 256")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="default run: time only the headline configuration")
    args = ap.parse_args()
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, rank, int(os.environ.get("WORLD_SIZE", "1")))
        return
    if args.workload == "memsim":
        run_memsim(args, int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")))
        return
    rank, world, local = dist_setup()
    if args.workload == "swap":
        run_swap(args, rank, world, local)
    elif args.workload == "prefix_cache":
        run_prefix_cache(args, rank, world, local)
    elif args.workload == "batch_sweep":
        run_batch_sweep(args, rank, world, local)
    elif args.workload in ("prefill", "prefill_f16"):
        run_prefill(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
