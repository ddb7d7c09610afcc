"""KV-cache memory waste: reservation baselines against paged blocks.

Host-only simulator of how much KV-cache memory holds tokens under four
allocation policies, on a seeded synthetic request trace:

* the three reservation baselines of the PagedAttention paper summary
  (section 7, "실험 환경 및 워크로드"): Orca-Max reserves the maximum
  sequence length for every request, Orca-Pow2 the prompt plus the output
  length rounded up to a power of two, Orca-Oracle exactly the prompt plus
  the true output length -- each as one contiguous region, first fit, in a
  linear KV address space;
* paged: the library's block allocator (blocks on demand, freed at the end).

Waste categories (the summary's section 3 and Figure 3, the blog page's
"従来手法の問題" list): for a request holding a region of R slots, with c
tokens so far and f tokens at its end,
  reserved               = min(R, f) - c   (slots its later tokens will fill),
  internal fragmentation = R - max(f, c)   (slots no token will ever fill),
  external fragmentation = the free space, at a step where the next waiting
                           request cannot be placed although the free space
                           in total would hold it.
Paged blocks have no reservation and no external fragmentation; their
internal fragmentation is the unfilled tail of each sequence's last block.

It also measures the block sharing of parallel sampling and beam search
(summary section 6, Figures 20-21): blocks in use with copy-on-write sharing
against every sequence holding its own copy.

Scheduling is the plainest iteration-level loop: first come first served,
a request is admitted when its region (paged: its prompt's blocks) fits,
every running request gains one token per step, a request leaves when its
output is complete.  A paged request is admitted when its prompt's blocks
fit with 1% of the pool to spare; a paged step that runs out of blocks
preempts the most recently admitted request (blocks freed, request
re-queued at the front to start over).

The request lengths are synthetic (the pages' ShareGPT and Alpaca traces are
not available): "long_tail" draws log-normal prompt and output lengths with
long tails, "short" draws short, narrow uniform ones.
"""
from __future__ import annotations

import bisect
import math
import random
from dataclasses import dataclass, field

POLICIES = ("orca_max", "orca_pow2", "orca_oracle", "paged")


@dataclass
class Request:
    rid: int
    prompt: int
    output: int

    @property
    def final(self) -> int:
        return self.prompt + self.output


def synthetic_trace(kind: str, n: int, seed: int = 0, max_len: int = 2048) -> list:
    """n requests with seeded lengths; prompt + output <= max_len."""
    rng = random.Random(seed)
    out = []
    for i in range(n):
        if kind == "long_tail":
            p = int(min(max(round(math.exp(rng.gauss(math.log(160), 1.0))), 4), max_len // 2))
            o = int(min(max(round(math.exp(rng.gauss(math.log(200), 1.0))), 1), max_len - p))
        elif kind == "short":
            p = rng.randint(8, 96)
            o = rng.randint(8, 160)
        else:
            raise ValueError(f"unknown trace kind {kind}")
        out.append(Request(i, p, o))
    return out


def reservation(policy: str, req: Request, max_len: int) -> int:
    if policy == "orca_max":
        return max_len
    if policy == "orca_pow2":
        return min(max_len, req.prompt + (1 << max(0, (req.output - 1).bit_length())))
    if policy == "orca_oracle":
        return req.final
    raise ValueError(policy)


class FirstFit:
    """Contiguous regions in [0, capacity): the lowest-addressed hole that
    fits is used; freed regions merge with free neighbours."""

    def __init__(self, capacity: int):
        self.capacity = capacity
        self.holes = [(0, capacity)]  # (start, size), sorted by start

    def alloc(self, size: int):
        for i, (st, sz) in enumerate(self.holes):
            if sz >= size:
                if sz == size:
                    self.holes.pop(i)
                else:
                    self.holes[i] = (st + size, sz - size)
                return st
        return None

    def free(self, start: int, size: int):
        i = bisect.bisect_left(self.holes, (start, 0))
        self.holes.insert(i, (start, size))
        merged = []
        for st, sz in self.holes:
            if merged and merged[-1][0] + merged[-1][1] == st:
                merged[-1] = (merged[-1][0], merged[-1][1] + sz)
            else:
                merged.append((st, sz))
        self.holes = merged

    def free_total(self) -> int:
        return sum(sz for _, sz in self.holes)


@dataclass
class SimResult:
    policy: str
    steps: int = 0
    completed: int = 0
    preemptions: int = 0
    token_slot_steps: int = 0      # sum over steps of tokens held
    reserved_steps: int = 0
    internal_steps: int = 0
    external_steps: int = 0
    batch_steps: int = 0           # sum over steps of running requests
    capacity: int = 0
    extra: dict = field(default_factory=dict)

    def summary(self) -> dict:
        occupied = self.token_slot_steps + self.reserved_steps + self.internal_steps + self.external_steps
        f = (lambda x: x / occupied) if occupied else (lambda x: 0.0)
        return {"policy": self.policy, "steps": self.steps, "completed": self.completed,
                "preemptions": self.preemptions,
                "token_fraction": f(self.token_slot_steps), "reserved_fraction": f(self.reserved_steps),
                "internal_fragmentation_fraction": f(self.internal_steps),
                "external_fragmentation_fraction": f(self.external_steps),
                "mean_batch": self.batch_steps / self.steps if self.steps else 0.0,
                "mean_capacity_used": (occupied - self.external_steps) / self.steps / self.capacity
                if self.steps else 0.0}


def simulate(policy: str, trace, capacity_tokens: int, block_size: int = 16, max_len: int = 2048,
             max_steps: int = 1_000_000) -> SimResult:
    """Run the trace to completion (or max_steps) under one policy."""
    from collections import deque

    res = SimResult(policy, capacity=capacity_tokens)
    queue = deque(trace)
    running = []  # [req, length so far, region start (contiguous) , region size]
    if policy == "paged":
        from . import BlockAllocator, PAError, PA_ERR_NO_FREE_BLOCKS

        nb = capacity_tokens // block_size
        alloc = BlockAllocator(nb, block_size)
        B = block_size
    else:
        ff = FirstFit(capacity_tokens)

    def admit_paged(req) -> bool:
        # the prompt's blocks plus a watermark of 1% of the pool (at least one
        # block) left for the running requests' growth
        need = -(-req.prompt // B) + max(1, nb // 100)
        if alloc.num_free() < need:
            return False
        alloc.add_seq(req.rid)
        for _ in range(req.prompt):
            alloc.append_slots([req.rid])
        return True

    while (queue or running) and res.steps < max_steps:
        blocked_need = 0
        while queue:
            req = queue[0]
            if policy == "paged":
                if not admit_paged(req):
                    break
                running.append([req, req.prompt, 0, 0])
            else:
                size = reservation(policy, req, max_len)
                if size > capacity_tokens:
                    raise ValueError(f"request {req.rid} needs {size} > capacity")
                st = ff.alloc(size)
                if st is None:
                    blocked_need = size
                    break
                running.append([req, req.prompt, st, size])
            queue.popleft()
        if not running:
            raise RuntimeError("nothing fits the capacity")
        # one decode step: every running request gains a token
        if policy == "paged":
            while True:
                try:
                    alloc.append_slots([r[0].rid for r in running])
                    break
                except PAError as e:
                    if e.status != PA_ERR_NO_FREE_BLOCKS or len(running) == 1:
                        raise
                    victim = running.pop()  # the most recently admitted
                    alloc.free_seq(victim[0].rid)
                    queue.appendleft(victim[0])
                    res.preemptions += 1
        for r in running:
            r[1] += 1
        # account this step
        res.steps += 1
        res.batch_steps += len(running)
        tokens = sum(r[1] for r in running)
        res.token_slot_steps += tokens
        if policy == "paged":
            used = (alloc.num_blocks - alloc.num_free()) * B
            res.internal_steps += used - tokens
        else:
            for req, c, _, R in running:
                res.reserved_steps += min(R, req.final) - c
                res.internal_steps += R - max(req.final, c)
            free = ff.free_total()
            if blocked_need and free >= blocked_need:
                res.external_steps += free
        # leave when complete
        keep = []
        for r in running:
            if r[1] >= r[0].final:
                res.completed += 1
                if policy == "paged":
                    alloc.free_seq(r[0].rid)
                else:
                    ff.free(r[2], r[3])
            else:
                keep.append(r)
        running = keep
    if policy == "paged":
        alloc.close()
    return res


def sharing_parallel_sampling(n_samples: int, prompt: int, outputs, block_size: int = 16) -> dict:
    """One prompt, n samples of the given output lengths: peak blocks with the
    prompt shared (fork after the prompt, copy-on-write of the shared partial
    block) against each sample holding its own copy of the prompt."""
    from . import BlockAllocator

    assert len(outputs) == n_samples
    B = block_size
    total = sum(-(-(prompt + o) // B) for o in outputs) + n_samples
    a = BlockAllocator(total, B)
    a.add_seq(0)
    for _ in range(prompt):
        a.append_slots([0])
    for s in range(1, n_samples):
        a.fork(0, s)
    left = list(outputs)
    peak = 0
    live = list(range(n_samples))
    while live:
        a.append_slots(live)
        peak = max(peak, a.num_blocks - a.num_free())
        for s in list(live):
            left[s] -= 1
            if left[s] == 0:
                live.remove(s)
    a.close()
    unshared = sum(-(-(prompt + o) // B) for o in outputs)
    return {"samples": n_samples, "shared_peak_blocks": peak, "unshared_blocks": unshared,
            "saving": 1.0 - peak / unshared}


def sharing_beam_search(width: int, prompt: int, steps: int, seed: int = 0, block_size: int = 16) -> dict:
    """Beam search of `width` beams for `steps` tokens after a prompt: each
    step every new beam extends a parent drawn from the current beams
    (favouring the better-ranked ones), the old beams are freed.  Blocks in
    use with sharing (fork + copy-on-write) against every beam holding its
    own copy, averaged over the steps."""
    from . import BlockAllocator

    rng = random.Random(seed)
    B = block_size
    cap = width * (-(-(prompt + steps) // B) + 2) + 4
    a = BlockAllocator(cap, B)
    a.add_seq(0)
    for _ in range(prompt):
        a.append_slots([0])
    beams = [0]
    nxt = 1
    shared_sum = unshared_sum = 0
    length = prompt
    for _ in range(steps):
        weights = [1.0 / (1 + i) for i in range(len(beams))]
        parents = rng.choices(beams, weights=weights, k=width)
        new = []
        for p in parents:
            a.fork(p, nxt)
            new.append(nxt)
            nxt += 1
        for b in beams:
            a.free_seq(b)
        a.append_slots(new)
        beams = new
        length += 1
        shared_sum += a.num_blocks - a.num_free()
        unshared_sum += width * -(-length // B)
    a.close()
    return {"width": width, "mean_shared_blocks": shared_sum / steps, "mean_unshared_blocks": unshared_sum / steps,
            "saving": 1.0 - shared_sum / unshared_sum}


def sharing_over_trace(trace, samples=(2, 4, 6), widths=(2, 4, 6), block_size: int = 16, max_steps: int = 256,
                       seed: int = 0) -> dict:
    """Parallel sampling (every sample as long as the request's output) and
    beam search (the request's output length, at most max_steps, as the beam
    steps) over the requests of a trace: total blocks with sharing against
    without, per sample count and beam width."""
    par, beam = {}, {}
    for n in samples:
        sh = un = 0
        for r in trace:
            x = sharing_parallel_sampling(n, r.prompt, [r.output] * n, block_size)
            sh += x["shared_peak_blocks"]
            un += x["unshared_blocks"]
        par[n] = 1.0 - sh / un
    for w in widths:
        sh = un = 0.0
        for r in trace:
            x = sharing_beam_search(w, r.prompt, min(r.output, max_steps), seed + r.rid, block_size)
            sh += x["mean_shared_blocks"]
            un += x["mean_unshared_blocks"]
        beam[w] = 1.0 - sh / un
    return {"parallel_sampling_saving": par, "beam_search_saving": beam}
