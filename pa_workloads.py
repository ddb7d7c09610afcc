"""Seeded synthetic inputs for the paged KV-cache hot path.

This module feeds both the CUDA path and the CPU oracle.  It holds none of
the method's arithmetic: no attention, no token-to-slot mapping, no block
allocation policy.  It only draws random values, context lengths, and the
physical block ids that each sequence's logical blocks are given (a block
table is an *input* of paged attention: "Efficient Memory Management for
Large Language Model Serving with PagedAttention", section 4, the kernel
translates logical positions through the block table).

Recipe (shared by tests and the benchmark):
  * values: torch.Generator(device).manual_seed(seed), fp32 N(0,1), then a
    round-to-nearest cast to fp16/bf16.  The same bits go to both sides.
  * lengths: their own seed (1 unless a workload says otherwise).
  * placement: a seeded torch.randperm of the pool; sequence s takes the
    next n_s ids in logical order, so blocks are fragmented at random.
  * pool size: ceil(1.1 * blocks in use) unless a workload pins it.
  * unused table entries are -1 (any read of them is an indexing bug).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}

SEED_DATA = 0
SEED_LENS = 1
SEED_SUFFIX = 2


def normal(shape, seed: int, dtype: torch.dtype, device="cpu") -> torch.Tensor:
    """fp32 N(0,1) draws from a seeded generator, cast to ``dtype``."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    return x.to(dtype)


def randint(lo: int, hi: int, n: int, seed: int) -> torch.Tensor:
    """n integers uniform in [lo, hi] (inclusive), int32, CPU."""
    g = torch.Generator()
    g.manual_seed(seed)
    return torch.randint(lo, hi + 1, (n,), generator=g, dtype=torch.int64).to(torch.int32)


def lognormal_lengths(n: int, median: float, sigma: float, lo: int, hi: int, seed: int) -> torch.Tensor:
    """round(exp(N(ln median, sigma))) clipped to [lo, hi], int32, CPU."""
    g = torch.Generator()
    g.manual_seed(seed)
    z = torch.randn(n, generator=g, dtype=torch.float64)
    x = torch.exp(math.log(median) + sigma * z).round().clamp(lo, hi)
    return x.to(torch.int32)


def blocks_for(capacity_tokens: int, block_size: int) -> int:
    """Whole blocks needed to hold ``capacity_tokens`` tokens (input sizing)."""
    return -(-int(capacity_tokens) // block_size)


def random_tables(capacities, block_size: int, num_blocks: int, seed: int):
    """Block tables that give sequence s ``blocks_for(capacities[s])`` distinct
    physical ids drawn from a seeded permutation of ``range(num_blocks)``.

    Returns (tables int32 [S][MB] padded with -1, max_blocks_per_seq).
    """
    nblk = [blocks_for(c, block_size) for c in capacities]
    need = sum(nblk)
    if need > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {need}")
    g = torch.Generator()
    g.manual_seed(seed)
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    mb = max(1, max(nblk) if nblk else 1)
    tables = torch.full((len(nblk), mb), -1, dtype=torch.int32)
    o = 0
    for s, n in enumerate(nblk):
        tables[s, :n] = perm[o:o + n]
        o += n
    return tables, mb


def pool_size(capacities, block_size: int, slack: float = 1.1) -> int:
    return int(math.ceil(slack * sum(blocks_for(c, block_size) for c in capacities)))


@dataclass
class DecodeWorkload:
    """One decode step: new token written at ``new_pos`` then attention over
    ``context_lens`` tokens.  Pools are [num_blocks][H][B][D]."""
    name: str
    num_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    dtype: str
    context_lens: torch.Tensor      # int32 [S]
    new_pos: torch.Tensor           # int32 [S] position of the token written this step
    block_tables: torch.Tensor      # int32 [S][MB]
    max_blocks_per_seq: int
    q: torch.Tensor                 # [S][H][D]
    k_new: torch.Tensor             # [S][H][D]
    v_new: torch.Tensor             # [S][H][D]
    k_pool: torch.Tensor            # [NB][H][B][D]
    v_pool: torch.Tensor
    scale: float
    extra: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.numel())


def _decode_workload(name, ctx, new_pos, H, D, B, dtype, seed=SEED_DATA, device="cpu",
                     num_blocks=None, scale=None, placement_seed=None) -> DecodeWorkload:
    ctx = ctx.to(torch.int32)
    new_pos = new_pos.to(torch.int32)
    caps = [max(int(c), int(p) + 1) for c, p in zip(ctx.tolist(), new_pos.tolist())]
    nb = num_blocks if num_blocks is not None else pool_size(caps, B)
    tables, mb = random_tables(caps, B, nb, seed if placement_seed is None else placement_seed)
    S = len(caps)
    dt = DTYPES[dtype]
    base = 1000 * seed
    return DecodeWorkload(
        name=name, num_heads=H, head_dim=D, block_size=B, num_blocks=nb, dtype=dtype,
        context_lens=ctx, new_pos=new_pos, block_tables=tables, max_blocks_per_seq=mb,
        q=normal((S, H, D), base + 1, dt, device),
        k_new=normal((S, H, D), base + 2, dt, device),
        v_new=normal((S, H, D), base + 3, dt, device),
        k_pool=normal((nb, H, B, D), base + 4, dt, device),
        v_pool=normal((nb, H, B, D), base + 5, dt, device),
        scale=(1.0 / math.sqrt(D)) if scale is None else scale,
    )


def tiny_decode(device="cpu") -> DecodeWorkload:
    """4 sequences, 4 heads, head_dim 64, block 16, contexts {1,16,17,45}, a
    32-block pool with random placement, fp16, scale 1/8.  The new token of
    each sequence goes into its next slot (position = context length)."""
    ctx = torch.tensor([1, 16, 17, 45], dtype=torch.int32)
    return _decode_workload("tiny_paged_decode", ctx, ctx.clone(), 4, 64, 16, "f16",
                            num_blocks=32, scale=1.0 / 8.0, device=device)


def llama13b_decode(device="cpu", num_seqs=64) -> DecodeWorkload:
    """LLaMA-13B-shaped single-layer decode: 64 sequences, 40 heads x 128,
    block 16, contexts uniform in [128, 2048], fp16, pool = blocks in use +10%.
    The step writes each sequence's newest token (position ctx-1) and attends
    over ctx tokens."""
    ctx = randint(128, 2048, num_seqs, SEED_LENS)
    return _decode_workload("llama13b_decode_b64", ctx, ctx - 1, 40, 128, 16, "f16", device=device)


def long_context_decode(device="cpu", num_seqs=256) -> DecodeWorkload:
    """256 sequences, 32 heads x 128, block 16, bf16, log-normal contexts
    (median 1024, sigma 1.0, clipped to [16, 16384]), random placement."""
    ctx = lognormal_lengths(num_seqs, 1024.0, 1.0, 16, 16384, SEED_LENS)
    return _decode_workload("long_context_decode_b256", ctx, ctx - 1, 32, 128, 16, "bf16", device=device)


@dataclass
class SharedPrefixScript:
    """Parallel sampling: ``num_prompts`` prompts of ``prompt_len`` tokens,
    each continued by ``samples`` sequences with their own suffix lengths.
    Each side (allocator + kernels, or the oracle's model) replays it."""
    num_prompts: int
    samples: int
    prompt_len: int
    suffix_lens: torch.Tensor       # int32 [num_prompts * samples]
    num_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    dtype: str
    prompt_k: torch.Tensor          # [P][prompt_len][H][D]
    prompt_v: torch.Tensor
    suffix_k: torch.Tensor          # [P*samples][max_suffix][H][D]
    suffix_v: torch.Tensor
    q: torch.Tensor                 # [P*samples][H][D]
    pool_init_k: torch.Tensor       # [NB][H][B][D] initial pool contents (garbage)
    pool_init_v: torch.Tensor
    scale: float


def shared_prefix(device="cpu", num_prompts=8, samples=8, prompt_len=1000, max_suffix=256,
                  H=40, D=128, B=16) -> SharedPrefixScript:
    """8 prompts x 8 samples, prompt 1000 tokens (last prompt block partial),
    suffix uniform in [1, 256], 40 heads x 128, block 16, fp16."""
    n = num_prompts * samples
    suf = randint(1, max_suffix, n, SEED_SUFFIX)
    prompt_blocks = blocks_for(prompt_len, B)
    # every sample may need one copied block plus blocks for its suffix
    per_sample = 1 + blocks_for(max_suffix, B)
    nb = int(math.ceil(1.1 * (num_prompts * prompt_blocks + n * per_sample)))
    dt = DTYPES["f16"]
    base = 1000 * SEED_DATA
    ms = int(suf.max())
    return SharedPrefixScript(
        num_prompts=num_prompts, samples=samples, prompt_len=prompt_len, suffix_lens=suf,
        num_heads=H, head_dim=D, block_size=B, num_blocks=nb, dtype="f16",
        prompt_k=normal((num_prompts, prompt_len, H, D), base + 11, dt, device),
        prompt_v=normal((num_prompts, prompt_len, H, D), base + 12, dt, device),
        suffix_k=normal((n, ms, H, D), base + 13, dt, device),
        suffix_v=normal((n, ms, H, D), base + 14, dt, device),
        q=normal((n, H, D), base + 15, dt, device),
        pool_init_k=normal((nb, H, B, D), base + 16, dt, device),
        pool_init_v=normal((nb, H, B, D), base + 17, dt, device),
        scale=1.0 / math.sqrt(D),
    )


@dataclass
class MixedWorkload:
    """Decode sequences plus prefill chunks sharing one paged pool.

    Sequence order in ``block_tables``/``context_lens``: the decode sequences
    first, then one entry per prefill chunk whose length is
    ctx_before + chunk_len (the chunk's own tokens are written first)."""
    decode: DecodeWorkload           # tables/pool below are shared with it
    chunk_lens: torch.Tensor         # int32 [C]
    ctx_before: torch.Tensor         # int32 [C]
    chunk_q: torch.Tensor            # [sum chunk_lens][H][D]
    chunk_k: torch.Tensor            # [sum chunk_lens][H][D] K/V of the chunk tokens
    chunk_v: torch.Tensor
    chunk_tables: torch.Tensor       # int32 [C][MB]


def mixed_prefill(device="cpu", num_decode=32, chunk_len=512, ctx_before=(1024, 3072),
                  H=40, D=128, B=256, dtype="bf16") -> MixedWorkload:
    """32 decode sequences (contexts uniform in [256, 4096]) plus 2 prefill
    chunks of 512 query tokens appended to paged contexts of 1024 and 3072
    tokens; 40 heads x 128, page size 256, bf16."""
    dctx = randint(256, 4096, num_decode, SEED_LENS)
    C = len(ctx_before)
    cb = torch.tensor(list(ctx_before), dtype=torch.int32)
    cl = torch.full((C,), chunk_len, dtype=torch.int32)
    all_ctx = torch.cat([dctx, cb + cl])
    new_pos = torch.cat([dctx - 1, cb + cl - 1])
    w = _decode_workload("mixed_chunked_prefill", all_ctx, new_pos, H, D, B, dtype, device=device)
    w.context_lens = dctx.clone()
    w.new_pos = (dctx - 1).to(torch.int32)
    tables = w.block_tables
    w.block_tables = tables[:num_decode].contiguous()
    w.q = w.q[:num_decode].contiguous()
    w.k_new = w.k_new[:num_decode].contiguous()
    w.v_new = w.v_new[:num_decode].contiguous()
    dt = DTYPES[dtype]
    base = 1000 * SEED_DATA
    T = int(cl.sum())
    return MixedWorkload(
        decode=w, chunk_lens=cl, ctx_before=cb,
        chunk_q=normal((T, H, D), base + 21, dt, device),
        chunk_k=normal((T, H, D), base + 22, dt, device),
        chunk_v=normal((T, H, D), base + 23, dt, device),
        chunk_tables=tables[num_decode:].contiguous(),
    )


def budget512_step(device="cpu") -> MixedWorkload:
    """One step under a 512-token budget, filled the way the continuous
    batching page's scheduler fills it: the 32 running requests' decode tokens
    first (contexts uniform in [256, 4096]), then 480 tokens of the prefill in
    progress -- the fourth 480-token chunk of a long prompt, at context 1440.
    40 heads x 128, page size 256, bf16."""
    return mixed_prefill(device=device, num_decode=32, chunk_len=480, ctx_before=(1440,))


def small_prefill(device="cpu", chunk_lens=(130, 77), ctx_before=(200, 37), H=3, D=128, B=16,
                  dtype="bf16", seed=SEED_DATA) -> MixedWorkload:
    """A small chunked-prefill case (ragged chunks, ragged contexts) that the
    oracle finishes in well under a second."""
    C = len(chunk_lens)
    cb = torch.tensor(list(ctx_before), dtype=torch.int32)
    cl = torch.tensor(list(chunk_lens), dtype=torch.int32)
    total = cb + cl
    w = _decode_workload("small_prefill", total, total - 1, H, D, B, dtype, seed=seed, device=device)
    dt = DTYPES[dtype]
    base = 1000 * seed
    T = int(cl.sum())
    return MixedWorkload(
        decode=w, chunk_lens=cl, ctx_before=cb,
        chunk_q=normal((T, H, D), base + 21, dt, device),
        chunk_k=normal((T, H, D), base + 22, dt, device),
        chunk_v=normal((T, H, D), base + 23, dt, device),
        chunk_tables=w.block_tables.clone(),
    )


def small_decode(device="cpu", ctx=(1, 15, 16, 17, 33, 300, 700, 1029), H=3, D=128, B=16,
                 dtype="f16", seed=SEED_DATA, num_blocks=None) -> DecodeWorkload:
    """A small multi-tile decode case with ragged tails (several 512-token
    partitions for the longest sequences)."""
    c = torch.tensor(list(ctx), dtype=torch.int32)
    return _decode_workload("small_decode", c, c - 1, H, D, B, dtype, seed=seed, device=device,
                            num_blocks=num_blocks)
