// Paged decode attention for sm_103a.
//
// Method: PagedAttention ("Efficient Memory Management for Large Language
// Model Serving with PagedAttention"), paper-summary page section 4 and
// Figure 6: one query per sequence attends to K/V kept in fixed-size,
// non-contiguous blocks found through a per-sequence block table.  The blog
// page ("SOSP 2023論文解説: vLLM", section "Attention計算の修正") states the
// result as softmax(q [K_1 | ... | K_n]^T / sqrt(d)) [V_1 | ... | V_n],
// computed block by block with an online softmax.
//
// Design (ours, for one GB300):
//  * The context of every sequence is cut into split-KV partitions of P
//    tokens; a unit of work is one (sequence, head, partition).  A one-CTA
//    planning kernel lists the (sequence, partition) items longest first
//    (counting sort on the partition's 16-token chunk count) so the
//    persistent grid finishes with short units.
//  * The decode kernel is persistent (SM count x resident CTAs) and warp
//    specialised:
//      warp 5  (scheduler) takes unit ids from a global counter, reads the
//              item and the table entries of the unit into a 4-deep unit
//              queue in shared memory, bulk-copies the unit's query row next
//              to them, and merges each finished unit;
//      warp 4  (producer)  streams the unit's 16-token K and V tiles (one
//              contiguous 16*D*2-byte run each in the [NB][H][B][D] pools)
//              into shared-memory ring slots with cp.async.bulk, completion
//              counted in bytes on one mbarrier per slot; tile j of a unit
//              goes to consumer warp j % 4, into that warp's own slots;
//      warps 0-3 (consumers) take every 4th tile of the unit: 8 lanes per
//              token row, 16-byte shared loads (conflict free), fp32 dot
//              products reduced with 3 shuffles, online softmax (running max
//              and sum, base-2 exponent with log2(e) folded into the query).
//    Each consumer warp leaves its (max, sum, output) for the unit in shared
//    memory and goes on to the next unit at once; the scheduler warp merges
//    the four shares (so no streaming warp ever waits on a merge).  A unit
//    that is the only partition of its sequence writes the output directly.
//    Otherwise the scheduler writes the normalised partial and (max, sum) to
//    the workspace, and the one that completes the last partition of a
//    (sequence, head) merges all partitions with the log-sum-exp rule in
//    partition order (so the result does not depend on scheduling, nor on
//    which physical blocks hold the tokens).
//  * Each CTA's first unit is its own index (no counter round trip at start);
//    the work items carry their token count and partition count, so the
//    scheduler's chain is counter -> item -> table entries.
//  * Both kernels are programmatic dependents of the kernel before them: the
//    planning kernel may overlap a slot scatter that releases it early and
//    waits for it only at its end; the decode grid is resident while the
//    planning runs and waits for it before reading anything.
//  * pa_mixed_step (end of this file) puts the chunked prefill between the
//    planning kernel and the decode kernel so that the two run concurrently.
//  * pa_decode_grouped: for groups of sequences that share a prompt's blocks
//    (parallel samples, beams), the planning kernel validates the groups and
//    lists only each sequence's own tokens; the group kernel (tensor-core
//    products of each tile with all of a group's queries) reads every shared
//    prefix once and streams the listed items too (see the group kernel).
//  * What the planning kernel writes (work list, counters, prefixes) is read
//    by its dependents with coherent loads: they run while it writes.
//  * Every wait is bounded; bad table entries are flagged, never trapped.
#include <math.h>

#include <atomic>
#include <cstdio>
#include <mutex>

#include <cudaTypedefs.h>

#include <type_traits>

#include "pa_common.cuh"

namespace pa {

#ifndef PA_DECODE_STAGES
#define PA_DECODE_STAGES 4
#endif
#ifndef PA_DECODE_CONSUMER_WARPS
#define PA_DECODE_CONSUMER_WARPS 4
#endif
#ifndef PA_DECODE_MIN_CTAS
#define PA_DECODE_MIN_CTAS 5
#endif

constexpr int kChunk = 16;                    // tokens per ring stage
constexpr int kConsumerWarps = PA_DECODE_CONSUMER_WARPS;
constexpr int kProducerWarp = kConsumerWarps;  // the warp after the consumers
constexpr int kSchedulerWarp = kConsumerWarps + 1;
constexpr int kDecodeThreads = (kConsumerWarps + 2) * 32;
constexpr int kStages = PA_DECODE_STAGES;
// Each consumer warp owns its own kSlotsPerWarp ring slots and consumes them
// strictly in order, so every waiter on a slot's mbarrier observes every
// phase of it: a parity wait can never alias a phase two ahead.
constexpr int kSlotsPerWarp = kStages / kConsumerWarps;
static_assert(kStages % kConsumerWarps == 0, "ring slots must split evenly over the consumer warps");
constexpr int kUnitQueue = 4;
constexpr int kMaxPartition = 1024;
constexpr int kMaxChunksPerUnit = kMaxPartition / kChunk;
constexpr int kPlanThreads = 1024;


struct DecodeArgs {
  void* out;
  int out_dtype;
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* context_lens;
  int max_context_len;
  int num_seqs;
  int num_heads;
  int block_size;
  int num_blocks;
  float qscale;  // scale * log2(e)
  int partition_size;
  int max_parts;
  int* counters;   // [0] unit counter, [1] item count, [2 + s*H + h] partition arrivals
  int4* items;     // (sequence, partition, first token, tokens | partitions << 11), processing order
  float2* part_ml; // [S][H][max_parts] (max, sum) in log2 units
  float* part_o;   // [S][H][max_parts][D] normalised partial outputs
  int32_t* err_flag;
  int dep_wait;    // 1: wait for the planning kernel (launched right before); 0: it completed before the
                   // kernel this one was launched behind
  // pa_decode_grouped only (num_groups == 0 otherwise): sequences
  // group_start[g] .. group_start[g+1]-1 share their first group_prefix[g]
  // tokens; the planning kernel validates each group and leaves in
  // seq_prefix[s] the tokens of s that the group kernel covers (0 if none).
  int num_groups;
  const int32_t* group_start;
  const int32_t* group_prefix;
  int32_t* seq_prefix;
};

template <int D, typename T>
struct DecodeSmem {
  T ring[kStages][2][kChunk * D];  // K tile, V tile
  T qbuf[kUnitQueue][D];
  int32_t chunk_blk[kUnitQueue][kMaxChunksPerUnit];
  int4 unit[kUnitQueue];  // sequence (< 0: no more units), head, partition, tokens in partition
  int unit_nparts[kUnitQueue];
  int unit_tok0[kUnitQueue];
  float co[kUnitQueue][kConsumerWarps][D];  // each consumer warp's share of a unit
  float cm[kUnitQueue][kConsumerWarps];
  float cl[kUnitQueue][kConsumerWarps];
  int slot_ok[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t ufull[kUnitQueue];  // unit published: 1 arrival + the query row's bytes
  uint64_t udone[kUnitQueue];  // every consumer warp has left its share of the unit
  int abort_flag;
};

__device__ __forceinline__ bool length_ok(const DecodeArgs& a, int ctx) {
  return ctx >= 0 && ctx <= a.max_context_len && (int64_t)ctx <= (int64_t)a.max_blocks_per_seq * a.block_size;
}

// ---------------------------------------------------------------------------------
// Planning kernel: one CTA.  Lists the (sequence, partition) items, longest
// first; resets the unit counter and the per-(sequence, head) arrival
// counters; writes zero rows for empty or invalid sequences.
constexpr int kGroupMax = 8;  // sequences of a group: the 8 columns of one mma n-block

// One warp per group (warp w of nw takes groups w, w + nw, ...): a group is
// used when its range lies in [0, S) and holds 1..kGroupMax sequences, its
// prefix is a multiple of 16 tokens (whole tiles: no tile reads a row past
// it) and at most every member's context length, and every member's table
// equals the first member's over the prefix's blocks.  Otherwise
// PA_FLAG_BAD_GROUP is raised and its members are decoded whole.
__device__ __forceinline__ void validate_groups(const DecodeArgs& a, int w, int nw, int lane) {
  const int S = a.num_seqs, B = a.block_size;
  for (int g = w; g < a.num_groups; g += nw) {
    const int g0 = __ldg(a.group_start + g), g1 = __ldg(a.group_start + g + 1);
    const int pre = __ldg(a.group_prefix + g);
    bool ok = g0 >= 0 && g1 > g0 && g1 <= S && g1 - g0 <= kGroupMax && pre >= 0 && pre % kChunk == 0;
    if (ok && pre > 0) {
      const int nblk = (pre + B - 1) / B;
      if ((long long)nblk > a.max_blocks_per_seq) ok = false;
      if (ok && lane < g1 - g0) {
        const int ctx = __ldg(a.context_lens + g0 + lane);
        if (!length_ok(a, ctx) || pre > ctx) ok = false;
      }
      if (ok) {
        const int32_t* t0 = a.block_tables + (size_t)g0 * a.max_blocks_per_seq;
        const int n = (g1 - g0 - 1) * nblk;  // (member, block) pairs after the first member
        for (int i = lane; i < n; i += 32) {
          const int m = 1 + i / nblk, b = i - (m - 1) * nblk;
          if (__ldg(a.block_tables + (size_t)(g0 + m) * a.max_blocks_per_seq + b) != __ldg(t0 + b)) ok = false;
        }
      }
      ok = __all_sync(0xffffffffu, ok);
    } else {
      ok = __all_sync(0xffffffffu, ok);
    }
    if (!ok) {
      if (lane == 0) atomicOr(a.err_flag, PA_FLAG_BAD_GROUP);
      continue;
    }
    if (lane < g1 - g0) a.seq_prefix[g0 + lane] = pre;
  }
}

template <int D>
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const DecodeArgs a) {
  griddep_launch_dependents();
  extern __shared__ int plan_smem[];
  const int P = a.partition_size;
  const int nb = P / kChunk;  // buckets: chunks in an item, 1..nb
  int* hist = plan_smem;
  int* offs = plan_smem + nb;
  int* cur = plan_smem + 2 * nb;
  const int tid = threadIdx.x;
  const int S = a.num_seqs, H = a.num_heads;
  for (int i = tid; i < nb; i += blockDim.x) {
    hist[i] = 0;
    cur[i] = 0;
  }
  for (int i = tid; i < S * H; i += blockDim.x) a.counters[2 + i] = 0;
  if (a.num_groups > 0) {
    for (int s = tid; s < S; s += blockDim.x) a.seq_prefix[s] = 0;
    __syncthreads();
    validate_groups(a, tid >> 5, blockDim.x >> 5, tid & 31);
  }
  __syncthreads();
  // item sizes: full partitions of P tokens, then the last part of each
  // sequence (1..P tokens); a shared prefix (grouped calls) is not listed:
  // the group kernel covers it, in partitions 0 .. ceil(prefix / P) - 1
  for (int s = tid; s < S; s += blockDim.x) {
    const int ctx = __ldg(a.context_lens + s);
    if (!length_ok(a, ctx) || ctx == 0) continue;
    const int rest = ctx - (a.num_groups > 0 ? a.seq_prefix[s] : 0);
    if (rest == 0) continue;
    const int nfull = (rest - 1) / P;
    const int last = rest - nfull * P;
    if (nfull > 0) atomicAdd(&hist[nb - 1], nfull);
    atomicAdd(&hist[(last + kChunk - 1) / kChunk - 1], 1);
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int b = nb - 1; b >= 0; --b) {
      offs[b] = acc;
      acc += hist[b];
    }
    a.counters[0] = 0;
    a.counters[1] = acc;
  }
  __syncthreads();
  for (int s = tid; s < S; s += blockDim.x) {
    const int ctx = __ldg(a.context_lens + s);
    if (!length_ok(a, ctx) || ctx == 0) {
      if (ctx != 0) atomicOr(a.err_flag, PA_FLAG_BAD_LENGTH);
      for (int i = 0; i < H * D; ++i) store_out(a.out, (size_t)s * H * D + i, a.out_dtype, 0.f);
      continue;
    }
    const int skip = a.num_groups > 0 ? a.seq_prefix[s] : 0;
    const int np0 = (skip + P - 1) / P;  // partitions of the shared prefix
    const int rest = ctx - skip;
    if (rest == 0) continue;
    const int nfull = (rest - 1) / P;
    const int last = rest - nfull * P;
    const int nparts = np0 + nfull + 1;
    if (nfull > 0) {
      const int base = offs[nb - 1] + atomicAdd(&cur[nb - 1], nfull);
      for (int p = 0; p < nfull; ++p) a.items[base + p] = make_int4(s, np0 + p, skip + p * P, P | (nparts << 11));
    }
    const int bkt = (last + kChunk - 1) / kChunk - 1;
    a.items[offs[bkt] + atomicAdd(&cur[bkt], 1)] =
        make_int4(s, np0 + nfull, skip + nfull * P, last | (nparts << 11));
  }
  // Launched as a programmatic dependent of the kernel before it (which may
  // still be running, e.g. the slot scatter writing the pool): finish only
  // after it has, so that the decode kernel's wait on this kernel also
  // covers it.  The planning itself reads only the context lengths, which
  // kernels that release their dependents early do not write.
  griddep_wait();
}

// Packed fp32 pairs: two independent IEEE fp32 operations per instruction
// (round to nearest even, as the scalar forms).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// The 8 elements of a 16-byte vector as 4 fp32 pairs (elements 2i, 2i+1).
template <typename T>
__device__ __forceinline__ void to_pairs(const uint4& u, uint64_t* p);
template <>
__device__ __forceinline__ void to_pairs<__nv_bfloat16>(const uint4& u, uint64_t* p) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = f2_pack(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}
template <>
__device__ __forceinline__ void to_pairs<__half>(const uint4& u, uint64_t* p) {
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 x = __half22float2(h[i]);
    p[i] = f2_pack(x.x, x.y);
  }
}

// ---------------------------------------------------------------------------------
// Consumer: one 16-token tile.  Lane (t4 = lane/8, c = lane%8) owns tokens
// t4, t4+4, t4+8, t4+12 of the tile and the 16-byte vectors c (+8) of each
// row: a group of 8 lanes reads one 128-byte stretch of a row, so the
// shared-memory loads are conflict free.  The query, the output and each
// row's elements are held as fp32 pairs (dimensions 2i, 2i+1); a score is the
// sum of the even and the odd dimensions' dot products.
template <int D, typename T>
__device__ __forceinline__ void consume_tile(const T* __restrict__ Ks, const T* __restrict__ Vs, int nvalid,
                                             const uint64_t* q2, float& m, float& l, uint64_t* o2, int lane) {
  constexpr int VPL = D / 64;
  const int t4 = lane >> 3;
  const int c = lane & 7;
  float sc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int tok = t4 + 4 * i;
    const T* row = Ks + tok * D;
    uint64_t acc2 = 0;  // (+0, +0)
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
      const uint4 u = *reinterpret_cast<const uint4*>(row + (c + 8 * v) * 8);
      uint64_t f[4];
      to_pairs<T>(u, f);
#pragma unroll
      for (int e = 0; e < 4; ++e) acc2 = f2_fma(q2[v * 4 + e], f[e], acc2);
    }
    const float2 ac = f2_unpack(acc2);
    float acc = ac.x + ac.y;
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    sc[i] = tok < nvalid ? acc : -INFINITY;
  }
  float cmax = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
  cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 8));
  cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, 16));
  const float m_new = fmaxf(m, cmax);
  const float alpha = exp2f(m - m_new);
  float pr[4];
  float psum = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    pr[i] = exp2f(sc[i] - m_new);
    psum += pr[i];
  }
  l = l * alpha + psum;
  const uint64_t alpha2 = f2_pack(alpha, alpha);
#pragma unroll
  for (int e = 0; e < 4 * VPL; ++e) o2[e] = f2_mul(o2[e], alpha2);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int tok = t4 + 4 * i;
    if (tok < nvalid) {  // rows past the context may hold any bits (even NaN)
      const T* row = Vs + tok * D;
      const uint64_t p2 = f2_pack(pr[i], pr[i]);
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        const uint4 u = *reinterpret_cast<const uint4*>(row + (c + 8 * v) * 8);
        uint64_t f[4];
        to_pairs<T>(u, f);
#pragma unroll
        for (int e = 0; e < 4; ++e) o2[v * 4 + e] = f2_fma(p2, f[e], o2[v * 4 + e]);
      }
    }
  }
  m = m_new;
}

// Merge of all partitions of one (sequence, head) by one warp, in partition
// order: M = max m_p, out = sum_p 2^(m_p - M) l_p o_p / sum_p 2^(m_p - M) l_p.
// The partials are read kMergeBatch at a time (their loads in flight
// together) and summed one by one in partition order, so the result does not
// depend on the batching.
constexpr int kMergeBatch = 4;
template <int D>
__device__ __forceinline__ void merge_partitions(const DecodeArgs& a, int s, int h, int nparts, int lane) {
  const size_t base = ((size_t)s * a.num_heads + h) * a.max_parts;
  float M = -INFINITY;
  for (int p0 = 0; p0 < nparts; p0 += kMergeBatch) {
    float mp[kMergeBatch];
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i) mp[i] = p0 + i < nparts ? __ldcg(&a.part_ml[base + p0 + i].x) : -INFINITY;
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i) M = fmaxf(M, mp[i]);
  }
  float L = 0.f;
  float O[D / 32];
#pragma unroll
  for (int i = 0; i < D / 32; ++i) O[i] = 0.f;
  for (int p0 = 0; p0 < nparts; p0 += kMergeBatch) {
    float2 ml[kMergeBatch];
    float ov[kMergeBatch][D / 32];
#pragma unroll
    for (int b = 0; b < kMergeBatch; ++b) {
      const bool in = p0 + b < nparts;
      ml[b] = in ? __ldcg(&a.part_ml[base + p0 + b]) : make_float2(-INFINITY, 0.f);
      const float* op = a.part_o + (base + p0 + b) * D;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) ov[b][i] = in ? __ldcg(op + lane + 32 * i) : 0.f;
    }
#pragma unroll
    for (int b = 0; b < kMergeBatch; ++b) {
      if (p0 + b >= nparts) break;
      const float w = (ml[b].x == -INFINITY) ? 0.f : exp2f(ml[b].x - M) * ml[b].y;
      L += w;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) O[i] = fmaf(w, ov[b][i], O[i]);
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const size_t ob = ((size_t)s * a.num_heads + h) * D;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) store_out(a.out, ob + lane + 32 * i, a.out_dtype, O[i] * inv);
  if (lane == 0) a.counters[2 + s * a.num_heads + h] = 0;
}

// Publish the CTA's k-th unit into queue slot k % kUnitQueue (whole warp).
// The first unit of every CTA is its own index; later ones come from the
// global counter.  Returns false when the work is exhausted: a "no more
// units" marker has been published instead.
template <int D, typename T>
__device__ __forceinline__ bool publish_unit(const DecodeArgs& a, DecodeSmem<D, T>& sm, int k,
                                             long long total_units, int lane) {
  const int H = a.num_heads;
  const int qs = k % kUnitQueue;
  int u = blockIdx.x;
  if (k > 0) {
    if (lane == 0) u = (int)gridDim.x + atomicAdd(a.counters, 1);
    u = __shfl_sync(0xffffffffu, u, 0);
  }
  if ((long long)u >= total_units) {
    if (lane == 0) {
      sm.unit[qs] = make_int4(-1, 0, 0, 0);
      mbar_arrive(&sm.ufull[qs]);
    }
    return false;
  }
  const int item = u / H;
  const int h = u - item * H;
  const int4 it = __ldcg(a.items + item);  // written by the planning kernel: coherent load
  const int s = it.x;
  const int tok0 = it.z;
  const int ntok = it.w & 2047;
  const int nchunks = (ntok + kChunk - 1) / kChunk;
  const int32_t* trow = a.block_tables + (size_t)s * a.max_blocks_per_seq;
  for (int j = lane; j < nchunks; j += 32) sm.chunk_blk[qs][j] = __ldg(trow + (tok0 + j * kChunk) / a.block_size);
  __syncwarp();
  if (lane == 0) {
    sm.unit[qs] = make_int4(s, h, it.y, ntok);
    sm.unit_nparts[qs] = it.w >> 11;
    sm.unit_tok0[qs] = tok0;
    __threadfence_block();
    mbar_arrive_expect_tx(&sm.ufull[qs], D * sizeof(T));
    bulk_g2s(sm.qbuf[qs], static_cast<const T*>(a.q) + ((size_t)s * H + h) * D, D * sizeof(T), &sm.ufull[qs]);
  }
  return true;
}

// Scheduler and merger (one warp).  Keeps kUnitQueue units published ahead
// of the consumers; when the consumer warps have all left their share of
// unit k, merges them (lane i owns output dimensions i, i+32, ...), writes
// the output or the partition's partial, and refills the slot with unit
// k + kUnitQueue.  The merge latency (global fences, the cross-partition
// merge) thus never stalls the warps that stream K and V.
template <int D, typename T>
__device__ __forceinline__ void run_scheduler(const DecodeArgs& a, DecodeSmem<D, T>& sm, int lane) {
  volatile int* abort_flag = &sm.abort_flag;
  const int H = a.num_heads;
  const long long total_units = (long long)__ldcg(a.counters + 1) * H;
  int published = 0;  // real units published
  bool more = true;
  while (more && published < kUnitQueue) {
    more = publish_unit<D, T>(a, sm, published, total_units, lane);
    if (more) ++published;
  }
  bool aborted = false;
  for (int k = 0; k < published; ++k) {
    const int qs = k % kUnitQueue;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(&sm.udone[qs], (k / kUnitQueue) & 1, abort_flag, a.err_flag);
    if (!__shfl_sync(0xffffffffu, ok, 0)) {
      aborted = true;
      break;
    }
    __syncwarp();
    const int4 un = sm.unit[qs];
    const int nparts = sm.unit_nparts[qs];
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm.cm[qs][w]);
    float L = 0.f;
    float O[D / 32];
#pragma unroll
    for (int i = 0; i < D / 32; ++i) O[i] = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float mw = sm.cm[qs][w];
      const float wt = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
      L = fmaf(wt, sm.cl[qs][w], L);
#pragma unroll
      for (int i = 0; i < D / 32; ++i) O[i] = fmaf(wt, sm.co[qs][w][lane + 32 * i], O[i]);
    }
    const int s = un.x, h = un.y, p = un.z;
    const float inv = L > 0.f ? 1.f / L : 0.f;
    if (nparts == 1) {
#pragma unroll
      for (int i = 0; i < D / 32; ++i)
        store_out(a.out, ((size_t)s * H + h) * D + lane + 32 * i, a.out_dtype, O[i] * inv);
    } else {
      const size_t pidx = ((size_t)s * H + h) * a.max_parts + p;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) a.part_o[pidx * D + lane + 32 * i] = O[i] * inv;
      if (lane == 0) a.part_ml[pidx] = make_float2(M, L);
      __threadfence();
      __syncwarp();
      int prev = 0;
      if (lane == 0) prev = atomicAdd(&a.counters[2 + s * H + h], 1);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if (prev == nparts - 1) {  // every partition of (s, h) is in: merge them
        __threadfence();
        merge_partitions<D>(a, s, h, nparts, lane);
      }
    }
    __syncwarp();
    if (more) {
      more = publish_unit<D, T>(a, sm, k + kUnitQueue, total_units, lane);
      if (more) ++published;
    }
  }
  if (lane == 0 && aborted) {  // let in-flight query copies land before exit
    for (int kk = max(0, published - kUnitQueue); kk < published; ++kk)
      mbar_wait_drain(&sm.ufull[kk % kUnitQueue], (kk / kUnitQueue) & 1);
  }
}

template <int D, typename T>
__device__ __forceinline__ void run_producer(const DecodeArgs& a, DecodeSmem<D, T>& sm) {
  constexpr uint32_t kTileBytes = kChunk * D * sizeof(T);
  volatile int* abort_flag = &sm.abort_flag;
  const int H = a.num_heads;
  const int B = a.block_size;
  const T* kp = static_cast<const T*>(a.k_pool);
  const T* vp = static_cast<const T*>(a.v_pool);
  uint32_t cnt[kConsumerWarps];  // tiles handed to each consumer warp so far
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) cnt[w] = 0;
  bool aborted = false;
  for (int k = 0; !aborted; ++k) {
    const int qs = k % kUnitQueue;
    if (!mbar_wait(&sm.ufull[qs], (k / kUnitQueue) & 1, abort_flag, a.err_flag)) break;
    const int4 un = sm.unit[qs];
    if (un.x < 0) break;
    const int h = un.y;
    const int tok0 = sm.unit_tok0[qs];
    const int nchunks = (un.w + kChunk - 1) / kChunk;
    for (int j0 = 0; j0 < nchunks && !aborted; j0 += kConsumerWarps) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const int j = j0 + w;
        if (j >= nchunks) break;
        const int slot = w * kSlotsPerWarp + (int)(cnt[w] % kSlotsPerWarp);
        if (!mbar_wait(&sm.empty[slot], ((cnt[w] / kSlotsPerWarp) & 1) ^ 1, abort_flag, a.err_flag)) {
          aborted = true;
          break;
        }
        const int32_t blk = sm.chunk_blk[qs][j];
        if (blk >= 0 && blk < a.num_blocks) {
          const int off = (tok0 + j * kChunk) % B;
          const size_t base = (((size_t)blk * H + h) * B + off) * D;
          sm.slot_ok[slot] = 1;
          mbar_arrive_expect_tx(&sm.full[slot], 2 * kTileBytes);
          bulk_g2s(sm.ring[slot][0], kp + base, kTileBytes, &sm.full[slot]);
          bulk_g2s(sm.ring[slot][1], vp + base, kTileBytes, &sm.full[slot]);
        } else {
          sm.slot_ok[slot] = 0;
          atomicOr(a.err_flag, PA_FLAG_BAD_BLOCK);
          mbar_arrive(&sm.full[slot]);
        }
        ++cnt[w];
      }
    }
  }
  if (*abort_flag) {  // let in-flight tile copies land before exit
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const uint32_t first = cnt[w] > (uint32_t)kSlotsPerWarp ? cnt[w] - kSlotsPerWarp : 0;
      for (uint32_t i = first; i < cnt[w]; ++i)
        mbar_wait_drain(&sm.full[w * kSlotsPerWarp + i % kSlotsPerWarp], (i / kSlotsPerWarp) & 1);
    }
  }
}

// Consumer warp: streams its tiles of each unit (every 4th tile, from its
// own ring slots, in order), then leaves its (max, sum, output) share of the
// unit in shared memory for the merger and moves straight on.
template <int D, typename T>
__device__ __forceinline__ void run_consumer(const DecodeArgs& a, DecodeSmem<D, T>& sm, int warp, int lane) {
  constexpr int VPL = D / 64;
  volatile int* abort_flag = &sm.abort_flag;
  const int c = lane & 7;
  uint32_t mine = 0;  // tiles this warp has taken so far (its own slots, in order)
  for (int k = 0;; ++k) {
    const int qs = k % kUnitQueue;
    bool ok = mbar_wait(&sm.ufull[qs], (k / kUnitQueue) & 1, abort_flag, a.err_flag);
    if (!__all_sync(0xffffffffu, ok)) break;
    const int4 un = sm.unit[qs];
    if (un.x < 0) break;
    uint64_t q2[4 * VPL];
    {
      const uint64_t qs2 = f2_pack(a.qscale, a.qscale);
#pragma unroll
      for (int v = 0; v < VPL; ++v) {
        const uint4 u = *reinterpret_cast<const uint4*>(&sm.qbuf[qs][(c + 8 * v) * 8]);
        to_pairs<T>(u, q2 + 4 * v);
      }
#pragma unroll
      for (int e = 0; e < 4 * VPL; ++e) q2[e] = f2_mul(q2[e], qs2);
    }

    const int ntok = un.w;
    const int nchunks = (ntok + kChunk - 1) / kChunk;
    float m = -INFINITY, l = 0.f;
    uint64_t o2[4 * VPL];
#pragma unroll
    for (int e = 0; e < 4 * VPL; ++e) o2[e] = 0;  // (+0, +0)
    bool aborted = false;
    for (int j = warp; j < nchunks; j += kConsumerWarps, ++mine) {
      const int slot = warp * kSlotsPerWarp + (int)(mine % kSlotsPerWarp);
      ok = mbar_wait(&sm.full[slot], (mine / kSlotsPerWarp) & 1, abort_flag, a.err_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        aborted = true;
        break;
      }
      if (sm.slot_ok[slot]) {
        consume_tile<D, T>(sm.ring[slot][0], sm.ring[slot][1], min(kChunk, ntok - j * kChunk), q2, m, l, o2, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[slot]);
    }
    if (aborted) break;

    // merge the 4 token groups of the warp, leave the share for the merger
    float o[8 * VPL];
#pragma unroll
    for (int e = 0; e < 4 * VPL; ++e) {
      const float2 x = f2_unpack(o2[e]);
      o[2 * e] = x.x;
      o[2 * e + 1] = x.y;
    }
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
#pragma unroll
    for (int e = 0; e < 8 * VPL; ++e) {
      o[e] += __shfl_xor_sync(0xffffffffu, o[e], 8);
      o[e] += __shfl_xor_sync(0xffffffffu, o[e], 16);
    }
    if (lane < 8) {
#pragma unroll
      for (int v = 0; v < VPL; ++v)
#pragma unroll
        for (int e = 0; e < 8; ++e) sm.co[qs][warp][(lane + 8 * v) * 8 + e] = o[v * 8 + e];
    }
    if (lane == 0) {
      sm.cm[qs][warp] = m;
      sm.cl[qs][warp] = l;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.udone[qs]);
  }
}

template <int D, typename T>
__global__ void __launch_bounds__(kDecodeThreads, PA_DECODE_MIN_CTAS) decode_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t decode_smem_raw[];
  auto& sm = *reinterpret_cast<DecodeSmem<D, T>*>(decode_smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < kUnitQueue; ++i) {
      mbar_init(&sm.ufull[i], 1);
      mbar_init(&sm.udone[i], kConsumerWarps);
    }
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (a.dep_wait) griddep_wait();  // the planning kernel's list and counters are visible from here
  if (warp == kSchedulerWarp) {
    run_scheduler<D, T>(a, sm, lane);
  } else if (warp == kProducerWarp) {
    if (lane == 0) run_producer<D, T>(a, sm);
  } else {
    run_consumer<D, T>(a, sm, warp, lane);
  }
}

// ---------------------------------------------------------------------------------
// Group kernel (pa_decode_grouped): the shared prefix of a group of up to 8
// sequences (parallel samples or beams of one prompt, whose tables hold the
// same blocks there) is read once for all of them.  Persistent: each warp
// takes units from a counter, first the prefix units (group, head, prefix
// partition of P tokens), then the planned items of every sequence's own
// tokens (one unit per item and head, one query column), and streams the
// unit's 16-token K/V tiles through kGSlots ring slots of its own, issuing
// the tensor copies itself.  Per tile, with the unit's queries as the 8
// columns of an mma n-block (warp-level m16n8k16 products, fp32 accumulation):
//   S^T[16 tokens][8 queries] = K_tile . Q^T       (head_dim / 16 products)
//   online softmax per query (column), P^T rounded to the pool's type
//   O^T[D][8] += V_tile^T . P^T                    (head_dim / 16 products)
// P^T leaves the products' accumulator layout (token rows) for their B
// operand layout (query columns) through an 8x8 register transpose
// (movmatrix).  A bf16 P is two parts, P_hi + P_lo, as in the prefill, so
// that the weights carry ~16 bits; an fp16 P is one.  A unit writes each
// column's normalised partial (max, sum, o) into the partial arrays, and
// whichever partition of a (sequence, head) arrives last merges them all; a
// sequence whose tokens form one partition gets its output row directly.
constexpr int kGWarps = 4;   // units per CTA
constexpr int kGSlots = 3;   // ring slots per warp
constexpr int kGHalfBytes = kChunk * 128;  // 16 rows x 64 columns of 2 bytes, 128-byte swizzled

template <int D>
struct GroupSmem {
  uint8_t ring[kGWarps][kGSlots][2][D / 64][kGHalfBytes];  // [warp][slot][K, V][64-column half]
  uint64_t full[kGWarps][kGSlots];
};

__device__ __forceinline__ void g_tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

template <typename T>
__device__ __forceinline__ void mma_16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma_16816<__half>(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma_16816<__nv_bfloat16>(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two weights of one token row (queries 2c, 2c+1) rounded to the pool's type,
// packed low/high; *rest gets what rounding left (the bf16 second part).
template <typename T>
__device__ __forceinline__ uint32_t pack_p(float p0, float p1, float* r0, float* r1);
template <>
__device__ __forceinline__ uint32_t pack_p<__half>(float p0, float p1, float* r0, float* r1) {
  const __half2 h = __floats2half2_rn(p0, p1);
  *r0 = __low2float(h);  // the rounded values (their sum is the row sum)
  *r1 = __high2float(h);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack_p<__nv_bfloat16>(float p0, float p1, float* r0, float* r1) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
  *r0 = p0 - __low2float(h);  // the remainders, for P_lo
  *r1 = p1 - __high2float(h);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <typename T>
__device__ __forceinline__ uint32_t pack2(float x0, float x1);
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float x0, float x1) {
  const __half2 h = __floats2half2_rn(x0, x1);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float x0, float x1) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int D, typename T>
__global__ void __launch_bounds__(kGWarps * 32) group_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                             const __grid_constant__ CUtensorMap tm_v,
                                                             const DecodeArgs a, int prefix_parts) {
  constexpr int kHalves = D / 64;
  constexpr int kKSteps = D / 16;
  constexpr bool kTwoPart = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t kSlotTx = 2u * kHalves * kGHalfBytes;
  static_assert(kMaxPartition / kChunk <= 64, "two block ids per lane");
  extern __shared__ uint8_t group_smem_raw[];
  auto& sm = *reinterpret_cast<GroupSmem<D>*>(
      (reinterpret_cast<uintptr_t>(group_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (lane == 0) {
    for (int i = 0; i < kGSlots; ++i) mbar_init(&sm.full[warp][i], 1);
    fence_barrier_init();
  }
  __syncwarp();
  // The planning kernel (launched right before) has completed from here on.
  // Its output (the work list, the counters, the prefixes) is read with
  // coherent loads: it was written during this grid's lifetime, which the
  // read-only cache path does not allow for.
  griddep_wait();

  const int H = a.num_heads, P = a.partition_size, S = a.num_seqs, B = a.block_size;
  const long long n_prefix = (long long)a.num_groups * H * prefix_parts;
  const long long total = n_prefix + (long long)__ldcg(a.counters + 1) * H;  // + the planned items, per head
  // lane's rows of an m16n8 accumulator: r0 = lane / 4 and r0 + 8; its
  // columns: c0 = 2 (lane % 4) and c0 + 1
  const int r0 = lane >> 2;
  const int c0 = 2 * (lane & 3);
  // ldmatrix row addresses: lane i feeds matrix i / 8, its row i % 8
  const int lr = (lane & 7) + ((lane >> 3) & 1) * 8;  // K: row (token) of matrices 0..3
  const int lc = lane >> 4;                          // K: second 8 columns for matrices 2, 3
  const int vr = (lane & 7) + (lane >> 4) * 8;        // V (transposed load): token row
  const int vc = (lane >> 3) & 1;                     // V: second 8 dimensions for matrices 1, 3
  uint32_t x0 = 0;  // tiles this warp has streamed so far: slot and phase of tile j are those of x0 + j

  for (;;) {
    int uu = 0;
    if (lane == 0) uu = atomicAdd(a.counters, 1);
    const long long u = __shfl_sync(0xffffffffu, uu, 0);
    if (u >= total) break;
    // the unit: queries (columns) of sequences g0 .. g0+gn-1, head h, tokens
    // [tok0, tok0 + ntok) of g0's table, partial index p of nparts
    int g0, gn, h, tok0, ntok, p, nparts;  // nparts: 0 = per member (a shared prefix)
    if (u < n_prefix) {
      const int g = (int)(u / ((long long)H * prefix_parts));
      const int r = (int)(u - (long long)g * H * prefix_parts);
      h = r / prefix_parts;
      p = r - h * prefix_parts;
      g0 = __ldg(a.group_start + g);
      const int g1 = __ldg(a.group_start + g + 1);
      if (g0 < 0 || g0 >= S || g1 <= g0 || g1 > S || g1 - g0 > kGroupMax) continue;
      const int prefix = __ldcg(a.seq_prefix + g0);  // 0 unless the planning kernel accepted the group
      tok0 = p * P;
      if (tok0 >= prefix) continue;
      gn = g1 - g0;
      ntok = min(P, prefix - tok0);
      nparts = 0;
    } else {  // a planned item: one sequence's own tokens, a one-column unit
      const long long v = u - n_prefix;
      const int4 it = __ldcg(a.items + v / H);
      h = (int)(v - (v / H) * H);
      g0 = it.x;
      gn = 1;
      p = it.y;
      tok0 = it.z;
      ntok = it.w & 2047;
      nparts = it.w >> 11;
    }
    const int ntiles = (ntok + kChunk - 1) / kChunk;
    const int32_t* trow = a.block_tables + (size_t)g0 * a.max_blocks_per_seq;

    // the queries: B operand of S^T = K Q^T, column n = lane / 4 (member n),
    // rows (dimensions) 16 kk + 2 (lane % 4) + {0, 1} and + 8
    uint32_t qb[kKSteps][2];
    {
      const int n = lane >> 2;
      const T* qrow = static_cast<const T*>(a.q) + ((size_t)(g0 + n) * H + h) * D + c0;
#pragma unroll
      for (int kk = 0; kk < kKSteps; ++kk) {
        qb[kk][0] = n < gn ? __ldg(reinterpret_cast<const unsigned int*>(qrow + 16 * kk)) : 0u;
        qb[kk][1] = n < gn ? __ldg(reinterpret_cast<const unsigned int*>(qrow + 16 * kk + 8)) : 0u;
      }
    }
    // the unit's block ids, tile j's in lane j % 32 of blk_r[j / 32], read
    // once up front so that no copy waits on a table read
    int32_t blk_r[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int j = lane + 32 * r;
      blk_r[r] = j < ntiles ? __ldg(trow + (tok0 + j * kChunk) / B) : -1;
    }
    uint32_t bad = 0;  // bit s: slot s holds no data
    auto issue = [&](int j) {
      const int s = (int)((x0 + j) % kGSlots);
      const int tok = tok0 + j * kChunk;
      const int32_t blk = __shfl_sync(0xffffffffu, (j >> 5) ? blk_r[1] : blk_r[0], j & 31);
      if (blk >= 0 && blk < a.num_blocks) {
        bad &= ~(1u << s);
        if (lane == 0) {
          const int row = (int)(((long long)blk * H + h) * B + tok % B);
          uint64_t* bar = &sm.full[warp][s];
          mbar_arrive_expect_tx(bar, kSlotTx);
#pragma unroll
          for (int hf = 0; hf < kHalves; ++hf) {
            g_tma_load_2d(smem_u32(sm.ring[warp][s][0][hf]), &tm_k, 64 * hf, row, bar);
            g_tma_load_2d(smem_u32(sm.ring[warp][s][1][hf]), &tm_v, 64 * hf, row, bar);
          }
        }
      } else {
        bad |= 1u << s;
        if (lane == 0) {
          atomicOr(a.err_flag, PA_FLAG_BAD_BLOCK);
          mbar_arrive(&sm.full[warp][s]);
        }
      }
    };
    for (int j = 0; j < ntiles && j < kGSlots; ++j) issue(j);

    float m[2] = {-INFINITY, -INFINITY};  // running max per column (query), log2 units
    float l[2] = {0.f, 0.f};              // this lane's part of the column sums
    float o[kKSteps][4];                  // O^T: rows 16 mb + r0 (+8) = dimensions, columns = queries
#pragma unroll
    for (int mb = 0; mb < kKSteps; ++mb) o[mb][0] = o[mb][1] = o[mb][2] = o[mb][3] = 0.f;

    int j_abort = -1;  // the tile whose wait gave up
    for (int j = 0; j < ntiles; ++j) {
      const uint32_t x = x0 + j;
      const int s = (int)(x % kGSlots);
      const bool ok = mbar_wait(&sm.full[warp][s], (x / kGSlots) & 1, nullptr, a.err_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        j_abort = j;
        break;
      }
      const int valid = ntok - j * kChunk;  // rows of this tile inside the unit (>= 1)
      if (!((bad >> s) & 1u)) {
        const uint32_t kbase = smem_u32(sm.ring[warp][s][0][0]);
        const uint32_t vbase = smem_u32(sm.ring[warp][s][1][0]);
        if (valid < kChunk) {
          // V rows past the sequence's end may hold any bits (even NaN), and
          // a zero weight times NaN is NaN: clear them before the product
          const int per_half = (kChunk - valid) * 8;
          for (int i = lane; i < per_half * kHalves; i += 32) {
            const int hf = i / per_half, rem = i - hf * per_half;
            const int row = valid + (rem >> 3);
            *reinterpret_cast<uint4*>(sm.ring[warp][s][1][hf] + row * 128 + (rem & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();  // before the slot's next tensor copy overwrites these bytes
          __syncwarp();
        }
        float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < kKSteps; ++kk) {
          const int hf = kk >> 2, ch = (kk & 3) * 2 + lc;
          uint32_t af[4];
          ldsm_x4(kbase + hf * kGHalfBytes + lr * 128 + ((ch ^ (lr & 7)) << 4), af);
          mma_16816<T>(c, af, qb[kk][0], qb[kk][1]);
        }
        // scores in log2 units; rows past the unit do not count
        float sc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] = (r0 + 8 * (e >> 1)) < valid ? c[e] * a.qscale : -INFINITY;
        float tmax[2] = {fmaxf(sc[0], sc[2]), fmaxf(sc[1], sc[3])};
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
          tmax[0] = fmaxf(tmax[0], __shfl_xor_sync(0xffffffffu, tmax[0], sh));
          tmax[1] = fmaxf(tmax[1], __shfl_xor_sync(0xffffffffu, tmax[1], sh));
        }
        float alpha[2], pr[4];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const float mn = fmaxf(m[q], tmax[q]);
          alpha[q] = mn == -INFINITY ? 1.f : exp2f(m[q] - mn);
          m[q] = mn;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) pr[e] = m[e & 1] == -INFINITY ? 0.f : exp2f(sc[e] - m[e & 1]);
        float rest[4];
        const uint32_t p01 = pack_p<T>(pr[0], pr[1], &rest[0], &rest[1]);
        const uint32_t p23 = pack_p<T>(pr[2], pr[3], &rest[2], &rest[3]);
        if (kTwoPart) {
          l[0] = l[0] * alpha[0] + (pr[0] + pr[2]);
          l[1] = l[1] * alpha[1] + (pr[1] + pr[3]);
        } else {  // the rounded weights
          l[0] = l[0] * alpha[0] + (rest[0] + rest[2]);
          l[1] = l[1] * alpha[1] + (rest[1] + rest[3]);
        }
        // P^T as the B operand: column n = lane / 4 (query), rows = tokens
        const uint32_t b0 = movmatrix_trans(p01), b1 = movmatrix_trans(p23);
        uint32_t b0l = 0, b1l = 0;
        if (kTwoPart) {
          b0l = movmatrix_trans(pack2<T>(rest[0], rest[1]));
          b1l = movmatrix_trans(pack2<T>(rest[2], rest[3]));
        }
#pragma unroll
        for (int mb = 0; mb < kKSteps; ++mb) {
          o[mb][0] *= alpha[0];
          o[mb][1] *= alpha[1];
          o[mb][2] *= alpha[0];
          o[mb][3] *= alpha[1];
          const int ch = 2 * mb + vc, hf = ch >> 3, cin = ch & 7;
          uint32_t af[4];
          ldsm_x4_trans(vbase + hf * kGHalfBytes + vr * 128 + ((cin ^ (vr & 7)) << 4), af);
          mma_16816<T>(o[mb], af, b0, b1);
          if (kTwoPart) mma_16816<T>(o[mb], af, b0l, b1l);
        }
      }
      __syncwarp();  // every lane's reads of the slot are done
      if (j + kGSlots < ntiles) issue(j + kGSlots);
    }
    if (j_abort >= 0) {  // tiles j_abort .. j_abort + kGSlots - 1 were issued: let them land before exit
      if (lane == 0)
        for (int t = j_abort; t < ntiles && t < j_abort + kGSlots; ++t)
          mbar_wait_drain(&sm.full[warp][(x0 + t) % kGSlots], ((x0 + t) / kGSlots) & 1);
      return;
    }
    x0 += (uint32_t)ntiles;

    // column sums over the 8 lanes of each column pair
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], sh);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], sh);
    }
    if (nparts == 1) {  // a sequence whose tokens form one partition: its output row
      if (c0 == 0) {
        const float inv = l[0] > 0.f ? 1.f / l[0] : 0.f;
        const size_t ob = ((size_t)g0 * H + h) * D;
#pragma unroll
        for (int mb = 0; mb < kKSteps; ++mb) {
          store_out(a.out, ob + 16 * mb + r0, a.out_dtype, o[mb][0] * inv);
          store_out(a.out, ob + 16 * mb + r0 + 8, a.out_dtype, o[mb][2] * inv);
        }
      }
      continue;
    }
    // each member's normalised partial for partition p
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int n = c0 + q;
      if (n >= gn) continue;
      const size_t pidx = ((size_t)(g0 + n) * H + h) * a.max_parts + p;
      const float inv = l[q] > 0.f ? 1.f / l[q] : 0.f;
      float* po = a.part_o + pidx * D;
#pragma unroll
      for (int mb = 0; mb < kKSteps; ++mb) {
        po[16 * mb + r0] = o[mb][q] * inv;
        po[16 * mb + r0 + 8] = o[mb][q + 2] * inv;
      }
      if (r0 == 0) a.part_ml[pidx] = make_float2(m[q], l[q]);
    }
    __threadfence();
    __syncwarp();
    for (int n = 0; n < gn; ++n) {
      const int s = g0 + n;
      int np = nparts;
      if (np == 0) {  // a member of a shared prefix: its prefix partitions, then its own
        const int prefix = __ldcg(a.seq_prefix + g0);
        const int rest = __ldg(a.context_lens + s) - prefix;
        np = (prefix + P - 1) / P + (rest > 0 ? (rest + P - 1) / P : 0);
      }
      int prev = 0;
      if (lane == 0) prev = atomicAdd(&a.counters[2 + s * H + h], 1);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if (prev == np - 1) {  // every partition of (s, h) is in: merge them
        __threadfence();
        merge_partitions<D>(a, s, h, np, lane);
      }
    }
  }
}

}  // namespace pa

// ---------------------------------------------------------------------------------
// Host side
namespace {

struct WsLayout {
  size_t counters, items, ml, o, total;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

WsLayout ws_layout(int S, int H, int D, int max_parts) {
  WsLayout w;
  size_t off = 0;
  w.counters = off;
  off = align_up(off + sizeof(int) * (2 + (size_t)S * H), 256);
  w.items = off;
  off = align_up(off + sizeof(int4) * (size_t)S * max_parts, 256);
  w.ml = off;
  off = align_up(off + sizeof(float2) * (size_t)S * H * max_parts, 256);
  w.o = off;
  off = align_up(off + sizeof(float) * (size_t)S * H * max_parts * D, 256);
  w.total = off;
  return w;
}

// Partitions of the longest sequence (no overflow near INT_MAX).
int decode_max_parts(int max_ctx, int P) { return max_ctx > 0 ? (max_ctx - 1) / P + 1 : 1; }

// A work item packs a sequence's partition count above 11 bits of token count
// into one int32: fewer than 2^20 partitions per sequence.
constexpr int kMaxPartsPerSeq = 1 << 20;

int resolve_partition(int S, int H, int max_ctx, int partition_size) {
  if (partition_size == 0) return pa_decode_partition_size(S, H, max_ctx);
  return partition_size;
}

template <int D, typename T>
int configure_decode(int* occ_out) {
  using Smem = pa::DecodeSmem<D, T>;
  const int smem = (int)sizeof(Smem);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  // resident CTAs per SM, per device; 0 until the kernel is configured there.
  // Host threads may race to configure a device: the setup is idempotent and
  // the value is published only after it.
  static std::atomic<int> occupancy[64];
  if (dev < 0 || dev >= 64) return PA_ERR_CUDA;
  int occ = occupancy[dev].load(std::memory_order_acquire);
  if (occ == 0) {
    if (cudaFuncSetAttribute(pa::decode_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return PA_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, pa::decode_kernel<D, T>, pa::kDecodeThreads, smem) !=
        cudaSuccess)
      return PA_ERR_CUDA;
    if (occ < 1) occ = 1;
    occupancy[dev].store(occ, std::memory_order_release);
  }
  *occ_out = occ;
  return PA_OK;
}

// The planning kernel, as a programmatic dependent of the kernel before it.
template <int D>
int launch_plan(const pa::DecodeArgs& a, cudaStream_t stream) {
  const int nb = a.partition_size / pa::kChunk;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(pa::kPlanThreads);
  cfg.dynamicSmemBytes = 3 * nb * sizeof(int);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pa::plan_kernel<D>, a) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// The persistent decode kernel, launched as a programmatic dependent of the
// kernel before it on the stream.
template <int D, typename T>
int launch_main(const pa::DecodeArgs& a, cudaStream_t stream) {
  int occ = 0;
  const int st = configure_decode<D, T>(&occ);
  if (st != PA_OK) return st;
  const int sms = pa_host::device_sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  const long long max_units = (long long)a.num_seqs * a.num_heads * a.max_parts;
  long long grid = (long long)sms * occ;
  if (grid > max_units) grid = max_units;
  if (grid < 1) grid = 1;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(pa::kDecodeThreads);
  cfg.dynamicSmemBytes = sizeof(pa::DecodeSmem<D, T>);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, pa::decode_kernel<D, T>, a) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

// Planning kernel, then the decode kernel behind it.
template <int D, typename T>
int launch_decode(const pa::DecodeArgs& a, cudaStream_t stream) {
  int occ = 0;
  int st = configure_decode<D, T>(&occ);  // attribute calls before the first launch of the pair
  if (st != PA_OK) return st;
  st = launch_plan<D>(a, stream);
  if (st != PA_OK) return st;
  return launch_main<D, T>(a, stream);
}

int configure_any(int head_dim, int dtype) {
  int occ = 0;
  if (head_dim == 128)
    return dtype == PA_F16 ? configure_decode<128, __half>(&occ) : configure_decode<128, __nv_bfloat16>(&occ);
  return dtype == PA_F16 ? configure_decode<64, __half>(&occ) : configure_decode<64, __nv_bfloat16>(&occ);
}

int launch_main_any(const pa::DecodeArgs& a, int head_dim, int dtype, cudaStream_t s) {
  if (head_dim == 128)
    return dtype == PA_F16 ? launch_main<128, __half>(a, s) : launch_main<128, __nv_bfloat16>(a, s);
  return dtype == PA_F16 ? launch_main<64, __half>(a, s) : launch_main<64, __nv_bfloat16>(a, s);
}

// Checks pa_decode's arguments and fills the kernel arguments; launches
// nothing.  *empty is set when there is no work (num_seqs == 0).
int decode_setup(void* out, int out_dtype, const void* q, const void* k_pool, const void* v_pool,
                 const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                 int max_context_len, int num_seqs, int num_heads, int head_dim, int block_size, int num_blocks,
                 float scale, int dtype, void* workspace, size_t workspace_bytes, int partition_size,
                 int32_t* err_flag, pa::DecodeArgs& a, bool& empty) {
  empty = false;
  if (!pa_host::is_kv_dtype(dtype) || !pa_host::is_out_dtype(out_dtype)) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (block_size <= 0 || block_size % pa::kChunk != 0 || block_size > 65536) return PA_ERR_UNSUPPORTED;
  if (num_seqs < 0 || num_heads <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || max_context_len < 0)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) {
    empty = true;
    return PA_OK;
  }
  if (!out || !q || !k_pool || !v_pool || !block_tables || !context_lens || !workspace || !err_flag)
    return PA_ERR_INVALID_ARG;
  if (!pa_host::aligned16(q) || !pa_host::aligned16(k_pool) || !pa_host::aligned16(v_pool) ||
      !pa_host::aligned16(workspace) || !pa_host::aligned16(out))
    return PA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return PA_ERR_INVALID_ARG;
  if ((long long)num_seqs * num_heads > (1ll << 30)) return PA_ERR_INVALID_ARG;
  const int P = resolve_partition(num_seqs, num_heads, max_context_len, partition_size);
  if (P < pa::kChunk || P > pa::kMaxPartition || P % pa::kChunk != 0) return PA_ERR_INVALID_ARG;
  const int max_parts = decode_max_parts(max_context_len, P);
  if (max_parts >= kMaxPartsPerSeq) return PA_ERR_UNSUPPORTED;
  const WsLayout w = ws_layout(num_seqs, num_heads, head_dim, max_parts);
  if (workspace_bytes < w.total) return PA_ERR_WORKSPACE;

  a.out = out;
  a.out_dtype = out_dtype;
  a.q = q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.max_context_len = max_context_len;
  a.num_seqs = num_seqs;
  a.num_heads = num_heads;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.qscale = scale * 1.4426950408889634f;
  a.partition_size = P;
  a.max_parts = max_parts;
  char* ws = static_cast<char*>(workspace);
  a.counters = reinterpret_cast<int*>(ws + w.counters);
  a.items = reinterpret_cast<int4*>(ws + w.items);
  a.part_ml = reinterpret_cast<float2*>(ws + w.ml);
  a.part_o = reinterpret_cast<float*>(ws + w.o);
  a.err_flag = err_flag;
  a.dep_wait = 1;
  a.num_groups = 0;
  a.group_start = nullptr;
  a.group_prefix = nullptr;
  a.seq_prefix = nullptr;
  return PA_OK;
}

// pa_decode_grouped's workspace: pa_decode's with one more partition per
// sequence (a shared prefix ends mid-partition at most once), then the
// validated prefix length of every sequence.
struct GroupedLayout {
  WsLayout base;
  size_t seq_prefix, total;
};

GroupedLayout grouped_layout(int S, int H, int D, int max_parts) {
  GroupedLayout g;
  g.base = ws_layout(S, H, D, max_parts + 1);
  g.seq_prefix = g.base.total;
  g.total = align_up(g.seq_prefix + sizeof(int32_t) * (size_t)S, 256);
  return g;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A pool [num_blocks][heads][block][head_dim] as rows of head_dim elements;
// a copy is 16 rows of one 64-column half, 128-byte swizzled.
int encode_pool_map(CUtensorMap* m, const void* pool, int dtype, int head_dim, uint64_t rows) {
  auto encode = tensor_map_encoder();
  if (encode == nullptr) return PA_ERR_CUDA;
  const CUtensorMapDataType tdt = dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)pa::kChunk};
  cuuint32_t es[2] = {1, 1};
  return encode(m, tdt, 2, const_cast<void*>(pool), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? PA_OK
             : PA_ERR_CUDA;
}

// The group kernel, a persistent grid of as many CTAs as fit on the SMs,
// launched as a programmatic dependent of the planning kernel: its CTAs set
// up while the planning finishes and wait for it (griddepcontrol.wait) before
// reading anything the planning writes.
template <int D, typename T>
int launch_group(const pa::DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, int prefix_parts,
                 cudaStream_t stream) {
  const int smem = (int)sizeof(pa::GroupSmem<D>) + 1024;  // + room to align the ring to 1024 bytes
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
  static std::atomic<int> occupancy[64];  // resident CTAs per SM, per device (0: not configured)
  int occ = occupancy[dev].load(std::memory_order_acquire);
  if (occ == 0) {
    if (cudaFuncSetAttribute(pa::group_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return PA_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, pa::group_kernel<D, T>, pa::kGWarps * 32, smem) !=
        cudaSuccess)
      return PA_ERR_CUDA;
    if (occ < 1) occ = 1;
    occupancy[dev].store(occ, std::memory_order_release);
  }
  const int sms = pa_host::device_sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sms * occ));
  cfg.blockDim = dim3(pa::kGWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // setup overlaps the planning kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pa::group_kernel<D, T>, tk, tv, a, prefix_parts) == cudaSuccess ? PA_OK
                                                                                                 : PA_ERR_CUDA;
}

}  // namespace

namespace pa_host {

int decode_check(void* out, int out_dtype, const void* q, const void* k_pool, const void* v_pool,
                 const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                 int max_context_len, int num_seqs, int num_heads, int head_dim, int block_size, int num_blocks,
                 float scale, int dtype, void* workspace, size_t workspace_bytes, int partition_size,
                 int32_t* err_flag) {
  pa::DecodeArgs a;
  bool empty = false;
  return decode_setup(out, out_dtype, q, k_pool, v_pool, block_tables, max_blocks_per_seq, context_lens,
                      max_context_len, num_seqs, num_heads, head_dim, block_size, num_blocks, scale, dtype, workspace,
                      workspace_bytes, partition_size, err_flag, a, empty);
}

}  // namespace pa_host

extern "C" {

// Partition length from the batch shape, for the 760-CTA grid (152 SMs x 5),
// every sequence counted at the longest context:
//  * 1024 when every context fits one partition and the (sequence, head)
//    pairs alone give half a wave: no partials and no merge at all;
//  * 1024 when even 1024-token units make 16 waves or more, so the tail of
//    the longer units is negligible;
//  * otherwise the longest of 512, 256, 128, 64 that gives half a wave of
//    units (64 if none does).  With a few waves of ragged contexts, 1024-token
//    units leave a longer tail than 512-token ones.
int pa_decode_partition_size(int num_seqs, int num_heads, int max_context_len) {
  if (num_seqs <= 0 || num_heads <= 0 || max_context_len <= 0) return 512;
  const long long pairs = (long long)num_seqs * num_heads;
  if (pairs >= 380 && (max_context_len <= 1024 || pairs * ((max_context_len + 1023) / 1024) >= 16 * 760)) return 1024;
  int P = 512;
  while (P > 64 && pairs * ((max_context_len + P - 1) / P) < 380) P /= 2;
  return P;
}

size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                 int partition_size) {
  if (num_seqs < 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0) return 0;
  const int P = resolve_partition(num_seqs, num_heads, max_context_len, partition_size);
  if (P < pa::kChunk || P > pa::kMaxPartition || P % pa::kChunk != 0) return 0;
  const int max_parts = decode_max_parts(max_context_len, P);
  if (max_parts >= kMaxPartsPerSeq) return 0;
  return ws_layout(num_seqs, num_heads, head_dim, max_parts).total;
}

int pa_decode(void* out, int out_dtype, const void* q, const void* k_pool, const void* v_pool,
              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens, int max_context_len,
              int num_seqs, int num_heads, int head_dim, int block_size, int num_blocks, float scale, int dtype,
              void* workspace, size_t workspace_bytes, int partition_size, int32_t* err_flag, void* stream) {
  pa_host::Range range("pa_decode");
  pa::DecodeArgs a;
  bool empty = false;
  int st = decode_setup(out, out_dtype, q, k_pool, v_pool, block_tables, max_blocks_per_seq, context_lens,
                        max_context_len, num_seqs, num_heads, head_dim, block_size, num_blocks, scale, dtype, workspace,
                        workspace_bytes, partition_size, err_flag, a, empty);
  if (st != PA_OK || empty) return st;
  if (pa_host::debug_checks()) {
    int64_t bad[2];
    st = pa_host::check_decode_inputs(block_tables, max_blocks_per_seq, context_lens, num_seqs, max_context_len,
                                      block_size, num_blocks, stream, bad);
    if (st != PA_OK) {
      std::fprintf(stderr, "pa_decode (PA_DEBUG): sequence %lld, logical block %lld is invalid\n", (long long)bad[0],
                   (long long)bad[1]);
      return st;
    }
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (head_dim == 128) {
    return dtype == PA_F16 ? launch_decode<128, __half>(a, s) : launch_decode<128, __nv_bfloat16>(a, s);
  }
  return dtype == PA_F16 ? launch_decode<64, __half>(a, s) : launch_decode<64, __nv_bfloat16>(a, s);
}

size_t pa_decode_grouped_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                         int partition_size) {
  if (num_seqs < 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0) return 0;
  const int P = resolve_partition(num_seqs, num_heads, max_context_len, partition_size);
  if (P < pa::kChunk || P > pa::kMaxPartition || P % pa::kChunk != 0) return 0;
  const int max_parts = decode_max_parts(max_context_len, P);
  if (max_parts + 1 >= kMaxPartsPerSeq) return 0;
  return grouped_layout(num_seqs, num_heads, head_dim, max_parts).total;
}

// pa_decode_grouped: pa_decode for a batch in which groups of sequences share
// a prompt's blocks (parallel sampling and beam search, [summary] section 6,
// Figures 9-10, and [blog] "Prefix Sharing"): the planning kernel (which
// validates the groups and lists every sequence's own tokens as items), then
// the group kernel, which reads each shared prefix once for its whole group
// and streams the items too.
int pa_decode_grouped(void* out, int out_dtype, const void* q, const void* k_pool, const void* v_pool,
                      const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                      int max_context_len, int num_seqs, int num_heads, int head_dim, int block_size,
                      int num_blocks, float scale, int dtype, const int32_t* group_start,
                      const int32_t* group_prefix, int num_groups, void* workspace, size_t workspace_bytes,
                      int partition_size, int32_t* err_flag, void* stream) {
  pa_host::Range range("pa_decode_grouped");
  if (num_groups < 0 || (num_groups > 0 && (group_start == nullptr || group_prefix == nullptr)))
    return PA_ERR_INVALID_ARG;
  pa::DecodeArgs a;
  bool empty = false;
  int st = decode_setup(out, out_dtype, q, k_pool, v_pool, block_tables, max_blocks_per_seq, context_lens,
                        max_context_len, num_seqs, num_heads, head_dim, block_size, num_blocks, scale, dtype, workspace,
                        workspace_bytes, partition_size, err_flag, a, empty);
  if (st != PA_OK || empty) return st;
  const int prefix_parts = a.max_parts;  // a group's prefix is at most max_context_len tokens
  if (prefix_parts + 1 >= kMaxPartsPerSeq) return PA_ERR_UNSUPPORTED;
  // the group kernel counts its units (prefix units, then items x heads) in an int
  if ((long long)num_groups * num_heads * prefix_parts + (long long)num_seqs * (prefix_parts + 1) * num_heads >=
      (1ll << 31))
    return PA_ERR_UNSUPPORTED;
  const GroupedLayout gl = grouped_layout(num_seqs, num_heads, head_dim, a.max_parts);
  if (workspace_bytes < gl.total) return PA_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  a.max_parts += 1;
  a.counters = reinterpret_cast<int*>(ws + gl.base.counters);
  a.items = reinterpret_cast<int4*>(ws + gl.base.items);
  a.part_ml = reinterpret_cast<float2*>(ws + gl.base.ml);
  a.part_o = reinterpret_cast<float*>(ws + gl.base.o);
  a.num_groups = num_groups;
  a.group_start = group_start;
  a.group_prefix = group_prefix;
  a.seq_prefix = reinterpret_cast<int32_t*>(ws + gl.seq_prefix);
  if (pa_host::debug_checks()) {
    int64_t bad[2];
    st = pa_host::check_decode_inputs(block_tables, max_blocks_per_seq, context_lens, num_seqs, max_context_len,
                                      block_size, num_blocks, stream, bad);
    if (st != PA_OK) {
      std::fprintf(stderr, "pa_decode_grouped (PA_DEBUG): sequence %lld, logical block %lld is invalid\n",
                   (long long)bad[0], (long long)bad[1]);
      return st;
    }
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (num_groups == 0) {
    return head_dim == 128
               ? (dtype == PA_F16 ? launch_decode<128, __half>(a, s) : launch_decode<128, __nv_bfloat16>(a, s))
               : (dtype == PA_F16 ? launch_decode<64, __half>(a, s) : launch_decode<64, __nv_bfloat16>(a, s));
  }
  const uint64_t pool_rows = (uint64_t)num_blocks * num_heads * block_size;
  if (pool_rows >= (1ull << 31)) return PA_ERR_INVALID_ARG;
  CUtensorMap tk, tv;
  st = encode_pool_map(&tk, k_pool, dtype, head_dim, pool_rows);
  if (st == PA_OK) st = encode_pool_map(&tv, v_pool, dtype, head_dim, pool_rows);
  if (st != PA_OK) return st;
  st = configure_any(head_dim, dtype);
  if (st != PA_OK) return st;
  st = head_dim == 128 ? launch_plan<128>(a, s) : launch_plan<64>(a, s);
  if (st != PA_OK) return st;
  return head_dim == 128 ? (dtype == PA_F16 ? launch_group<128, __half>(a, tk, tv, prefix_parts, s)
                                            : launch_group<128, __nv_bfloat16>(a, tk, tv, prefix_parts, s))
                         : (dtype == PA_F16 ? launch_group<64, __half>(a, tk, tv, prefix_parts, s)
                                            : launch_group<64, __nv_bfloat16>(a, tk, tv, prefix_parts, s));
}

// pa_mixed_step: one step of a batch that mixes decode sequences and prefill
// chunks, the two parts running at the same time.  The continuous-batching
// page ("연속 배치 처리 아키텍처", "Chunked prefill" and the scheduler) fills a
// step's token budget with decode tokens and prefill chunks and runs them as
// one forward pass.  The decode streams K/V from HBM with CUDA-core
// arithmetic; the prefill is bound by the tensor cores; so they overlap:
// the planning kernel runs first, then the prefill's persistent grid, capped
// to a share of the SMs, then the decode kernel as a programmatic dependent
// of the prefill.  Every prefill CTA releases its dependents as it starts,
// so the decode grid fills the SMs the prefill left free; the decode skips
// its wait on the planning kernel, which completed before the prefill began.
int pa_mixed_step(void* dec_out, int dec_out_dtype, const void* dec_q, const int32_t* dec_block_tables,
                  int dec_max_blocks_per_seq, const int32_t* context_lens, int max_context_len, int num_seqs,
                  void* workspace, size_t workspace_bytes, void* pf_out, int pf_out_dtype, const void* pf_q,
                  const int32_t* cu_q_lens, const int32_t* ctx_before, const int32_t* pf_block_tables,
                  int pf_max_blocks_per_seq, int num_chunks, int total_q, int max_q_len, const void* k_pool,
                  const void* v_pool, int num_heads, int head_dim, int block_size, int num_blocks, float scale,
                  int dtype, int prefill_sms, int32_t* err_flag, void* stream) {
  pa_host::Range range("pa_mixed_step");
  pa::DecodeArgs a;
  bool dec_empty = false;
  int st = decode_setup(dec_out, dec_out_dtype, dec_q, k_pool, v_pool, dec_block_tables, dec_max_blocks_per_seq,
                        context_lens, max_context_len, num_seqs, num_heads, head_dim, block_size, num_blocks, scale,
                        dtype, workspace, workspace_bytes, 0, err_flag, a, dec_empty);
  if (st != PA_OK) return st;
  st = pa_host::prefill_check(pf_out, pf_out_dtype, pf_q, cu_q_lens, ctx_before, k_pool, v_pool, pf_block_tables,
                              pf_max_blocks_per_seq, num_chunks, total_q, max_q_len, num_heads, head_dim, block_size,
                              num_blocks, scale, dtype, err_flag);
  if (st != PA_OK) return st;
  const bool pf_empty = num_chunks == 0 || total_q == 0 || max_q_len == 0;
  if (pa_host::debug_checks() && !dec_empty) {
    int64_t bad[2];
    st = pa_host::check_decode_inputs(dec_block_tables, dec_max_blocks_per_seq, context_lens, num_seqs,
                                      max_context_len, block_size, num_blocks, stream, bad);
    if (st != PA_OK) {
      std::fprintf(stderr, "pa_mixed_step (PA_DEBUG): sequence %lld, logical block %lld is invalid\n",
                   (long long)bad[0], (long long)bad[1]);
      return st;
    }
  }
  if (pa_host::debug_checks() && !pf_empty) {
    int64_t bad[2];
    st = pa_host::check_prefill_inputs(cu_q_lens, ctx_before, pf_block_tables, pf_max_blocks_per_seq, num_chunks,
                                       total_q, max_q_len, block_size, num_blocks, stream, bad);
    if (st != PA_OK) {
      std::fprintf(stderr, "pa_mixed_step (PA_DEBUG): chunk %lld, logical block %lld is invalid\n",
                   (long long)bad[0], (long long)bad[1]);
      return st;
    }
  }
  const int sms = pa_host::device_sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  int cap = prefill_sms > 0 ? (prefill_sms < sms ? prefill_sms : sms) : (sms * PA_MIXED_PREFILL_SHARE + 50) / 100;
  if (cap < 1) cap = 1;
  auto prefill = [&](int ctas, int head_group) {
    return pa_host::prefill_launch(pf_out, pf_out_dtype, pf_q, cu_q_lens, ctx_before, k_pool, v_pool,
                                   pf_block_tables, pf_max_blocks_per_seq, num_chunks, total_q, max_q_len,
                                   num_heads, head_dim, block_size, num_blocks, scale, dtype, err_flag, ctas,
                                   head_group, stream);
  };
  if (dec_empty) return pf_empty ? PA_OK : prefill(0, 0);
  cudaStream_t s = (cudaStream_t)stream;
  if (pf_empty) {
    return head_dim == 128
               ? (dtype == PA_F16 ? launch_decode<128, __half>(a, s) : launch_decode<128, __nv_bfloat16>(a, s))
               : (dtype == PA_F16 ? launch_decode<64, __half>(a, s) : launch_decode<64, __nv_bfloat16>(a, s));
  }
  st = configure_any(head_dim, dtype);
  if (st != PA_OK) return st;
  st = head_dim == 128 ? launch_plan<128>(a, s) : launch_plan<64>(a, s);
  if (st != PA_OK) return st;
  // Beside the decode, which streams its K/V through L2 at several TB/s, a
  // line survives in L2 for only some tens of microseconds.  The prefill
  // therefore deals its heads one at a time: every query tile of a (chunk,
  // head) lands in the same round, on neighbouring CTAs, and they read that
  // head's K/V together instead of once per round from HBM.
  st = prefill(cap, 1);
  if (st != PA_OK) return st;
  a.dep_wait = 0;
  return launch_main_any(a, head_dim, dtype, s);
}

}  // extern "C"

// ---------------------------------------------------------------------------------
// pa_decode_static_scratch: pa_decode for callers that cannot allocate device
// memory.  Its scratch is this fixed array, resident on every device that
// loads the library; the host looks its address up once per device.
static __device__ __align__(256) unsigned char g_decode_static_scratch[PA_DECODE_STATIC_SCRATCH_BYTES];

namespace {
std::mutex g_static_scratch_mutex;
void* g_static_scratch_addr[64] = {nullptr};
}  // namespace

extern "C" int pa_decode_static_scratch(void* out, int out_dtype, const void* q, const void* k_pool,
                                        const void* v_pool, const int32_t* block_tables, int max_blocks_per_seq,
                                        const int32_t* context_lens, int max_context_len, int num_seqs,
                                        int num_heads, int head_dim, int block_size, int num_blocks, float scale,
                                        int dtype, int partition_size, int32_t* err_flag, void* stream) {
  pa_host::Range range("pa_decode_static_scratch");
  const size_t need = pa_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, partition_size);
  if (need > (size_t)PA_DECODE_STATIC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_static_scratch_mutex);
    if (g_static_scratch_addr[dev] == nullptr) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_decode_static_scratch) != cudaSuccess || addr == nullptr) return PA_ERR_CUDA;
      g_static_scratch_addr[dev] = addr;
    }
    scratch = g_static_scratch_addr[dev];
  }
  return pa_decode(out, out_dtype, q, k_pool, v_pool, block_tables, max_blocks_per_seq, context_lens,
                   max_context_len, num_seqs, num_heads, head_dim, block_size, num_blocks, scale, dtype, scratch,
                   (size_t)PA_DECODE_STATIC_SCRATCH_BYTES, partition_size, err_flag, stream);
}
