// Chunked-prefill attention over paged K/V on the sm_103a tensor cores.
//
// Method: the continuous-batching page ("연속 배치 처리 아키텍처", section
// "Chunked prefill") splits a long prompt into chunks that run over several
// steps; each chunk's queries attend causally (the j <= i of the section 4
// equation of the PagedAttention paper summary) to the sequence's paged K/V,
// which already holds every earlier token and the chunk's own tokens.
//
// Design (ours, for one GB300):
//  * Persistent: one CTA per SM (its shared and tensor memory allow one),
//    each walking a list of items -- (128-query tile, chunk, head) -- in
//    longest-first order, 10 warps:
//      warp 9  (loader)  walks the item list and publishes each runnable
//              item (its chunk, head, rows, context, key-tile count and
//              whether every block-table entry it reads is in range) in a
//              4-slot shared-memory ring that the other roles read, so that
//              they do no lookups of their own between items;
//              TMA: per item the query tile (3-D tensor map over
//              [token][head][dim]) once the previous item's last S = Q K^T is
//              done with the buffer; per 128-key tile the K rows and the V
//              rows of its pages into 2- and 3-stage rings (2-D tensor maps
//              over the pool seen as [block*H*B + slot][dim]), one lane per
//              page piece issuing that piece's copies, its table entry read a
//              tile ahead; pages outside the table are read at an
//              out-of-range row, which the TMA fills with zeros;
//      warp 8  (MMA)     one thread issues tcgen05.mma (kind::f16, M = N = 128,
//              K = 16, fp32 accumulators in tensor memory): S(j) = Q K_j^T
//              into one of two score buffers, and for each half h of the key
//              tile O_h += P_h(j) V_h(j), with P_h(j) read back from the same
//              buffer (A operand in tensor memory), into one of two output
//              accumulators;
//      warps 0-7 (softmax) two threads per query row (TMEM lane): warp w
//              owns keys 64*(w/4) .. +63 of every key tile for the rows of
//              lane quarter w%4, with its own running max, sum and output
//              accumulator O_(w/4), so the two halves of a row never wait for
//              each other; they merge by log-sum-exp once, at the end of the
//              item.  Each thread reads its 64 scores with one tcgen05.ld,
//              masks (only tiles on the diagonal, at the context end or with a
//              bad page), runs the online softmax (running max in raw score
//              units, exponents (s - m) * scale * log2 e, so the maximum's
//              weight is exactly 1), and writes P over its own 64 score
//              columns with tcgen05.st.  In a bf16 pool P is two bf16 parts,
//              P = P_hi + P_lo (upper 16 bits of P and of the remainder), so
//              that O_h += P_hi V + P_lo V carries ~16 bits of P: a single
//              bf16 P carries 8 bits, and its rounding alone moves a peaked
//              row's output by ~2^-9 |v|.  In an fp16 pool P is one fp16
//              value (11 bits, kept at 2^7 x the numerator) and one product
//              O_h += P V, the row sum adding the rounded values.
//    The MMA thread issues S(0), S(1), then per key tile j: P_0(j) V, P_1(j)
//    V (two parts each in a bf16 pool), S(j+2): the score buffer of tile j+1
//    is ready while the softmax of tile j runs.  An output accumulator is rescaled lazily (only when its
//    half-row max grew by more than 2^8: it is read, scaled and written back
//    in tensor memory); only then does the softmax of tile j wait for
//    P_h(j-1) V, otherwise it overlaps it.  Ring stages and barrier phases
//    follow running per-CTA counters, so the next item's query load and first
//    two S products overlap the current item's last tiles and epilogue.  The
//    output leaves through a 2 KB shared-memory slab per softmax warp, so
//    that a store instruction writes 8 rows' 64-byte pieces.
//  * Operands in shared memory are 128-byte swizzled: K-major for Q and K;
//    V is consumed MN-major (dims contiguous), straight from the pool layout.
//  * Keys past the context or in a bad page, and keys past a query's
//    position, are masked; V rows past the context are zeroed in shared
//    memory before the product, so pool bits past a sequence's end (even NaN)
//    cannot reach the output.
//  * Work order: every CTA ranks the (chunk, query tile) pairs by their
//    key-tile count; the items (pairs times heads) are dealt to the CTAs in
//    that order, forward and backward in alternate rounds.
#include <cudaTypedefs.h>
#include <math.h>

#include <atomic>
#include <cstdio>
#include <mutex>
#include <type_traits>

#include "pa_common.cuh"

namespace pa {

constexpr int kPfRows = 128;   // query rows per tile (MMA M)
constexpr int kPfKeys = 128;   // keys per tile (N of S = Q K^T, K of O += P V)
constexpr int kPfThreads = 320;
constexpr int kPfMmaWarp = 8;
constexpr int kPfLoadWarp = 9;
constexpr int kKStages = 2;
constexpr int kVStages = 3;
constexpr uint32_t kHalfBytes = kPfRows * 64 * 2;  // 128 rows x 64 columns x 2 bytes
constexpr uint32_t kTileBytes = 2 * kHalfBytes;     // one 128 x 128 16-bit tile
constexpr float kRescaleThreshold = 8.0f;           // log2 units
// An fp16 pool's P is one fp16 value kept at 2^7 times the softmax
// numerator: with the lazy rescale its largest value is 2^(8+7), inside the
// fp16 range, and weights down to 2^-21 of the row maximum keep full fp16
// precision (the scale cancels in the final division by the row sum).
constexpr float kPScaleLog2 = 7.0f;
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns: two score buffers (later P) and the two half-row outputs
__device__ __forceinline__ uint32_t tmem_s(int b) { return b ? 128u : 0u; }
__device__ __forceinline__ uint32_t tmem_o(int h) { return h ? 384u : 256u; }

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;             // kKStages stages
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;  // kVStages stages
// Output staging: 2 KB per softmax warp, 32 rows x 64 bytes, so that a warp
// stores whole 64-byte row pieces instead of one 16-byte piece per row.
constexpr uint32_t kStageBytes = 32 * 64;
constexpr uint32_t kOffStage = kOffV + kVStages * kTileBytes;
constexpr uint32_t kOffBar = kOffStage + 8 * kStageBytes;
constexpr int kPfRankMax = 1024;  // (chunk, query tile) pairs ranked in-kernel

// An item as the loader publishes it to the MMA thread and the softmax warps.
// The loader fills slot k % kItemSlots for its k-th runnable item after it has
// issued V of the previous item's last key tile, which waits for the P V
// product three tiles back; the softmax warps (and, ahead of them, the MMA
// thread) copy a slot when they start its item, before any of the item's P.
// Three tiles back lie at most three items back, so four slots are never
// overwritten before they are read.
constexpr int kItemSlots = 4;
enum { kSlotNeedZero = 1, kSlotTableOk = 2, kSlotEnd = 4 };
struct PfSlot {
  int c, h, q0, n_c, row0, c0, ctx_total, n_kv;
  int flags;  // kSlotNeedZero: the last key tile runs past the context; kSlotTableOk: every table
              // entry the item reads is in range; kSlotEnd: no more items
};

struct PfBars {
  uint64_t item_full[kItemSlots];  // the loader wrote the slot, one phase per use
  uint64_t q_full, q_empty;  // query tile loaded / its last S = Q K^T done
  uint64_t k_full[kKStages];  // (a K stage is free again when its S = Q K^T is done: s_full)
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2];      // per score buffer; also frees K stage x % 2 (kKStages == 2)
  uint64_t p_full[2][2];   // [half][buffer]: every row wrote P_h(j), buffer j % 2, one phase per use
  uint64_t pv_done[2];     // both halves' P(j) V complete, barrier j % 2, one phase per use
  uint64_t v_zeroed;       // V rows past the context zeroed (last key tile)
  uint64_t xbar[4];        // per lane quarter: both halves' (max, sum) written (end of an item)
  uint64_t o_free;         // every softmax warp has read the output accumulators (end of an item)
  uint64_t drain;
  uint32_t tmem_base;
  float xm[2][kPfRows];  // half-row running max (raw score) at the end: [half][row]
  float xl[2][kPfRows];  // half-row sum at the end: [half][row]
  int abort_flag;
  uint16_t order[kPfRankMax];  // (chunk, query tile) pairs, longest first
  PfSlot items[kItemSlots];
};
constexpr uint32_t kPfSmemBytes = kOffBar + sizeof(PfBars) + 1024;  // + alignment slack
static_assert(kPfSmemBytes <= 227 * 1024, "shared memory beyond the per-CTA limit");
static_assert(kKStages == 2, "s_full[x & 1] frees K stage x % kKStages");

struct PrefillArgs {
  void* out;
  int out_dtype;
  const int32_t* cu_q_lens;
  const int32_t* ctx_before;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  int num_heads;
  int block_size;
  int num_blocks;
  int rows_per_load;  // gcd(block_size, 128): a piece of that many keys never straddles a page
  int rpl_shift;      // log2(rows_per_load)
  int pool_rows;      // num_blocks * H * B: any row at or past it reads zeros
  int num_chunks;
  int qtiles;         // query tiles per chunk in the grid: ceil(max_q_len / 128)
  int head_group;     // heads dealt together (num_heads: one group)
  float qscale;       // scale * log2(e)
  uint32_t idesc_s;   // instruction descriptors
  uint32_t idesc_pv;
  int32_t* err_flag;
};

// ---- tcgen05 / TMA helpers ------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // version
  d |= (uint64_t)2 << 61;  // SWIZZLE_128B
  return d;
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.  The load and its
// wait sit in one asm statement, so no use of the registers can be scheduled
// before the data has arrived.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 2^x by the hardware's approximate base-2 exponential (relative error
// below 2^-22; 2^-inf = +0), flushing subnormal results to zero.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
      "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
      "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
      "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
      "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Two fp32 values as one 64-bit pair, and back.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack_f32x2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// max(a, b, c) in one instruction (an operand that is NaN is ignored, as in fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (a - m) * q and (b - m) * q with the packed fp32-pair instructions: one
// subtraction and one multiplication per two values.  mm = (m, m), qq = (q, q).
__device__ __forceinline__ float2 sub_mul_f32x2(float a, float b, uint64_t mm, uint64_t qq) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack_f32x2(a, b)), "l"(mm));
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(d) : "l"(qq));
  return unpack_f32x2(d);
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// (x, y) as two packed bf16 pairs, hi + lo carrying ~16 significant bits.
// bf16 is the upper half of an fp32: hi keeps the upper 16 bits of x and y
// (truncation), the remainder x - hi is exact in fp32 and is truncated the
// same way.  hi + lo is within 2^-15 of x relative; no conversion
// instructions, only bit selects and one packed subtraction.
__device__ __forceinline__ void split2_bf16(float x, float y, uint32_t& hi, uint32_t& lo) {
  const uint32_t xb = __float_as_uint(x), yb = __float_as_uint(y);
  const float2 r = unpack_f32x2(sub_f32x2(pack_f32x2(x, y), pack_f32x2(__uint_as_float(xb & 0xffff0000u),
                                                                          __uint_as_float(yb & 0xffff0000u))));
  hi = __byte_perm(xb, yb, 0x7632);
  lo = __byte_perm(__float_as_uint(r.x), __float_as_uint(r.y), 0x7632);
}

// tcgen05.mma with A read from tensor memory (the "TS" form): D += A B.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}


// 64 consecutive fp32 columns of this thread's TMEM lane, load and wait in one
// asm statement.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// One unit of work: a 128-row query tile of one chunk, for one head.
struct PfItem {
  int c, h;         // chunk, head
  int q0, n_c;      // chunk's first row in q / out, its query count
  int row0, rows;   // tile's first query row within the chunk, rows in the tile
  int c0, ctx_total;
  int n_kv;         // key tiles the tile's queries see
  bool need_zero;   // the last key tile runs past the context
};

enum { kItemRun = 0, kItemEmpty = 1, kItemBadLength = 2 };

// Item at position `pos` of the list.  The heads are dealt in groups of
// a.head_group: within a group the list is the (chunk, query tile) pairs in
// `order` (or, past kPfRankMax pairs, later query tiles first), each expanded
// over the group's heads, so that while a group runs, the CTAs read the K/V of
// its heads only.  Odd groups take the pairs in reverse (shortest first), so
// that the rounds dealt forward and backward over the CTAs stay balanced
// across group boundaries; one group (every head) is plain longest-first.
__device__ __forceinline__ int pf_item(const PrefillArgs& a, const uint16_t* order, int npairs, int pos, PfItem& it) {
  const int H = a.num_heads;
  const int G = a.head_group;
  const int per_group = npairs * G;  // positions of a full group (fits int: the host bounds npairs * H)
  const int gi = pos / per_group;
  const int within = pos - gi * per_group;
  const int h0 = gi * G;
  const int gsz = min(G, H - h0);  // the last group may hold fewer heads
  int rank = within / gsz;
  it.h = h0 + within - rank * gsz;
  if (gi & 1) rank = npairs - 1 - rank;
  int c, qt;
  if (npairs <= kPfRankMax) {
    const int pair = order[rank];
    c = pair / a.qtiles;
    qt = pair - c * a.qtiles;
  } else {
    const int from_end = rank / a.num_chunks;
    c = rank - from_end * a.num_chunks;
    qt = a.qtiles - 1 - from_end;
  }
  it.c = c;
  it.q0 = __ldg(a.cu_q_lens + c);
  it.n_c = __ldg(a.cu_q_lens + c + 1) - it.q0;
  it.row0 = qt * kPfRows;
  if (it.row0 >= it.n_c) return kItemEmpty;
  it.c0 = __ldg(a.ctx_before + c);
  // the context must fit the table and keep key positions well inside int32
  const int64_t total = (int64_t)it.c0 + it.n_c;
  if (it.c0 < 0 || total > (int64_t)a.max_blocks_per_seq * a.block_size || total > INT32_MAX - 2 * kPfKeys)
    return kItemBadLength;
  it.ctx_total = (int)total;
  it.rows = min(kPfRows, it.n_c - it.row0);
  it.n_kv = (it.c0 + it.row0 + it.rows - 1) / kPfKeys + 1;
  it.need_zero = it.n_kv * kPfKeys > it.ctx_total;
  return kItemRun;
}

// Position of this CTA's round-r item in the longest-first list: rounds go
// forward and backward over the CTAs in turn (CTA b takes b, 2G-1-b, 2G+b,
// ...), so the CTA that drew the shortest item of one round draws the longest
// of the next.
__device__ __forceinline__ long long pf_round_pos(int r) {
  const int G = gridDim.x, b = blockIdx.x;
  return (long long)r * G + ((r & 1) ? (G - 1 - b) : b);
}

// D = head_dim, 64 or 128: tiles are D / 64 swizzled 64-column halves.
template <typename T, int D>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  constexpr int kHalves = D / 64;
  constexpr uint32_t kLoadBytes = kHalves * kHalfBytes;  // bytes of one loaded Q, K or V tile
  // P V as P_hi V + P_lo V in bf16 (bf16 pool: 8-bit P alone is not accurate
  // enough), or as one product with an fp16 P (fp16 pool: 11 bits are)
  constexpr int kPParts = std::is_same<T, __nv_bfloat16>::value ? 2 : 1;
  // a kernel launched behind this one as a programmatic dependent may start
  // as soon as every CTA is resident (pa_mixed_step's decode); it must not
  // read this kernel's output without waiting for it
  griddep_launch_dependents();
  extern __shared__ uint8_t pf_smem_raw[];
  const uint32_t raw = smem_u32(pf_smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = pf_smem_raw + (base - raw);
  PfBars& bars = *reinterpret_cast<PfBars*>(gbase + kOffBar);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = a.num_heads;
  const int B = a.block_size;
  const int npairs = a.num_chunks * a.qtiles;
  const long long n_items = (long long)npairs * H;

  // ---- rank the (chunk, query tile) pairs by key-tile count, longest first
  if (npairs <= kPfRankMax) {
    int* cost = reinterpret_cast<int*>(gbase + kOffV);  // scratch, before any V tile is loaded
    for (int e = threadIdx.x; e < npairs; e += blockDim.x) {
      const int cc = e / a.qtiles, tt = e - cc * a.qtiles;
      const int nq = __ldg(a.cu_q_lens + cc + 1) - __ldg(a.cu_q_lens + cc);
      const int last = min(tt * kPfRows + kPfRows - 1, nq - 1);
      cost[e] = tt * kPfRows < nq ? (__ldg(a.ctx_before + cc) + last) / kPfKeys + 1 : 0;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < npairs; e += blockDim.x) {
      const int ke = cost[e];
      int rank = 0;
      for (int f = 0; f < npairs; ++f) rank += (cost[f] > ke) || (cost[f] == ke && f < e);
      bars.order[rank] = (uint16_t)e;
    }
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < kItemSlots; ++i) mbar_init(&bars.item_full[i], 1);
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_empty, 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&bars.k_full[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
    }
    mbar_init(&bars.s_full[0], 1);
    mbar_init(&bars.s_full[1], 1);
    mbar_init(&bars.pv_done[0], 1);
    mbar_init(&bars.pv_done[1], 1);
    for (int hh = 0; hh < 2; ++hh) {
      mbar_init(&bars.p_full[hh][0], 4);
      mbar_init(&bars.p_full[hh][1], 4);
    }
    mbar_init(&bars.v_zeroed, 4);
    mbar_init(&bars.o_free, 8);
    for (int q = 0; q < 4; ++q) mbar_init(&bars.xbar[q], 2);
    mbar_init(&bars.drain, 1);
    bars.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort_flag = &bars.abort_flag;
  const uint16_t* order = bars.order;

  // The loader walks this CTA's items and publishes each runnable one; the
  // MMA thread and the softmax warps take them from the item ring in the same
  // order.  Ring stages and barrier phases follow running counters: g = key
  // tiles of this CTA's earlier items (the global index of a key tile is
  // g + t), k = items run so far.
  if (warp == kPfLoadWarp) {
    // ---------------------------------------------------------------- loader
    const int rpl = a.rows_per_load;
    const int loads = kPfKeys / rpl;  // page pieces per key tile (1..8)
    int g = 0, k = 0, k_issued = 0, v_issued = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const long long ipos = pf_round_pos(r);
      if (ipos >= n_items) break;
      PfItem it;
      const int st = pf_item(a, order, npairs, (int)ipos, it);
      if (st == kItemBadLength && lane == 0) atomicOr(a.err_flag, PA_FLAG_BAD_LENGTH);
      if (st != kItemRun) continue;
      const int32_t* trow = a.block_tables + (size_t)it.c * a.max_blocks_per_seq;
      {  // publish the item, with whether every table entry it reads is in range
        const int kend = min(it.ctx_total, it.n_kv * kPfKeys);
        const int npages = (kend + B - 1) / B;
        bool bad = false;
#pragma unroll 4
        for (int p = lane; p < npages; p += 32) {
          const int32_t e = __ldg(trow + p);
          bad |= (e < 0 || e >= a.num_blocks);
        }
        const bool table_ok = !__any_sync(0xffffffffu, bad);
        if (lane == 0) {
          PfSlot& sl = bars.items[k % kItemSlots];
          sl.c = it.c;
          sl.h = it.h;
          sl.q0 = it.q0;
          sl.n_c = it.n_c;
          sl.row0 = it.row0;
          sl.c0 = it.c0;
          sl.ctx_total = it.ctx_total;
          sl.n_kv = it.n_kv;
          sl.flags = (it.need_zero ? kSlotNeedZero : 0) | (table_ok ? kSlotTableOk : 0);
          mbar_arrive(&bars.item_full[k % kItemSlots]);
        }
      }
      int wok = 1;
      if (lane == 0) {  // the query tile, once the previous item's last S = Q K^T is done with the buffer
        wok = mbar_wait(&bars.q_empty, (k & 1) ^ 1, abort_flag, a.err_flag);
        if (wok) {
          mbar_arrive_expect_tx(&bars.q_full, kLoadBytes);
          for (int hf = 0; hf < kHalves; ++hf)
            tma_load_3d(base + kOffQ + hf * kHalfBytes, &tm_q, hf * 64, it.h, it.q0 + it.row0, &bars.q_full);
        }
      }
      if (!__shfl_sync(0xffffffffu, wok, 0)) break;
      // Lane i < loads owns page piece i of every key tile: it looks up the
      // piece's table entry one tile ahead and issues the piece's copies
      // itself, so the pieces of a tile go out in parallel.
      const bool owner = lane < loads;
      auto fetch = [&](int t) -> int32_t {  // table entry of this lane's piece of tile t; -2: past the context
        const int pos = t * kPfKeys + lane * rpl;
        return (owner && t < it.n_kv && pos < it.ctx_total) ? __ldg(trow + pos / B) : -2;
      };
      int32_t entry = fetch(0);
      int prev_row = a.pool_rows;  // this lane's page row of the previous key tile (its V is loaded one step later)
      for (int t = 0; t <= it.n_kv; ++t) {
        int row = a.pool_rows;  // out of range: the TMA fills zeros
        if (entry != -2) {
          const int pos = t * kPfKeys + lane * rpl;
          if (entry >= 0 && entry < a.num_blocks) {
            row = (entry * H + it.h) * B + pos % B;
          } else {
            atomicOr(a.err_flag, PA_FLAG_BAD_BLOCK);
          }
        }
        entry = fetch(t + 1);
        int wk = 1;
        if (t < it.n_kv) {  // K of tile t
          const int x = g + t;
          const int stg = x % kKStages;
          // stage x % 2 held K(x-2): free once S(x-2) is done, the previous phase of s_full[x & 1]
          if (lane == 0) wk = mbar_wait(&bars.s_full[stg], ((x / kKStages) & 1) ^ 1, abort_flag, a.err_flag);
          if (!__shfl_sync(0xffffffffu, wk, 0)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&bars.k_full[stg], kLoadBytes);
          __syncwarp();
          if (owner) {
            const uint32_t dst = base + kOffK + stg * kTileBytes + (uint32_t)lane * rpl * 128u;
            tma_load_2d(dst, &tm_k, 0, row, &bars.k_full[stg]);
            if (kHalves == 2) tma_load_2d(dst + kHalfBytes, &tm_k, 64, row, &bars.k_full[stg]);
          }
          ++k_issued;
        }
        if (t >= 1) {  // V of tile t - 1
          const int x = g + t - 1;
          const int stg = x % kVStages;
          if (lane == 0) wk = mbar_wait(&bars.v_empty[stg], ((x / kVStages) & 1) ^ 1, abort_flag, a.err_flag);
          if (!__shfl_sync(0xffffffffu, wk, 0)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&bars.v_full[stg], kLoadBytes);
          __syncwarp();
          if (owner) {
            const uint32_t dst = base + kOffV + stg * kTileBytes + (uint32_t)lane * rpl * 128u;
            tma_load_2d(dst, &tm_v, 0, prev_row, &bars.v_full[stg]);
            if (kHalves == 2) tma_load_2d(dst + kHalfBytes, &tm_v, 64, prev_row, &bars.v_full[stg]);
          }
          ++v_issued;
        }
        prev_row = row;
      }
      g += it.n_kv;
      ++k;
    }
    if (ok && lane == 0) {  // the end of the list
      bars.items[k % kItemSlots].flags = kSlotEnd;
      mbar_arrive(&bars.item_full[k % kItemSlots]);
    }
    if (lane == 0 && *abort_flag) {  // let in-flight copies land before exit
      if (k > 0) mbar_wait_drain(&bars.q_full, (k - 1) & 1);
      for (int x = max(0, k_issued - kKStages); x < k_issued; ++x)
        mbar_wait_drain(&bars.k_full[x % kKStages], (x / kKStages) & 1);
      for (int x = max(0, v_issued - kVStages); x < v_issued; ++x)
        mbar_wait_drain(&bars.v_full[x % kVStages], (x / kVStages) & 1);
    }
  } else if (warp == kPfMmaWarp) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint64_t qdesc = smem_desc_sw128(base + kOffQ, 16, 1024);
      int g = 0, nz = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        ok = mbar_wait(&bars.item_full[k % kItemSlots], (k / kItemSlots) & 1, abort_flag, a.err_flag);
        if (!ok) break;
        const int flags = bars.items[k % kItemSlots].flags;
        if (flags & kSlotEnd) break;
        const int n_kv = bars.items[k % kItemSlots].n_kv;
        const bool need_zero = (flags & kSlotNeedZero) != 0;
        ok = mbar_wait(&bars.q_full, k & 1, abort_flag, a.err_flag);
        if (!ok) break;
        // S(x) = Q K_x^T into score buffer x % 2; after the item's last one the query buffer is free
        auto issue_s = [&](int t) -> bool {
          const int x = g + t;
          if (!mbar_wait(&bars.k_full[x % kKStages], (x / kKStages) & 1, abort_flag, a.err_flag)) return false;
          tc_fence_after();
          // descriptors advance by adding (byte offset >> 4) to the start-address field
          const uint64_t kdesc = smem_desc_sw128(base + kOffK + (x % kKStages) * kTileBytes, 16, 1024);
          const uint32_t d = tmem + tmem_s(x & 1);
#pragma unroll
          for (int kk = 0; kk < 4 * kHalves; ++kk) {  // K = head_dim in steps of 16
            const uint32_t koff = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
            umma_f16(d, qdesc + koff, kdesc + koff, a.idesc_s, kk > 0);
          }
          umma_commit(&bars.s_full[x & 1]);  // the scores, and K stage x % 2 free again
          if (t == n_kv - 1) umma_commit(&bars.q_empty);
          return true;
        };
        ok = issue_s(0);
        if (ok && n_kv > 1) ok = issue_s(1);
        for (int t = 0; ok && t < n_kv; ++t) {
          const int x = g + t;
          ok = mbar_wait(&bars.v_full[x % kVStages], (x / kVStages) & 1, abort_flag, a.err_flag);
          if (ok && need_zero && t == n_kv - 1) ok = mbar_wait(&bars.v_zeroed, nz & 1, abort_flag, a.err_flag);
          // the previous item's epilogue has read both output accumulators
          if (ok && t == 0) ok = mbar_wait(&bars.o_free, (k & 1) ^ 1, abort_flag, a.err_flag);
          const uint64_t vdesc = smem_desc_sw128(base + kOffV + (x % kVStages) * kTileBytes, kHalfBytes, 1024);
          const uint32_t pb = tmem + tmem_s(x & 1);
          const uint32_t first = t > 0 ? 1u : 0u;
#pragma unroll
          for (int hh = 0; hh < 2 && ok; ++hh) {  // O_h += P_h V_h: keys 64h .. 64h+63 of the tile
            ok = mbar_wait(&bars.p_full[hh][x & 1], (x >> 1) & 1, abort_flag, a.err_flag);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int part = 0; part < kPParts; ++part) {  // P V, or P_hi V then P_lo V
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                umma_f16_ts(tmem + tmem_o(hh), pb + hh * 64 + part * 32 + kk * 8,
                            vdesc + (((hh * 4 + kk) * 2048) >> 4), a.idesc_pv, (kk > 0 || part > 0) ? 1u : first);
              }
            }
            if (hh == 1) umma_commit(&bars.pv_done[x & 1]);  // both halves' products (issued in order)
          }
          if (!ok) break;
          umma_commit(&bars.v_empty[x % kVStages]);
          if (t + 2 < n_kv) ok = issue_s(t + 2);  // after P(x) V in issue order: its buffer is free then
        }
        if (need_zero) ++nz;
        g += n_kv;
      }
      // every issued MMA has finished before tensor memory is released
      umma_commit(&bars.drain);
      mbar_wait_drain(&bars.drain, 0);
    }
  } else if (warp < 8) {
    // ---------------------------------------------------------------- softmax warps
    const int quarter = warp & 3;      // TMEM lane quarter this warp may access
    const int half = warp >> 2;        // columns 64*half .. 64*half+63
    const int r = quarter * 32 + lane; // query row within the tile = TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t full_mask = (1u << (kPfKeys / a.rows_per_load)) - 1u;
    const int col0 = half * 64;
    const uint32_t s_half = lane_addr + col0;  // + score buffer: this half's 64 columns
    const uint32_t o_mine = lane_addr + tmem_o(half);
    const int rpl = a.rows_per_load;
    const int pieces = kPfKeys / rpl;
    int g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      ok = mbar_wait(&bars.item_full[k % kItemSlots], (k / kItemSlots) & 1, abort_flag, a.err_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      PfItem it;
      bool all_ok;
      {
        const PfSlot& sl = bars.items[k % kItemSlots];
        if (sl.flags & kSlotEnd) break;
        it.c = sl.c;
        it.h = sl.h;
        it.q0 = sl.q0;
        it.n_c = sl.n_c;
        it.row0 = sl.row0;
        it.c0 = sl.c0;
        it.ctx_total = sl.ctx_total;
        it.n_kv = sl.n_kv;
        it.need_zero = (sl.flags & kSlotNeedZero) != 0;
        all_ok = (sl.flags & kSlotTableOk) != 0;
      }
      const int n_kv = it.n_kv;
      const int qrow = it.row0 + r;
      const int pos = it.c0 + qrow;
      const int tile_first_pos = it.c0 + it.row0;
      const int ctx_total = it.ctx_total;
      // Page pieces of a key tile whose table entry is usable: the loader
      // zero-fills the others and they are masked here.  Each lane < pieces
      // reads one table entry, one tile ahead so the load latency is hidden.
      const int32_t* trow = a.block_tables + (size_t)it.c * a.max_blocks_per_seq;
      auto piece_entry = [&](int t) -> int32_t {
        const int p = t * kPfKeys + lane * rpl;
        return (t < n_kv && lane < pieces && p < ctx_total) ? __ldg(trow + p / B) : -1;
      };
      // Every table entry the item reads in range (the loader checked): then
      // no key tile needs a per-piece mask and the per-tile lookups are skipped.
      int32_t entry_next = all_ok ? 0 : piece_entry(0);
      float m_used = -INFINITY;
      float l = 0.f;
      for (int t = 0; t < n_kv; ++t) {
        const int x = g + t;
        const int sb = x & 1;
        uint32_t kmask = full_mask;
        if (!all_ok) {
          kmask = __ballot_sync(0xffffffffu, entry_next >= 0 && entry_next < a.num_blocks);
          entry_next = piece_entry(t + 1);
        }
        ok = mbar_wait(&bars.s_full[sb], (x >> 1) & 1, abort_flag, a.err_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[64];
        tmem_ld64(s_half + tmem_s(sb), s);

        const int key0 = t * kPfKeys;
        const bool interior =
            key0 + kPfKeys - 1 <= tile_first_pos && key0 + kPfKeys <= ctx_total && kmask == full_mask;
        if (!interior) {
          const int lim = min(pos, ctx_total - 1) - key0;  // last admissible column of this row
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            const int col = col0 + i;
            const bool valid = col <= lim && ((kmask >> (col >> a.rpl_shift)) & 1u);
            s[i] = valid ? s[i] : -INFINITY;
          }
        }
        float mx4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
        for (int i = 4; i < 64; i += 2) mx4[(i >> 1) & 3] = fmax3(mx4[(i >> 1) & 3], s[i], s[i + 1]);
        // the running max is kept in raw score units, so that the exponent
        // (s - m) * qscale of the row's maximum is exactly 0 and its weight
        // exactly 1 (a rounded m * qscale would leave its rounding error there)
        const float rmax = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        const float m_new = fmaxf(m_used, rmax);
        // rescale when the max grew by more than 2^kRescaleThreshold (qscale > 0);
        // also true when m_used is -inf
        const bool resc = (m_new - m_used) * a.qscale > kRescaleThreshold;
        const float m_next = resc ? m_new : m_used;
        const float alpha = resc ? ((m_used == -INFINITY) ? 0.f : ex2_approx((m_used - m_next) * a.qscale)) : 1.f;
        l *= alpha;
        const float mref = (m_next == -INFINITY) ? 0.f : m_next;
        const uint64_t mm2 = pack_f32x2(mref, mref), qq2 = pack_f32x2(a.qscale, a.qscale);
        uint64_t sum2[2] = {0, 0};  // packed (even, odd) partial sums; 0 bits = (0.f, 0.f)
        uint32_t hw[32], lw[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float2 x2 = sub_mul_f32x2(s[2 * e], s[2 * e + 1], mm2, qq2);
          if (kPParts == 2) {
            const float p0 = ex2_approx(x2.x);
            const float p1 = ex2_approx(x2.y);
            sum2[e & 1] = add_f32x2(sum2[e & 1], pack_f32x2(p0, p1));
            split2_bf16(p0, p1, hw[e], lw[e]);
          } else {
            // fp16 P at 2^7 x the numerator; the row sum adds the rounded
            // values the product uses, so a weight's rounding moves the
            // output by at most 2^-11 w |v - o|
            const __half2 h2 = __floats2half2_rn(ex2_approx(x2.x + kPScaleLog2), ex2_approx(x2.y + kPScaleLog2));
            sum2[e & 1] = add_f32x2(sum2[e & 1], pack_f32x2(__low2float(h2), __high2float(h2)));
            hw[e] = *reinterpret_cast<const uint32_t*>(&h2);
          }
        }
        const float2 sa = unpack_f32x2(sum2[0]), sb2 = unpack_f32x2(sum2[1]);
        l += (sa.x + sa.y) + (sb2.x + sb2.y);
        // This half's columns of the buffer held P_h(x-2).  Its P V needs no
        // wait: S(x) was issued after it, and a commit tracks every earlier
        // MMA of the issuing thread, so S(x) complete means P_h(x-2) V is too.
        // A rescale of O_h also needs P_h(x-1) V (same item) in it.
        const bool any_resc = t > 0 && __any_sync(0xffffffffu, resc);
        if (any_resc)
          ok = mbar_wait(&bars.pv_done[(x - 1) & 1], ((x - 1) >> 1) & 1, abort_flag, a.err_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // P_h over this half's scores: P (or P_hi) in its first 32 words, P_lo in the next 32
        const uint32_t pw = s_half + tmem_s(sb);
        tmem_st16(pw, hw);
        tmem_st16(pw + 16, hw + 16);
        if (kPParts == 2) {
          tmem_st16(pw + 32, lw);
          tmem_st16(pw + 48, lw + 16);
        }
        if (any_resc) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            float o[32];
            tmem_ld32(o_mine + cc * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(o_mine + cc * 32, o);
          }
        }
        tmem_st_wait();
        if (half == 0 && it.need_zero && t == n_kv - 1) {
          // zero the V rows of this last key tile that lie past the context
          ok = mbar_wait(&bars.v_full[x % kVStages], (x / kVStages) & 1, abort_flag, a.err_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          if (key0 + r >= ctx_total) {
            uint8_t* vbuf = gbase + kOffV + (x % kVStages) * kTileBytes;
            const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              *reinterpret_cast<uint4*>(vbuf + r * 128 + ch * 16) = z;
              if (kHalves == 2) *reinterpret_cast<uint4*>(vbuf + kHalfBytes + r * 128 + ch * 16) = z;
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.v_zeroed);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full[half][sb]);
        m_used = m_next;
      }
      if (!ok) break;
      // ---- epilogue: merge the two half-rows (log-sum-exp), write this half's 64 output columns
      const int xl_ = g + n_kv - 1;  // the item's last key tile
      ok = mbar_wait(&bars.pv_done[xl_ & 1], (xl_ >> 1) & 1, abort_flag, a.err_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      bars.xm[half][r] = m_used;
      bars.xl[half][r] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.xbar[quarter]);
      ok = mbar_wait(&bars.xbar[quarter], k & 1, abort_flag, a.err_flag);
      // the partner's output must be complete too before its columns are read
      // (pv_done covers the partner half's product of the last tile too)
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float m0 = bars.xm[0][r], m1 = bars.xm[1][r];
      const float M = fmaxf(m0, m1);
      const float w0 = m0 == -INFINITY ? 0.f : ex2_approx((m0 - M) * a.qscale);
      const float w1 = m1 == -INFINITY ? 0.f : ex2_approx((m1 - M) * a.qscale);
      const float lt = w0 * bars.xl[0][r] + w1 * bars.xl[1][r];
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float c0w = w0 * inv, c1w = w1 * inv;
      // This warp's 32 rows x 64 output columns leave through its staging slab
      // in 64-byte row pieces: a thread writes its row's piece (16-byte unit j
      // at j ^ ((row >> 1) & 3), so that 8 consecutive rows cover all banks),
      // then four lanes per row store 8 rows at a time.
      const int ocol0 = half * (D / 2);  // this warp writes output columns ocol0 .. ocol0 + D/2 - 1
      uint8_t* stage = gbase + kOffStage + warp * kStageBytes;
      const int swz = (lane >> 1) & 3;
      const int prow = lane >> 2, pj = lane & 3;  // copy-out: row within a group of 8, 16-byte unit
      const bool f32_out = a.out_dtype == PA_F32;
      const int esize = f32_out ? 4 : 2;
      const int wrow0 = it.row0 + quarter * 32;  // this warp's first row within the chunk
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        float oa[32], ob[32];
        tmem_ld32(lane_addr + tmem_o(0) + ocol0 + cc * 32, oa);
        tmem_ld32(lane_addr + tmem_o(1) + ocol0 + cc * 32, ob);
        float o[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = c0w * oa[i] + c1w * ob[i];
#pragma unroll
        for (int ps = 0; ps < 2; ++ps) {  // 64-byte pieces: one for 16-bit outputs, two for fp32
          if (ps == 1 && !f32_out) break;
          uint4 v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (f32_out) {
              const float* f = o + 16 * ps + 4 * j;
              v[j] = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                                __float_as_uint(f[3]));
            } else {
              const float* f = o + 8 * j;
              if (a.out_dtype == PA_BF16) {
                v[j] = make_uint4(pack2<__nv_bfloat16>(f[0], f[1]), pack2<__nv_bfloat16>(f[2], f[3]),
                                  pack2<__nv_bfloat16>(f[4], f[5]), pack2<__nv_bfloat16>(f[6], f[7]));
              } else {
                v[j] = make_uint4(pack2<__half>(f[0], f[1]), pack2<__half>(f[2], f[3]), pack2<__half>(f[4], f[5]),
                                  pack2<__half>(f[6], f[7]));
              }
            }
            *reinterpret_cast<uint4*>(stage + lane * 64 + ((j ^ swz) << 4)) = v[j];
          }
          const int col = ocol0 + cc * 32 + (f32_out ? ps * 16 : 0);  // first output column of this piece
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int R = i * 8 + prow;
            const uint4 w = *reinterpret_cast<const uint4*>(stage + R * 64 + ((pj ^ ((R >> 1) & 3)) << 4));
            const int qr = wrow0 + R;
            if (qr < it.n_c) {
              uint8_t* dst = static_cast<uint8_t*>(a.out) +
                             (((size_t)(it.q0 + qr) * H + it.h) * D + col) * esize + pj * 16;
              *reinterpret_cast<uint4*>(dst) = w;
            }
          }
          __syncwarp();
        }
      }
      // this warp is done with both accumulators and with xm / xl of this item
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.o_free);
      g += n_kv;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

}  // namespace pa

// ---------------------------------------------------------------------------------
// Host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulate, A/B in
// `ab_format` (0 = fp16, 1 = bf16), M = 128, N = n, B K-major or MN-major.
uint32_t make_idesc(uint32_t ab_format, bool b_mn_major, int n) {
  uint32_t d = 0;
  d |= 1u << 4;                 // D format: f32
  d |= ab_format << 7;          // A format
  d |= ab_format << 10;         // B format
  d |= (b_mn_major ? 1u : 0u) << 16;
  d |= (uint32_t)(n >> 3) << 17;  // N
  d |= (uint32_t)(128 >> 4) << 24;  // M
  return d;
}

// Checks pa_prefill_chunk's arguments, encodes the tensor maps and fills the
// kernel arguments; launches nothing.  *empty is set when there is no work.
int prefill_setup(void* out, int out_dtype, const void* q, const int32_t* cu_q_lens, const int32_t* ctx_before,
                  const void* k_pool, const void* v_pool, const int32_t* block_tables, int max_blocks_per_seq,
                  int num_chunks, int total_q, int max_q_len, int num_heads, int head_dim, int block_size,
                  int num_blocks, float scale, int dtype, int32_t* err_flag, pa::PrefillArgs& a, CUtensorMap& tm_q,
                  CUtensorMap& tm_k, CUtensorMap& tm_v, bool& empty) {
  empty = false;
  if (!pa_host::is_kv_dtype(dtype) || !pa_host::is_out_dtype(out_dtype)) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (block_size <= 0 || block_size % 16 != 0 || block_size > 65536) return PA_ERR_UNSUPPORTED;
  if (num_chunks < 0 || total_q < 0 || max_q_len < 0 || num_heads <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_chunks == 0 || total_q == 0 || max_q_len == 0) {
    empty = true;
    return PA_OK;
  }
  if (num_heads > 65535) return PA_ERR_INVALID_ARG;
  if (!out || !q || !cu_q_lens || !ctx_before || !k_pool || !v_pool || !block_tables || !err_flag)
    return PA_ERR_INVALID_ARG;
  if (!pa_host::aligned16(q) || !pa_host::aligned16(k_pool) || !pa_host::aligned16(v_pool) ||
      !pa_host::aligned16(out))
    return PA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return PA_ERR_INVALID_ARG;
  const uint64_t pool_rows = (uint64_t)num_blocks * num_heads * block_size;
  if (pool_rows >= (1ull << 31)) return PA_ERR_INVALID_ARG;
  const long long qtiles = (max_q_len + pa::kPfRows - 1) / pa::kPfRows;
  if (qtiles * num_chunks * num_heads >= (1ll << 31)) return PA_ERR_INVALID_ARG;

  auto encode = get_encode_fn();
  if (encode == nullptr) return PA_ERR_CUDA;
  const CUtensorMapDataType tdt = dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  {
    cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_heads, (cuuint64_t)total_q};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)num_heads * head_dim * 2};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode(&tm_q, tdt, 3, const_cast<void*>(q), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PA_ERR_CUDA;
  }
  int rows_per_load = 128;  // gcd(block_size, 128), a power of two from 16 to 128
  while (block_size % rows_per_load != 0) rows_per_load /= 2;
  for (int which = 0; which < 2; ++which) {
    cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)pool_rows};
    cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)rows_per_load};
    cuuint32_t es[2] = {1, 1};
    if (encode(which ? &tm_v : &tm_k, tdt, 2, const_cast<void*>(which ? v_pool : k_pool), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PA_ERR_CUDA;
  }

  a.out = out;
  a.out_dtype = out_dtype;
  a.cu_q_lens = cu_q_lens;
  a.ctx_before = ctx_before;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_heads = num_heads;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.rows_per_load = rows_per_load;
  a.rpl_shift = 31 - __builtin_clz((unsigned)rows_per_load);
  a.pool_rows = (int)pool_rows;
  a.qscale = scale * 1.4426950408889634f;
  const uint32_t fmt = dtype == PA_BF16 ? 1u : 0u;
  a.idesc_s = make_idesc(fmt, false, pa::kPfKeys);
  a.idesc_pv = make_idesc(fmt, true, head_dim);
  a.err_flag = err_flag;
  a.num_chunks = num_chunks;
  a.qtiles = (int)qtiles;
  return PA_OK;
}

}  // namespace

namespace pa_host {

int prefill_check(void* out, int out_dtype, const void* q, const int32_t* cu_q_lens, const int32_t* ctx_before,
                  const void* k_pool, const void* v_pool, const int32_t* block_tables, int max_blocks_per_seq,
                  int num_chunks, int total_q, int max_q_len, int num_heads, int head_dim, int block_size,
                  int num_blocks, float scale, int dtype, int32_t* err_flag) {
  pa::PrefillArgs a;
  CUtensorMap tm_q, tm_k, tm_v;
  bool empty = false;
  return prefill_setup(out, out_dtype, q, cu_q_lens, ctx_before, k_pool, v_pool, block_tables, max_blocks_per_seq,
                       num_chunks, total_q, max_q_len, num_heads, head_dim, block_size, num_blocks, scale, dtype,
                       err_flag, a, tm_q, tm_k, tm_v, empty);
}

int prefill_launch(void* out, int out_dtype, const void* q, const int32_t* cu_q_lens, const int32_t* ctx_before,
                   const void* k_pool, const void* v_pool, const int32_t* block_tables, int max_blocks_per_seq,
                   int num_chunks, int total_q, int max_q_len, int num_heads, int head_dim, int block_size,
                   int num_blocks, float scale, int dtype, int32_t* err_flag, int max_ctas, int head_group,
                   void* stream) {
  pa::PrefillArgs a;
  CUtensorMap tm_q, tm_k, tm_v;
  bool empty = false;
  int st = prefill_setup(out, out_dtype, q, cu_q_lens, ctx_before, k_pool, v_pool, block_tables,
                         max_blocks_per_seq, num_chunks, total_q, max_q_len, num_heads, head_dim, block_size,
                         num_blocks, scale, dtype, err_flag, a, tm_q, tm_k, tm_v, empty);
  if (st != PA_OK || empty) return st;
  if (debug_checks()) {
    int64_t bad[2];
    st = check_prefill_inputs(cu_q_lens, ctx_before, block_tables, max_blocks_per_seq, num_chunks, total_q,
                              max_q_len, block_size, num_blocks, stream, bad);
    if (st != PA_OK) {
      std::fprintf(stderr, "pa_prefill_chunk (PA_DEBUG): chunk %lld, logical block %lld is invalid\n",
                   (long long)bad[0], (long long)bad[1]);
      return st;
    }
  }

  auto kern = head_dim == 128
                  ? (dtype == PA_BF16 ? pa::prefill_kernel<__nv_bfloat16, 128> : pa::prefill_kernel<__half, 128>)
                  : (dtype == PA_BF16 ? pa::prefill_kernel<__nv_bfloat16, 64> : pa::prefill_kernel<__half, 64>);
  const int variant = (dtype == PA_BF16 ? 1 : 0) + (head_dim == 128 ? 2 : 0);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
  // per kernel variant and device; host threads may race to configure (idempotent)
  static std::atomic<bool> configured[4][64];
  if (!configured[variant][dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pa::kPfSmemBytes) !=
        cudaSuccess)
      return PA_ERR_CUDA;
    configured[variant][dev].store(true, std::memory_order_release);
  }
  const long long n_items = (long long)a.qtiles * num_chunks * num_heads;
  const int sms = device_sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  // persistent: at most one CTA per SM (shared and tensor memory allow one)
  long long ctas = max_ctas > 0 && max_ctas < sms ? max_ctas : sms;
  if (ctas > n_items) ctas = n_items;
  // head_group > 0: the caller's group size.  Otherwise a launch of many
  // rounds deals its heads in groups of at least three rounds' worth of items,
  // so that the CTAs stream one group's K/V at a time (it can stay in L2 for
  // the group's other query tiles) instead of every head's.
  a.head_group = num_heads;
  if (head_group > 0) {
    a.head_group = head_group < num_heads ? head_group : num_heads;
  } else if (n_items >= 8 * ctas) {
    const long long npairs = (long long)a.qtiles * num_chunks;
    const long long g = (3 * ctas + npairs - 1) / npairs;
    if (g < num_heads) {
      const int ngroups = num_heads / (int)g;
      a.head_group = (num_heads + ngroups - 1) / ngroups;
    }
  }
  kern<<<dim3((unsigned)ctas), pa::kPfThreads, pa::kPfSmemBytes, (cudaStream_t)stream>>>(tm_q, tm_k, tm_v, a);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa_host

extern "C" int pa_prefill_chunk(void* out, int out_dtype, const void* q, const int32_t* cu_q_lens,
                                const int32_t* ctx_before, const void* k_pool, const void* v_pool,
                                const int32_t* block_tables, int max_blocks_per_seq, int num_chunks, int total_q,
                                int max_q_len, int num_heads, int head_dim, int block_size, int num_blocks,
                                float scale, int dtype, int32_t* err_flag, void* stream) {
  pa_host::Range range("pa_prefill_chunk");
  return pa_host::prefill_launch(out, out_dtype, q, cu_q_lens, ctx_before, k_pool, v_pool, block_tables,
                                 max_blocks_per_seq, num_chunks, total_q, max_q_len, num_heads, head_dim, block_size,
                                 num_blocks, scale, dtype, err_flag, 0, 0, stream);
}
