/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle for paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this file's library.  It shares no
 * code, header or table with the CUDA library; neither includes the other.
 *
 * What it computes, and where the definitions come from
 * ("Efficient Memory Management for Large Language Model Serving with
 *  PagedAttention", as summarised on the three source pages):
 *   - attention: section 4 equation, A_ij = exp(q_i.k_j/sqrt d) / sum_{j'<=i}
 *     exp(q_i.k_j'/sqrt d), o_i = sum_{j<=i} A_ij v_j.  The scale is a
 *     parameter (1/sqrt(d) by default).
 *   - paging: section 4, the j-th token (1-based) lives in block
 *     floor((j-1)/B), slot (j-1) mod B; 0-based position p lives in logical
 *     block p/B, slot p%B, and the block table maps the logical block to a
 *     physical one.  Pools are laid out [num_blocks][H][B][D]; the offset of
 *     (block, head, slot, dim) is written out in pool_offset() below.
 *   - the paged result equals plain attention over the reassembled
 *     sequence ("Attention計算の修正" section of the blog page), so the
 *     oracle reassembles K and V and applies the definition directly, with
 *     no blocking, splitting or online softmax.
 *   - the KV write: the pseudo-code's append_token stores the token's k and
 *     v in the next free slot of the last block; here that slot is given
 *     as slot = block*B + offset, and slot < 0 means "skip" (padding).
 *   - copy-on-write: the whole source block (every slot, K and V) is copied
 *     into the destination block.
 *   - chunked prefill (continuous-batching page, "Chunked prefill"): a chunk
 *     of n query tokens placed after c0 context tokens; query i is at
 *     position c0+i and attends positions 0..c0+i (the causal j <= i of the
 *     section 4 equation).
 *
 * Inputs arrive as the raw 16-bit patterns of fp16 or bf16 values and are
 * decoded exactly to double.  Everything is computed in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F16 = 0, OR_BF16 = 1 };
enum { OR_OK = 0, OR_BAD_ARG = 1, OR_BAD_INDEX = 2, OR_NO_MEMORY = 3 };

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^(1-15-10) */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m + 1024), e - 25); /* (1 + m/1024) * 2^(e-15) */
  return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double decode_elt(uint16_t bits, int dtype) {
  return dtype == OR_BF16 ? oracle_bf16_to_double(bits) : oracle_f16_to_double(bits);
}

/* Element offset of (physical block, head, slot, dim) in a [NB][H][B][D] pool. */
static int64_t pool_offset(int64_t block, int head, int slot, int dim, int H, int B, int D) {
  return ((block * H + head) * (int64_t)B + slot) * D + dim;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads the parallel loops use from now on (n >= 1); returns the number in
 * effect afterwards (1 without OpenMP).  Only the CPU-baseline timing uses
 * it, to time the oracle single-threaded beside its OpenMP run. */
int oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}

/*
 * Attention of one query row over the first n tokens of one sequence's
 * paged K/V for one head.  Steps, in the order the definition gives them:
 *   1. reassemble K_s[p], V_s[p] for p < n through the block table;
 *   2. x_p = scale * q . K_s[p];
 *   3. A_p = exp(x_p - max x) / sum exp(x - max x)   (the max shift only
 *      guards against overflow; it cancels exactly in the ratio);
 *   4. o = sum_p A_p V_s[p].
 * Returns OR_BAD_INDEX if the table sends a position outside the pool.
 */
static int attend_one(double* o, const uint16_t* q_row, const uint16_t* k_pool,
                      const uint16_t* v_pool, const int32_t* table_row, int n, int head,
                      int H, int D, int B, int NB, double scale, int dtype,
                      double* kbuf, double* vbuf, double* xbuf) {
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (n <= 0) return OR_OK;
  /* 1. reassembly */
  for (int p = 0; p < n; ++p) {
    int32_t blk = table_row[p / B];
    int slot = p % B;
    if (blk < 0 || blk >= NB) return OR_BAD_INDEX;
    for (int d = 0; d < D; ++d) {
      int64_t off = pool_offset(blk, head, slot, d, H, B, D);
      kbuf[(int64_t)p * D + d] = decode_elt(k_pool[off], dtype);
      vbuf[(int64_t)p * D + d] = decode_elt(v_pool[off], dtype);
    }
  }
  /* 2. scores */
  double qd[512];
  for (int d = 0; d < D; ++d) qd[d] = decode_elt(q_row[d], dtype);
  double xmax = -INFINITY;
  for (int p = 0; p < n; ++p) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += qd[d] * kbuf[(int64_t)p * D + d];
    xbuf[p] = scale * acc;
    if (xbuf[p] > xmax) xmax = xbuf[p];
  }
  /* 3. softmax weights */
  double denom = 0.0;
  for (int p = 0; p < n; ++p) {
    xbuf[p] = exp(xbuf[p] - xmax);
    denom += xbuf[p];
  }
  /* 4. weighted sum of values */
  for (int p = 0; p < n; ++p) {
    double a = xbuf[p] / denom;
    for (int d = 0; d < D; ++d) o[d] += a * vbuf[(int64_t)p * D + d];
  }
  return OR_OK;
}

/*
 * Single-query decode attention for every (sequence, head):
 *   out[s][h][:] = attention of q[s][h] over context_lens[s] tokens.
 * q: [S][H][D] bits; pools: [NB][H][B][D] bits; block_tables: [S][MB];
 * out: [S][H][D] double.  context_lens[s] == 0 gives a zero row.
 * OpenMP (when compiled in) runs independent (s, h) pairs in parallel.
 */
int oracle_decode(double* out, const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                  const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                  int num_seqs, int num_heads, int head_dim, int block_size, int num_blocks,
                  double scale, int dtype) {
  const int S = num_seqs, H = num_heads, D = head_dim, B = block_size;
  if (D <= 0 || D > 512 || B <= 0 || S < 0 || H <= 0) return OR_BAD_ARG;
  int maxn = 0;
  for (int s = 0; s < S; ++s) {
    if (context_lens[s] < 0) return OR_BAD_ARG;
    if ((int64_t)context_lens[s] > (int64_t)max_blocks_per_seq * B) return OR_BAD_INDEX;
    if (context_lens[s] > maxn) maxn = context_lens[s];
  }
  int status = OR_OK;
#pragma omp parallel
  {
    double* kbuf = (double*)malloc(sizeof(double) * ((size_t)maxn * D + 1));
    double* vbuf = (double*)malloc(sizeof(double) * ((size_t)maxn * D + 1));
    double* xbuf = (double*)malloc(sizeof(double) * ((size_t)maxn + 1));
    if (!kbuf || !vbuf || !xbuf) {
#pragma omp atomic write
      status = OR_NO_MEMORY;
    } else {
#pragma omp for collapse(2) schedule(dynamic, 1)
      for (int s = 0; s < S; ++s) {
        for (int h = 0; h < H; ++h) {
          int r = attend_one(out + ((int64_t)s * H + h) * D, q + ((int64_t)s * H + h) * D, k_pool,
                             v_pool, block_tables + (int64_t)s * max_blocks_per_seq,
                             context_lens[s], h, H, D, B, num_blocks, scale, dtype, kbuf, vbuf,
                             xbuf);
          if (r != OR_OK) {
#pragma omp atomic write
            status = r;
          }
        }
      }
    }
    free(kbuf);
    free(vbuf);
    free(xbuf);
  }
  return status;
}

/*
 * Causal attention of prefill chunks over paged K/V.  Chunk c has query rows
 * cu_q_lens[c] .. cu_q_lens[c+1]-1 of q ([total][H][D]); row i of the chunk
 * sits at position ctx_before[c] + i and attends positions
 * 0 .. ctx_before[c] + i of sequence c (block_tables row c).  The chunk's own
 * K/V must already be in the pool.
 */
int oracle_prefill(double* out, const uint16_t* q, const int32_t* cu_q_lens,
                   const int32_t* ctx_before, const uint16_t* k_pool, const uint16_t* v_pool,
                   const int32_t* block_tables, int max_blocks_per_seq, int num_chunks,
                   int num_heads, int head_dim, int block_size, int num_blocks, double scale,
                   int dtype) {
  const int C = num_chunks, H = num_heads, D = head_dim, B = block_size;
  if (D <= 0 || D > 512 || B <= 0 || C < 0 || H <= 0) return OR_BAD_ARG;
  int maxn = 0;
  for (int c = 0; c < C; ++c) {
    int n = cu_q_lens[c + 1] - cu_q_lens[c];
    if (n < 0 || ctx_before[c] < 0) return OR_BAD_ARG;
    int last = ctx_before[c] + n;
    if ((int64_t)last > (int64_t)max_blocks_per_seq * B) return OR_BAD_INDEX;
    if (last > maxn) maxn = last;
  }
  const int total = C > 0 ? cu_q_lens[C] : 0;
  int status = OR_OK;
#pragma omp parallel
  {
    double* kbuf = (double*)malloc(sizeof(double) * ((size_t)maxn * D + 1));
    double* vbuf = (double*)malloc(sizeof(double) * ((size_t)maxn * D + 1));
    double* xbuf = (double*)malloc(sizeof(double) * ((size_t)maxn + 1));
    if (!kbuf || !vbuf || !xbuf) {
#pragma omp atomic write
      status = OR_NO_MEMORY;
    } else {
#pragma omp for collapse(2) schedule(dynamic, 1)
      for (int r = 0; r < total; ++r) {
        for (int h = 0; h < H; ++h) {
          int c = 0;
          while (c + 1 < C && cu_q_lens[c + 1] <= r) ++c;
          int i = r - cu_q_lens[c];
          int n = ctx_before[c] + i + 1; /* positions 0 .. c0+i inclusive */
          int rr = attend_one(out + ((int64_t)r * H + h) * D, q + ((int64_t)r * H + h) * D,
                              k_pool, v_pool, block_tables + (int64_t)c * max_blocks_per_seq, n,
                              h, H, D, B, num_blocks, scale, dtype, kbuf, vbuf, xbuf);
          if (rr != OR_OK) {
#pragma omp atomic write
            status = rr;
          }
        }
      }
    }
    free(kbuf);
    free(vbuf);
    free(xbuf);
  }
  return status;
}

/*
 * Slot-scatter KV write: for each token t with slot_mapping[t] >= 0, copy
 * the bits of k_new[t][h][:] and v_new[t][h][:] into slot
 * slot_mapping[t] % B of physical block slot_mapping[t] / B, for every head.
 * A slot beyond the pool returns OR_BAD_INDEX (tokens before it are written).
 */
int oracle_reshape_and_cache(const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_pool,
                             uint16_t* v_pool, const int64_t* slot_mapping, int num_tokens,
                             int num_heads, int head_dim, int block_size, int num_blocks) {
  const int H = num_heads, D = head_dim, B = block_size;
  for (int t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= (int64_t)num_blocks * B) return OR_BAD_INDEX;
    int64_t blk = slot / B;
    int off = (int)(slot % B);
    for (int h = 0; h < H; ++h)
      for (int d = 0; d < D; ++d) {
        int64_t dst = pool_offset(blk, h, off, d, H, B, D);
        int64_t src = ((int64_t)t * H + h) * D + d;
        k_pool[dst] = k_new[src];
        v_pool[dst] = v_new[src];
      }
  }
  return OR_OK;
}

/* Block swap between two pools ([summary] section 5: a preempted sequence's
 * KV blocks are swapped out to CPU memory and back in; [cb] "오프로딩": the
 * blocks are copied into a pinned CPU buffer and copied back on resume).
 * For each pair (s, d): dst block d := src block s, K and V, every head and
 * slot.  A pair with an id outside its pool is skipped; the return value is
 * the number of skipped pairs. */
int oracle_swap_blocks(const uint16_t* src_k, const uint16_t* src_v, int src_num_blocks, uint16_t* dst_k,
                       uint16_t* dst_v, int dst_num_blocks, const int32_t* pairs, int num_pairs, int num_heads,
                       int head_dim, int block_size) {
  const int64_t per_block = (int64_t)num_heads * block_size * head_dim;
  int skipped = 0;
  for (int i = 0; i < num_pairs; ++i) {
    const int32_t s = pairs[2 * i], d = pairs[2 * i + 1];
    if (s < 0 || s >= src_num_blocks || d < 0 || d >= dst_num_blocks) {
      ++skipped;
      continue;
    }
    memcpy(dst_k + d * per_block, src_k + s * per_block, sizeof(uint16_t) * per_block);
    memcpy(dst_v + d * per_block, src_v + s * per_block, sizeof(uint16_t) * per_block);
  }
  return skipped;
}

/*
 * Copy-on-write block copy: for each pair (src, dst) in order, every slot of
 * every head of block src is copied bitwise into block dst, in K and in V.
 */
int oracle_copy_blocks(uint16_t* k_pool, uint16_t* v_pool, const int32_t* pairs, int num_pairs,
                       int num_heads, int head_dim, int block_size, int num_blocks) {
  const int64_t per_block = (int64_t)num_heads * block_size * head_dim;
  for (int i = 0; i < num_pairs; ++i) {
    int32_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) return OR_BAD_INDEX;
    memcpy(k_pool + dst * per_block, k_pool + src * per_block, sizeof(uint16_t) * per_block);
    memcpy(v_pool + dst * per_block, v_pool + src * per_block, sizeof(uint16_t) * per_block);
  }
  return OR_OK;
}
