// KV write (slot scatter), copy-on-write block copy, block swap between a
// GPU pool and a pinned host pool, and the error-flag and status entry points
// of the C ABI.
//
// The kernels are pure byte movers: 16-byte vector loads and stores,
// grid-stride loops.  The scatter and the block copy are bound by HBM
// bandwidth, the swap by the CPU-GPU link.
#include <atomic>
#include <cstdio>

#include "pa_common.cuh"

namespace pa {

// One thread moves one 16-byte vector of K and the matching one of V.
// Vector index -> (token t, head h, vector v of head_dim/8).
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(const uint4* __restrict__ k_new,
                                                                const uint4* __restrict__ v_new,
                                                                uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                                                                const int64_t* __restrict__ slot_mapping,
                                                                int64_t total_vecs, int vecs_per_head, int num_heads,
                                                                int block_size, int64_t num_slots, int32_t* err_flag) {
  // a kernel launched behind this one as a programmatic dependent (pa_decode's
  // planning kernel) may start at once; it waits for this one before it ends
  griddep_launch_dependents();
  const int64_t vecs_per_token = (int64_t)vecs_per_head * num_heads;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total_vecs;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / vecs_per_token;
    const int64_t r = i - t * vecs_per_token;  // = h * vecs_per_head + v
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (r == 0) atomicOr(err_flag, PA_FLAG_BAD_SLOT);
      continue;
    }
    const int64_t blk = slot / block_size;
    const int64_t off = slot - blk * block_size;
    const int64_t h = r / vecs_per_head;
    const int64_t v = r - h * vecs_per_head;
    // [blk][h][off][v] in vectors
    const int64_t dst = ((blk * num_heads + h) * block_size + off) * vecs_per_head + v;
    k_pool[dst] = __ldg(k_new + i);
    v_pool[dst] = __ldg(v_new + i);
  }
}

// grid.y = pair index; each CTA walks a strided share of the block's vectors.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                                                          const int32_t* __restrict__ pairs, int64_t vecs_per_block,
                                                          int num_blocks, int32_t* err_flag) {
  const int pair = blockIdx.y;
  const int32_t src = __ldg(pairs + 2 * pair);
  const int32_t dst = __ldg(pairs + 2 * pair + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(err_flag, PA_FLAG_BAD_BLOCK);
    return;
  }
  const uint4* ks = k_pool + (int64_t)src * vecs_per_block;
  const uint4* vs = v_pool + (int64_t)src * vecs_per_block;
  uint4* kd = k_pool + (int64_t)dst * vecs_per_block;
  uint4* vd = v_pool + (int64_t)dst * vecs_per_block;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < vecs_per_block;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 a = ks[i];
    const uint4 b = vs[i];
    kd[i] = a;
    vd[i] = b;
  }
}

// Whole-block moves between two pools, either of which may be pinned host
// memory read or written through its device address (swap-out / swap-in).
// grid.y = pair; each CTA walks a strided share of the block's K and V
// vectors with four vectors of each in flight per thread, since a load from
// the host side of the link takes several times an HBM load's latency.
__global__ void __launch_bounds__(256) swap_blocks_kernel(const uint4* __restrict__ src_k,
                                                          const uint4* __restrict__ src_v, int src_num_blocks,
                                                          uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
                                                          int dst_num_blocks, const int32_t* __restrict__ pairs,
                                                          int64_t vecs_per_block, int32_t* err_flag) {
  const int pair = blockIdx.y;
  const int32_t src = __ldg(pairs + 2 * pair);
  const int32_t dst = __ldg(pairs + 2 * pair + 1);
  if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(err_flag, PA_FLAG_BAD_BLOCK);
    return;
  }
  const uint4* ks = src_k + (int64_t)src * vecs_per_block;
  const uint4* vs = src_v + (int64_t)src * vecs_per_block;
  uint4* kd = dst_k + (int64_t)dst * vecs_per_block;
  uint4* vd = dst_v + (int64_t)dst * vecs_per_block;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  for (; i + 3 * stride < vecs_per_block; i += 4 * stride) {
    uint4 a[4], b[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      a[u] = ks[i + u * stride];
      b[u] = vs[i + u * stride];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      kd[i + u * stride] = a[u];
      vd[i + u * stride] = b[u];
    }
  }
  for (; i < vecs_per_block; i += stride) {
    const uint4 a = ks[i];
    const uint4 b = vs[i];
    kd[i] = a;
    vd[i] = b;
  }
}

}  // namespace pa

namespace pa_host {

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  // per device; host threads may race to fill an entry, all with the same value
  static std::atomic<int> cached[64];
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace pa_host

extern "C" {

int pa_version(void) { return 100; }

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported dtype, head_dim or block_size";
    case PA_ERR_NO_FREE_BLOCKS: return "no free KV-cache blocks";
    case PA_ERR_REFCOUNT: return "reference count underflow";
    case PA_ERR_BAD_INDEX: return "block, slot or length out of range (device flag)";
    case PA_ERR_CUDA: return "CUDA runtime error";
    case PA_ERR_TIMEOUT: return "device wait timed out (device flag)";
    case PA_ERR_WORKSPACE: return "workspace too small";
    default: return "unknown status";
  }
}

int pa_device_sm_count(void) { return pa_host::device_sm_count(); }

int pa_reshape_and_cache(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                         const int64_t* slot_mapping, int num_tokens, int num_heads, int head_dim, int block_size,
                         int num_blocks, int dtype, int32_t* err_flag, void* stream) {
  pa_host::Range range("pa_reshape_and_cache");
  if (num_tokens < 0 || num_heads <= 0 || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
  if (!pa_host::is_kv_dtype(dtype)) return PA_ERR_UNSUPPORTED;
  if (head_dim <= 0 || head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!k_new || !v_new || !k_pool || !v_pool || !slot_mapping || !err_flag) return PA_ERR_INVALID_ARG;
  if (!pa_host::aligned16(k_new) || !pa_host::aligned16(v_new) || !pa_host::aligned16(k_pool) ||
      !pa_host::aligned16(v_pool))
    return PA_ERR_INVALID_ARG;
  const int vecs_per_head = head_dim / 8;
  const int64_t total = (int64_t)num_tokens * num_heads * vecs_per_head;
  const int threads = 256;
  const int sms = pa_host::device_sm_count();
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 8;
  if (blocks > cap) blocks = cap;
  pa::reshape_and_cache_kernel<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(
      (const uint4*)k_new, (const uint4*)v_new, (uint4*)k_pool, (uint4*)v_pool, slot_mapping, total, vecs_per_head,
      num_heads, block_size, (int64_t)num_blocks * block_size, err_flag);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_copy_blocks(void* k_pool, void* v_pool, const int32_t* pairs, int n_pairs, int num_heads, int head_dim,
                   int block_size, int num_blocks, int dtype, int32_t* err_flag, void* stream) {
  pa_host::Range range("pa_copy_blocks");
  if (n_pairs < 0 || num_heads <= 0 || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
  if (!pa_host::is_kv_dtype(dtype)) return PA_ERR_UNSUPPORTED;
  if (head_dim <= 0 || head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
  if (n_pairs == 0) return PA_OK;
  if (n_pairs > 65535) return PA_ERR_INVALID_ARG;
  if (!k_pool || !v_pool || !pairs || !err_flag) return PA_ERR_INVALID_ARG;
  if (!pa_host::aligned16(k_pool) || !pa_host::aligned16(v_pool)) return PA_ERR_INVALID_ARG;
  const int64_t vecs_per_block = (int64_t)num_heads * block_size * head_dim / 8;
  const int threads = 256;
  int64_t per_pair = (vecs_per_block + threads - 1) / threads;
  if (per_pair > 64) per_pair = 64;
  dim3 grid((unsigned)per_pair, (unsigned)n_pairs);
  pa::copy_blocks_kernel<<<grid, threads, 0, (cudaStream_t)stream>>>((uint4*)k_pool, (uint4*)v_pool, pairs,
                                                                     vecs_per_block, num_blocks, err_flag);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_swap_blocks(const void* src_k, const void* src_v, int src_num_blocks, void* dst_k, void* dst_v,
                   int dst_num_blocks, const int32_t* pairs, int n_pairs, int num_heads, int head_dim,
                   int block_size, int dtype, int32_t* err_flag, void* stream) {
  pa_host::Range range("pa_swap_blocks");
  if (n_pairs < 0 || num_heads <= 0 || src_num_blocks <= 0 || dst_num_blocks <= 0 || block_size <= 0)
    return PA_ERR_INVALID_ARG;
  if (!pa_host::is_kv_dtype(dtype)) return PA_ERR_UNSUPPORTED;
  if (head_dim <= 0 || head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
  if (n_pairs == 0) return PA_OK;
  if (n_pairs > 65535) return PA_ERR_INVALID_ARG;
  if (!src_k || !src_v || !dst_k || !dst_v || !pairs || !err_flag) return PA_ERR_INVALID_ARG;
  if (!pa_host::aligned16(src_k) || !pa_host::aligned16(src_v) || !pa_host::aligned16(dst_k) ||
      !pa_host::aligned16(dst_v))
    return PA_ERR_INVALID_ARG;
  const int64_t vecs_per_block = (int64_t)num_heads * block_size * head_dim / 8;
  const int threads = 256;
  int64_t per_pair = (vecs_per_block + 4 * threads - 1) / (4 * threads);
  if (per_pair > 64) per_pair = 64;
  if (per_pair < 1) per_pair = 1;
  dim3 grid((unsigned)per_pair, (unsigned)n_pairs);
  pa::swap_blocks_kernel<<<grid, threads, 0, (cudaStream_t)stream>>>(
      (const uint4*)src_k, (const uint4*)src_v, src_num_blocks, (uint4*)dst_k, (uint4*)dst_v, dst_num_blocks, pairs,
      vecs_per_block, err_flag);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_get_error(int32_t* err_flag, int32_t* flags_out, void* stream) {
  pa_host::Range range("pa_get_error");
  if (err_flag == nullptr) return PA_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, err_flag, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaMemsetAsync(err_flag, 0, sizeof(int32_t), s) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  if (flags_out) *flags_out = h;
  if (h & PA_FLAG_TIMEOUT) return PA_ERR_TIMEOUT;
  if (h != 0) return PA_ERR_BAD_INDEX;
  return PA_OK;
}

}  // extern "C"
