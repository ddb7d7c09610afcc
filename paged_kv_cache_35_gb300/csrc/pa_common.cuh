// Shared device helpers for the sm_103a kernels: inline PTX for mbarriers,
// bulk-async copies, the PDL grid-dependency controls and bounded waits.
//
// Every wait on an mbarrier here is bounded in time: after kWaitLimitNs of
// %globaltimer it gives up, sets PA_FLAG_TIMEOUT in the caller's error flag
// and returns false, so no kernel of this library can spin forever.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include "../../include/pa.h"

namespace pa {

constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier ----------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async proxy (bulk copies,
// tensor-core commits) before first use.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false if
// the CTA-wide abort flag is raised or the time limit passes (then the
// abort flag and PA_FLAG_TIMEOUT are raised).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* err_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (abort_flag != nullptr && *abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        if (abort_flag != nullptr) *abort_flag = 1;
        atomicOr(err_flag, PA_FLAG_TIMEOUT);
        return false;
      }
    }
  }
}

// Bounded wait that ignores the abort flag (used while draining copies).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ---- bulk-async copies ---------------------------------------------------------
// Global -> shared, completion counted in bytes on an mbarrier.  Both
// addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---- programmatic dependent launch ----------------------------------------------
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- conversions -------------------------------------------------------------------
template <typename T>
struct Elt;

template <>
struct Elt<__half> {
  __device__ __forceinline__ static void to_float8(const uint4& u, float* f) {
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 x = __half22float2(h[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
};

template <>
struct Elt<__nv_bfloat16> {
  __device__ __forceinline__ static void to_float8(const uint4& u, float* f) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 x = __bfloat1622float2(h[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
};

// Store one float as the requested output dtype (round to nearest even).
__device__ __forceinline__ void store_out(void* out, size_t idx, int out_dtype, float v) {
  if (out_dtype == PA_F32) {
    static_cast<float*>(out)[idx] = v;
  } else if (out_dtype == PA_BF16) {
    static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  } else {
    static_cast<__half*>(out)[idx] = __float2half_rn(v);
  }
}

}  // namespace pa

// Host-side helpers shared by the launch wrappers.
namespace pa_host {

inline int elt_bytes(int dtype) { return dtype == PA_F32 ? 4 : 2; }

inline bool is_kv_dtype(int dtype) { return dtype == PA_F16 || dtype == PA_BF16; }

inline bool is_out_dtype(int dtype) { return dtype == PA_F16 || dtype == PA_BF16 || dtype == PA_F32; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int device_sm_count();

// An NVTX range named after the C-ABI call, open for the call's host-side
// duration (visible in Nsight timelines; costs nothing measurable without a
// tool attached).
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};

// True when the environment variable PA_DEBUG is set to a non-empty value
// other than "0" (read once per process): the decode and prefill entry points
// then validate their tables and lengths on the host before launching.
bool debug_checks();
int check_decode_inputs(const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                        int num_seqs, int max_context_len, int block_size, int num_blocks, void* stream,
                        int64_t* bad_out);
int check_prefill_inputs(const int32_t* cu_q_lens, const int32_t* ctx_before, const int32_t* block_tables,
                         int max_blocks_per_seq, int num_chunks, int total_q, int max_q_len, int block_size,
                         int num_blocks, void* stream, int64_t* bad_out);

// Argument checks of pa_decode / pa_prefill_chunk that launch nothing, and
// the prefill launch with its persistent grid capped at max_ctas CTAs
// (0 = one per SM).  Defined next to the kernels.
int decode_check(void* out, int out_dtype, const void* q, const void* k_pool, const void* v_pool,
                 const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                 int max_context_len, int num_seqs, int num_heads, int head_dim, int block_size, int num_blocks,
                 float scale, int dtype, void* workspace, size_t workspace_bytes, int partition_size,
                 int32_t* err_flag);
int prefill_check(void* out, int out_dtype, const void* q, const int32_t* cu_q_lens, const int32_t* ctx_before,
                  const void* k_pool, const void* v_pool, const int32_t* block_tables, int max_blocks_per_seq,
                  int num_chunks, int total_q, int max_q_len, int num_heads, int head_dim, int block_size,
                  int num_blocks, float scale, int dtype, int32_t* err_flag);
int prefill_launch(void* out, int out_dtype, const void* q, const int32_t* cu_q_lens, const int32_t* ctx_before,
                   const void* k_pool, const void* v_pool, const int32_t* block_tables, int max_blocks_per_seq,
                   int num_chunks, int total_q, int max_q_len, int num_heads, int head_dim, int block_size,
                   int num_blocks, float scale, int dtype, int32_t* err_flag, int max_ctas, int head_group,
                   void* stream);

}  // namespace pa_host
