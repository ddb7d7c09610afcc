// Host-side validation of block tables and lengths (debug aid), and a
// self-test of the kernels' bounded waits.
//
// The kernels never trap: a table entry outside the pool or a length past a
// table only sets a bit in the device error flag and the bad work is skipped.
// These checks find the first bad entry on the host instead, before anything
// is launched: they copy the tables and lengths from the device, synchronise
// the stream, and walk exactly the entries the kernels would read (the
// entries covering each sequence's or chunk's context; the paper summary's
// section 4 block mapping, position p in logical block p / B).
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "pa_common.cuh"

namespace {

template <typename T>
int fetch(std::vector<T>& dst, const T* src, size_t n, cudaStream_t s) {
  dst.resize(n);
  if (n == 0) return PA_OK;
  if (src == nullptr) return PA_ERR_INVALID_ARG;
  if (cudaMemcpyAsync(dst.data(), src, n * sizeof(T), cudaMemcpyDeviceToHost, s) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

void report(int64_t* bad_out, int64_t row, int64_t logical_block) {
  if (bad_out != nullptr) {
    bad_out[0] = row;
    bad_out[1] = logical_block;
  }
}

}  // namespace

namespace pa {

// Self-test of the bounded waits every kernel uses: one CTA puts a bulk copy
// in flight on barrier `landed`, then waits on barrier `never`, which nothing
// arrives at.  After the wait limit the wait sets PA_FLAG_TIMEOUT and gives
// up; the CTA then waits (bounded, ignoring the abort) for its own copy to
// land before it exits, as every kernel does on an abort.
__global__ void selftest_wait_kernel(const uint4* __restrict__ src, int32_t* err_flag, int32_t* result) {
  __shared__ __align__(128) uint4 buf[256];  // 4 KiB
  __shared__ uint64_t landed, never;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&landed, 1);
    mbar_init(&never, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&landed, sizeof(buf));
    bulk_g2s(buf, src, sizeof(buf), &landed);
    const bool ok = mbar_wait(&never, 0, &abort_flag, err_flag);
    const bool drained = mbar_wait_drain(&landed, 0);
    result[0] = ok ? 1 : 0;
    result[1] = drained ? 1 : 0;
    result[2] = drained ? (int32_t)buf[255].w : -1;
  }
}

}  // namespace pa

namespace pa_host {

bool debug_checks() {
  static const bool on = [] {
    const char* v = std::getenv("PA_DEBUG");
    return v != nullptr && v[0] != '\0' && std::strcmp(v, "0") != 0;
  }();
  return on;
}

int check_decode_inputs(const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                        int num_seqs, int max_context_len, int block_size, int num_blocks, void* stream,
                        int64_t* bad_out) {
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  std::vector<int32_t> lens, tables;
  int st = fetch(lens, context_lens, (size_t)num_seqs, s);
  if (st == PA_OK) st = fetch(tables, block_tables, (size_t)num_seqs * max_blocks_per_seq, s);
  if (st != PA_OK) return st;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  for (int i = 0; i < num_seqs; ++i) {
    const int n = lens[i];
    if (n < 0 || n > max_context_len || (int64_t)n > (int64_t)max_blocks_per_seq * block_size) {
      report(bad_out, i, -1);
      return PA_ERR_BAD_INDEX;
    }
    for (int b = 0; b < (n + block_size - 1) / block_size; ++b) {
      const int32_t id = tables[(size_t)i * max_blocks_per_seq + b];
      if (id < 0 || id >= num_blocks) {
        report(bad_out, i, b);
        return PA_ERR_BAD_INDEX;
      }
    }
  }
  report(bad_out, -1, -1);
  return PA_OK;
}

int check_prefill_inputs(const int32_t* cu_q_lens, const int32_t* ctx_before, const int32_t* block_tables,
                         int max_blocks_per_seq, int num_chunks, int total_q, int max_q_len, int block_size,
                         int num_blocks, void* stream, int64_t* bad_out) {
  if (num_chunks < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  std::vector<int32_t> cu, cb, tables;
  int st = fetch(cu, cu_q_lens, (size_t)num_chunks + 1, s);
  if (st == PA_OK) st = fetch(cb, ctx_before, (size_t)num_chunks, s);
  if (st == PA_OK) st = fetch(tables, block_tables, (size_t)num_chunks * max_blocks_per_seq, s);
  if (st != PA_OK) return st;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  if (cu[0] != 0 || cu[num_chunks] != total_q) {
    report(bad_out, -1, -1);
    return PA_ERR_BAD_INDEX;
  }
  for (int c = 0; c < num_chunks; ++c) {
    const int n = cu[c + 1] - cu[c];
    const int64_t ctx = (int64_t)cb[c] + n;
    if (n < 0 || n > max_q_len || cb[c] < 0 || ctx > (int64_t)max_blocks_per_seq * block_size) {
      report(bad_out, c, -1);
      return PA_ERR_BAD_INDEX;
    }
    for (int64_t b = 0; b < (ctx + block_size - 1) / block_size; ++b) {
      const int32_t id = tables[(size_t)c * max_blocks_per_seq + b];
      if (id < 0 || id >= num_blocks) {
        report(bad_out, c, b);
        return PA_ERR_BAD_INDEX;
      }
    }
  }
  report(bad_out, -1, -1);
  return PA_OK;
}

}  // namespace pa_host

extern "C" {

int pa_check_decode_inputs(const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                           int num_seqs, int max_context_len, int block_size, int num_blocks, void* stream,
                           int64_t* bad_out) {
  pa_host::Range r("pa_check_decode_inputs");
  return pa_host::check_decode_inputs(block_tables, max_blocks_per_seq, context_lens, num_seqs, max_context_len,
                                      block_size, num_blocks, stream, bad_out);
}

int pa_check_prefill_inputs(const int32_t* cu_q_lens, const int32_t* ctx_before, const int32_t* block_tables,
                            int max_blocks_per_seq, int num_chunks, int total_q, int max_q_len, int block_size,
                            int num_blocks, void* stream, int64_t* bad_out) {
  pa_host::Range r("pa_check_prefill_inputs");
  return pa_host::check_prefill_inputs(cu_q_lens, ctx_before, block_tables, max_blocks_per_seq, num_chunks, total_q,
                                       max_q_len, block_size, num_blocks, stream, bad_out);
}

int pa_selftest_wait_timeout(const void* src, int32_t* err_flag, int32_t* result, void* stream) {
  pa_host::Range r("pa_selftest_wait_timeout");
  if (src == nullptr || err_flag == nullptr || result == nullptr || !pa_host::aligned16(src)) return PA_ERR_INVALID_ARG;
  pa::selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(static_cast<const uint4*>(src), err_flag, result);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"
