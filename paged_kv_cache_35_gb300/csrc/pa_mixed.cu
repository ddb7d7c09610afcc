// pa_mixed_step: one step of a batch that mixes decode sequences and prefill
// chunks, with the two kinds of work running at the same time.
//
// Method: the continuous-batching page ("연속 배치 처리 아키텍처", sections
// "Chunked prefill" and the scheduler) fills one step's token budget with the
// running requests' decode tokens first and prefill chunks after them, and
// runs them as one forward pass.
//
// Design (ours, for one GB300): the two parts stress different units -- the
// decode streams K/V from HBM with CUDA-core arithmetic, the prefill is bound
// by the tensor cores -- so they overlap.  The prefill's persistent grid is
// capped to a share of the SMs and launched first, on a second stream, so its
// CTAs hold those SMs; the decode's persistent grid then fills the rest of the
// GPU on the caller's stream.  Events order the second stream after the
// caller's earlier work and the caller's later work after both parts.
#include "pa_common.cuh"

extern "C" int pa_mixed_step(void* dec_out, int dec_out_dtype, const void* dec_q, const int32_t* dec_block_tables,
                             int dec_max_blocks_per_seq, const int32_t* context_lens, int max_context_len,
                             int num_seqs, void* workspace, size_t workspace_bytes, void* pf_out, int pf_out_dtype,
                             const void* pf_q, const int32_t* cu_q_lens, const int32_t* ctx_before,
                             const int32_t* pf_block_tables, int pf_max_blocks_per_seq, int num_chunks, int total_q,
                             int max_q_len, const void* k_pool, const void* v_pool, int num_heads, int head_dim,
                             int block_size, int num_blocks, float scale, int dtype, int prefill_sms,
                             int32_t* err_flag, void* stream, void* aux_stream) {
  if (aux_stream == nullptr || aux_stream == stream) return PA_ERR_INVALID_ARG;
  int st = pa_host::decode_check(dec_out, dec_out_dtype, dec_q, k_pool, v_pool, dec_block_tables,
                                 dec_max_blocks_per_seq, context_lens, max_context_len, num_seqs, num_heads, head_dim,
                                 block_size, num_blocks, scale, dtype, workspace, workspace_bytes, 0, err_flag);
  if (st != PA_OK) return st;
  st = pa_host::prefill_check(pf_out, pf_out_dtype, pf_q, cu_q_lens, ctx_before, k_pool, v_pool, pf_block_tables,
                              pf_max_blocks_per_seq, num_chunks, total_q, max_q_len, num_heads, head_dim, block_size,
                              num_blocks, scale, dtype, err_flag);
  if (st != PA_OK) return st;
  const int sms = pa_host::device_sm_count();
  if (sms <= 0) return PA_ERR_CUDA;
  int cap = prefill_sms > 0 ? (prefill_sms < sms ? prefill_sms : sms) : (sms * PA_MIXED_PREFILL_SHARE + 50) / 100;
  if (cap < 1) cap = 1;

  cudaStream_t s = (cudaStream_t)stream, aux = (cudaStream_t)aux_stream;
  cudaEvent_t fork = nullptr, join = nullptr;
  if (cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess) {
    cudaEventDestroy(fork);
    return PA_ERR_CUDA;
  }
  int result = PA_OK;
  if (cudaEventRecord(fork, s) != cudaSuccess || cudaStreamWaitEvent(aux, fork, 0) != cudaSuccess) {
    result = PA_ERR_CUDA;
  } else {
    // prefill first: its CTAs take their SMs before the decode's grid fills the GPU
    const int pst = pa_host::prefill_launch(pf_out, pf_out_dtype, pf_q, cu_q_lens, ctx_before, k_pool, v_pool,
                                            pf_block_tables, pf_max_blocks_per_seq, num_chunks, total_q, max_q_len,
                                            num_heads, head_dim, block_size, num_blocks, scale, dtype, err_flag, cap,
                                            aux_stream);
    const int dst = pa_decode(dec_out, dec_out_dtype, dec_q, k_pool, v_pool, dec_block_tables,
                              dec_max_blocks_per_seq, context_lens, max_context_len, num_seqs, num_heads, head_dim,
                              block_size, num_blocks, scale, dtype, workspace, workspace_bytes, 0, err_flag, stream);
    if (cudaEventRecord(join, aux) != cudaSuccess || cudaStreamWaitEvent(s, join, 0) != cudaSuccess)
      result = PA_ERR_CUDA;
    if (pst != PA_OK) result = pst;
    else if (dst != PA_OK) result = dst;
  }
  cudaEventDestroy(fork);  // released once the recorded work has completed
  cudaEventDestroy(join);
  return result;
}
