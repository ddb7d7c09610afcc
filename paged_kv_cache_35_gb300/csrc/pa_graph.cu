// Decode graphs: pa_decode recorded once per padded batch shape and replayed.
//
// Method: the continuous-batching page ("연속 배치 처리 아키텍처", section
// "CUDA 그래프") removes each step's CPU dispatch work by recording the GPU
// work once and replaying it for batches of the same shape; since the shape
// changes every step, query counts and KV lengths are padded up to multiples
// of fixed intervals, the recorded graphs are cached by padded shape, and an
// unseen shape triggers a new recording.
//
// Design (ours): the object owns only host state -- a capture stream and a
// map from (padded sequence count, padded KV length) to an instantiated
// graph.  The graphs read and write the caller's static device buffers given
// at creation.  Padding rows get a context length of 0, which pa_decode turns
// into zero rows without reading their tables.
#include <map>
#include <utility>

#include "pa_common.cuh"

struct pa_decode_graphs {
  void* out;
  int out_dtype;
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* tables;
  int max_blocks_per_seq;
  int32_t* ctx;
  int max_seqs, max_ctx;
  int num_heads, head_dim, block_size, num_blocks;
  float scale;
  int dtype;
  void* workspace;
  size_t workspace_bytes;
  int seq_interval, kv_interval;
  int32_t* err_flag;
  int device;
  cudaStream_t capture_stream;
  std::map<std::pair<int, int>, cudaGraphExec_t> graphs;
};

namespace {

int round_up(int x, int m) { return (int)(((long long)x + m - 1) / m * m); }

// Largest padded shapes a call can produce.
void padded_limits(int max_seqs, int max_ctx, int seq_interval, int kv_interval, int* s_pad, int* c_pad) {
  *s_pad = round_up(max_seqs, seq_interval);
  *c_pad = round_up(max_ctx > 0 ? max_ctx : 1, kv_interval);
}

size_t graphs_workspace_bytes(int max_seqs, int num_heads, int head_dim, int max_ctx, int seq_interval,
                              int kv_interval) {
  int s_max = 0, c_max = 0;
  padded_limits(max_seqs, max_ctx, seq_interval, kv_interval, &s_max, &c_max);
  size_t need = 0;
  for (int s = seq_interval; s <= s_max; s += seq_interval) {
    for (int c = kv_interval; c <= c_max; c += kv_interval) {
      const size_t b = pa_decode_workspace_bytes(s, num_heads, head_dim, c, 0);
      if (b == 0) return 0;
      if (b > need) need = b;
    }
  }
  return need;
}

}  // namespace

extern "C" {

size_t pa_decode_graphs_workspace_bytes(int max_seqs, int num_heads, int head_dim, int max_context_len,
                                        int seq_interval, int kv_interval) {
  if (max_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0 || seq_interval <= 0 ||
      kv_interval <= 0)
    return 0;
  if ((long long)round_up(max_seqs, seq_interval) / seq_interval * (round_up(max_context_len + 1, kv_interval) /
                                                                    kv_interval) > 1000000)
    return 0;  // too many buckets to enumerate
  return graphs_workspace_bytes(max_seqs, num_heads, head_dim, max_context_len, seq_interval, kv_interval);
}

int pa_decode_graphs_create(void* out_buf, int out_dtype, const void* q_buf, const void* k_pool, const void* v_pool,
                            const int32_t* tables_buf, int max_blocks_per_seq, int32_t* ctx_buf, int max_seqs,
                            int max_context_len, int num_heads, int head_dim, int block_size, int num_blocks,
                            float scale, int dtype, void* workspace, size_t workspace_bytes, int seq_interval,
                            int kv_interval, int32_t* err_flag, pa_decode_graphs** out) {
  if (out == nullptr) return PA_ERR_INVALID_ARG;
  *out = nullptr;
  if (max_seqs <= 0 || max_context_len < 0 || seq_interval <= 0 || kv_interval <= 0) return PA_ERR_INVALID_ARG;
  const size_t need = pa_decode_graphs_workspace_bytes(max_seqs, num_heads, head_dim, max_context_len, seq_interval,
                                                       kv_interval);
  if (need == 0) return PA_ERR_INVALID_ARG;
  if (workspace_bytes < need) return PA_ERR_WORKSPACE;
  int s_pad = 0, c_pad = 0;
  padded_limits(max_seqs, max_context_len, seq_interval, kv_interval, &s_pad, &c_pad);
  // the static buffers must hold the largest padded batch; check every other
  // argument the way pa_decode will
  const int st = pa_host::decode_check(out_buf, out_dtype, q_buf, k_pool, v_pool, tables_buf, max_blocks_per_seq,
                                       ctx_buf, c_pad, s_pad, num_heads, head_dim, block_size, num_blocks, scale,
                                       dtype, workspace, workspace_bytes, 0, err_flag);
  if (st != PA_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return PA_ERR_CUDA;
  pa_decode_graphs* g = new pa_decode_graphs();
  g->out = out_buf;
  g->out_dtype = out_dtype;
  g->q = q_buf;
  g->k_pool = k_pool;
  g->v_pool = v_pool;
  g->tables = tables_buf;
  g->max_blocks_per_seq = max_blocks_per_seq;
  g->ctx = ctx_buf;
  g->max_seqs = s_pad;
  g->max_ctx = c_pad;
  g->num_heads = num_heads;
  g->head_dim = head_dim;
  g->block_size = block_size;
  g->num_blocks = num_blocks;
  g->scale = scale;
  g->dtype = dtype;
  g->workspace = workspace;
  g->workspace_bytes = workspace_bytes;
  g->seq_interval = seq_interval;
  g->kv_interval = kv_interval;
  g->err_flag = err_flag;
  g->device = dev;
  g->capture_stream = cs;
  *out = g;
  return PA_OK;
}

void pa_decode_graphs_destroy(pa_decode_graphs* g) {
  if (g == nullptr) return;
  for (auto& kv : g->graphs) cudaGraphExecDestroy(kv.second);
  cudaStreamDestroy(g->capture_stream);
  delete g;
}

int pa_decode_graphs_count(const pa_decode_graphs* g) { return g ? (int)g->graphs.size() : -1; }

int pa_decode_graphs_run(pa_decode_graphs* g, int num_seqs, int max_context_len, void* stream) {
  pa_host::Range range("pa_decode_graphs_run");
  if (g == nullptr || num_seqs < 0 || max_context_len < 0) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  const int s_pad = round_up(num_seqs, g->seq_interval);
  const int c_pad = round_up(max_context_len > 0 ? max_context_len : 1, g->kv_interval);
  if (s_pad > g->max_seqs || c_pad > g->max_ctx) return PA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != g->device) return PA_ERR_CUDA;
  const std::pair<int, int> key(s_pad, c_pad);
  auto it = g->graphs.find(key);
  if (it == g->graphs.end()) {
    // record pa_decode for this padded shape on the object's own stream
    cudaStream_t cs = g->capture_stream;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) return PA_ERR_CUDA;
    const int st = pa_decode(g->out, g->out_dtype, g->q, g->k_pool, g->v_pool, g->tables, g->max_blocks_per_seq,
                             g->ctx, c_pad, s_pad, g->num_heads, g->head_dim, g->block_size, g->num_blocks, g->scale,
                             g->dtype, g->workspace, g->workspace_bytes, 0, g->err_flag, cs);
    cudaGraph_t graph = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(cs, &graph);
    if (st != PA_OK || ce != cudaSuccess || graph == nullptr) {
      if (graph) cudaGraphDestroy(graph);
      cudaGetLastError();
      return st != PA_OK ? st : PA_ERR_CUDA;
    }
    cudaGraphExec_t exec = nullptr;
    const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ie != cudaSuccess || exec == nullptr) return PA_ERR_CUDA;
    it = g->graphs.emplace(key, exec).first;
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (s_pad > num_seqs &&
      cudaMemsetAsync(g->ctx + num_seqs, 0, sizeof(int32_t) * (size_t)(s_pad - num_seqs), s) != cudaSuccess)
    return PA_ERR_CUDA;
  return cudaGraphLaunch(it->second, s) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"
