/*
 * pa.h -- C ABI of libpa: paged KV-cache attention for one NVIDIA GB300
 * (sm_103a).
 *
 * Sources of the operations (the method is PagedAttention, "Efficient
 * Memory Management for Large Language Model Serving with PagedAttention";
 * three pages describe it):
 *   [summary]  paper-summary page of that title (urban-dandelion.tistory.com/4)
 *   [blog]     "SOSP 2023論文解説: vLLM — PagedAttentionによるKVキャッシュメモリ管理の革新"
 *   [cb]       "연속 배치 처리 아키텍처" (continuous-batching architecture page)
 *
 * Conventions shared by every call
 * --------------------------------
 *  - KV pools: two arrays, K and V, each [num_blocks][num_heads][block_size][head_dim]
 *    of fp16 or bf16, row-major.  One (block, head) tile is contiguous.
 *  - Positions are 0-based: token p of a sequence sits in logical block p / B,
 *    slot p % B; the block table maps logical block i to a physical block
 *    ([summary] section 4: 1-based token j in block floor((j-1)/B), slot
 *    (j-1) mod B).  A "slot" index is physical_block * B + slot.
 *  - Block tables: int32 [rows][max_blocks_per_seq], row-major, device memory.
 *    Only the entries that cover a sequence's tokens are read.
 *  - dtype codes: PA_F16, PA_BF16 for q/K/V; outputs may also be PA_F32.
 *  - head_dim must be 64 or 128; block_size a multiple of 16 (16..65536).
 *  - Device pointers are plain CUDA device addresses owned by the caller;
 *    the library allocates no device memory and keeps no device state.
 *    `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *    Every launch is asynchronous on that stream.
 *  - Return value: PA_OK, or an error code for bad arguments detected on the
 *    host before anything is launched (nothing is launched then).
 *  - Device-side problems (a table entry outside the pool, a slot outside the
 *    pool, a context longer than its table, a wait that ran out of time) never
 *    trap: the kernel ORs a PA_FLAG_* bit into the caller's int32 `err_flag`
 *    (device memory, zero-initialised by the caller) and skips the bad work.
 *    pa_get_error() reads and clears it.
 *  - Threads: every kernel entry point may be called from several host
 *    threads at once (on one device or several); the library's only
 *    process-wide state is a per-device cache of kernel settings, filled
 *    idempotently.  Allocator handles and decode-graph objects are not
 *    thread-safe: one per thread, or lock around them.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------------- */
#define PA_OK 0
#define PA_ERR_INVALID_ARG 1    /* null pointer, bad size, misaligned pointer */
#define PA_ERR_UNSUPPORTED 2    /* dtype, head_dim or block_size not supported */
#define PA_ERR_NO_FREE_BLOCKS 3 /* allocator: pool exhausted ([blog] MemoryError) */
#define PA_ERR_REFCOUNT 4       /* allocator: reference count would go below 0 */
#define PA_ERR_BAD_INDEX 5      /* device flag: block / slot / length out of range */
#define PA_ERR_CUDA 6           /* a CUDA runtime call failed */
#define PA_ERR_TIMEOUT 7        /* device flag: a bounded wait ran out of time */
#define PA_ERR_WORKSPACE 8      /* workspace too small */

/* ---- dtypes ------------------------------------------------------------------------ */
#define PA_F16 0
#define PA_BF16 1
#define PA_F32 2

/* ---- device error-flag bits ---------------------------------------------------------- */
#define PA_FLAG_BAD_BLOCK 1   /* block-table entry or copy pair outside [0, num_blocks) */
#define PA_FLAG_BAD_SLOT 2    /* slot_mapping entry >= num_blocks * block_size */
#define PA_FLAG_BAD_LENGTH 4  /* context length < 0, > max_context_len, or > table capacity */
#define PA_FLAG_TIMEOUT 8     /* an mbarrier wait exceeded its time limit */
#define PA_FLAG_BAD_GROUP 16  /* pa_decode_grouped: a group was not usable; its sequences were decoded whole */

/* Library version (major*10000 + minor*100 + patch). */
int pa_version(void);

/* Human-readable name of a status code (static string). */
const char* pa_status_string(int status);

/* Number of multiprocessors of the current device (0 if no device). */
int pa_device_sm_count(void);

/*
 * pa_reshape_and_cache -- slot-scatter write of new K/V into the paged pools.
 * [blog] "アルゴリズムの擬似コード": append_token stores the token's k and v in
 * slot num_filled of the sequence's last block.  Here the caller gives each
 * token's slot directly:
 *   for t in [0, num_tokens), slot = slot_mapping[t]:
 *     slot < 0  -> token skipped (padding);
 *     otherwise K_pool[slot / B][h][slot % B][:] = k_new[t][h][:] for every head h,
 *               and the same for V (bit copy).
 * k_new, v_new: device [num_tokens][num_heads][head_dim], dtype `dtype`.
 * slot_mapping: device int64 [num_tokens].  Slots must be distinct (else the
 * result for the repeated slot is one of the writers).  A slot >= num_blocks*B
 * sets PA_FLAG_BAD_SLOT and that token is skipped.  num_tokens == 0 is a no-op.
 * A kernel launched behind it with programmatic stream serialization may
 * start while it runs and must wait (griddepcontrol.wait) before reading the
 * pools.
 */
int pa_reshape_and_cache(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                         const int64_t* slot_mapping, int num_tokens, int num_heads, int head_dim,
                         int block_size, int num_blocks, int dtype, int32_t* err_flag, void* stream);

/*
 * pa_copy_blocks -- copy-on-write block copy.
 * [blog] "アルゴリズムの擬似コード" copy_on_write: the new block receives a copy of the
 * whole source block's K and V ([summary] section 6, parallel sampling).
 *   for i in [0, n_pairs): (src, dst) = (pairs[2i], pairs[2i+1]):
 *     K_pool[dst][:][:][:] = K_pool[src][:][:][:], same for V (all heads, all slots).
 * pairs: device int32 [n_pairs][2].  No block may be both a source and a
 * destination, and destinations must be distinct (pairs are applied
 * concurrently).  An id outside [0, num_blocks) sets PA_FLAG_BAD_BLOCK and that
 * pair is skipped.  n_pairs == 0 is a no-op.
 */
int pa_copy_blocks(void* k_pool, void* v_pool, const int32_t* pairs, int n_pairs, int num_heads,
                   int head_dim, int block_size, int num_blocks, int dtype, int32_t* err_flag, void* stream);

/*
 * pa_swap_blocks -- move whole blocks between two pools, one of which may be
 * a pinned host pool: swap-out of a preempted request's blocks to CPU memory
 * and swap-in when it resumes.
 * [summary] section 5: under memory pressure the preemptive scheduler swaps
 * some sequences' KV blocks to CPU memory (or recomputes them), and Figure 26
 * compares the two by block size; [cb] "오프로딩" (offloading): the request's
 * KV blocks are copied into a pre-allocated pinned CPU buffer, every request
 * that fits the swap pool in one batched transfer, and copied back to the GPU
 * when space frees up.
 *   for i in [0, n_pairs): (s, d) = (pairs[2i], pairs[2i+1]):
 *     dst_K[d][:][:][:] = src_K[s][:][:][:], same for V (all heads, all slots).
 * src_k, src_v: the source pool [src_num_blocks][num_heads][block_size][head_dim];
 * dst_k, dst_v: the destination pool [dst_num_blocks][...], same shape per block
 * and dtype.  Each pool is either device memory or pinned host memory that
 * the GPU can address (cudaHostAlloc / cudaMallocHost, or cudaHostRegister
 * with cudaHostRegisterMapped; with unified addressing the host address is
 * the device address).  The copy is one kernel launch for the whole batch:
 * the GPU reads and writes the host pool directly over the CPU-GPU link, so
 * neither the block size nor the scattering of the block ids adds a per-copy
 * cost.  Bit-exact.
 * pairs: device int32 [n_pairs][2], n_pairs <= 65535.  Destinations must be
 * distinct and, when both pools are the same memory, disjoint from the
 * sources.  An id outside its pool sets PA_FLAG_BAD_BLOCK and that pair is
 * skipped.  n_pairs == 0 is a no-op.  The host pool must stay pinned until
 * the stream has passed the call.
 */
int pa_swap_blocks(const void* src_k, const void* src_v, int src_num_blocks, void* dst_k, void* dst_v,
                   int dst_num_blocks, const int32_t* pairs, int n_pairs, int num_heads, int head_dim,
                   int block_size, int dtype, int32_t* err_flag, void* stream);

/*
 * Split-KV partition length (tokens) that pa_decode uses when called with
 * partition_size == 0, chosen from the batch shape alone (no device query):
 * with pairs = num_seqs * num_heads and units(P) = pairs *
 * ceil(max_context_len / P), it is 1024 when pairs >= 380 and either
 * max_context_len <= 1024 or units(1024) >= 12160 (16 waves of a 152-SM x
 * 5-CTA grid); otherwise the largest of 512, 256, 128 with units(P) >= 380
 * (half a wave), else 64.  512 when an argument is not positive.
 */
int pa_decode_partition_size(int num_seqs, int num_heads, int max_context_len);

/*
 * Bytes of device workspace pa_decode needs for these sizes (partition_size 0 =
 * the automatic choice above).  0 on bad arguments.
 */
size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                 int partition_size);

/*
 * pa_decode -- single-query paged decode attention.
 * [summary] section 4 equation and Figure 6; [blog] "Attention計算の修正":
 *   for each sequence s and head h, with n = context_lens[s]:
 *     x_j = scale * q[s][h] . K_s[j],  j in [0, n), K_s[j] = K_pool[table[s][j/B]][h][j%B]
 *     out[s][h] = sum_j softmax(x)_j V_s[j]
 * computed block by block with an online softmax inside each split-KV
 * partition and a log-sum-exp combine of the partitions (in token order, so
 * the result is deterministic).  A sequence is cut into partitions of
 * `partition_size` tokens (the last one partial).  n == 0 gives a zero row.
 * q: device [num_seqs][num_heads][head_dim], dtype `dtype`.
 * out: device [num_seqs][num_heads][head_dim], dtype `out_dtype`.
 * context_lens: device int32 [num_seqs], each <= max_context_len and
 *   <= max_blocks_per_seq * block_size (else PA_FLAG_BAD_LENGTH, zero row).
 * workspace: device memory of at least pa_decode_workspace_bytes(...) bytes,
 *   16-byte aligned; no initial contents required; not to be shared by two
 *   pa_decode calls that may run at the same time.
 * partition_size: 0 = automatic, else a multiple of 16 in [16, 1024];
 *   ceil(max_context_len / partition) must stay below 2^20 (up to 2^24
 *   tokens at partition 16, 2^30 at 1024), else PA_ERR_UNSUPPORTED.
 * A table entry outside [0, num_blocks) sets PA_FLAG_BAD_BLOCK; the 16-token
 * chunk it covers is left out of that sequence's sum.
 * Launches: a one-CTA planning kernel, then the persistent decode kernel, on
 * `stream`, each a programmatic dependent of the kernel before it: the
 * planning (which reads only context_lens and writes only out rows of empty
 * sequences and the workspace) may overlap a previous kernel that releases
 * its dependents early, and completes only after that kernel has; the decode
 * kernel waits for the planning kernel before reading anything.
 */
int pa_decode(void* out, int out_dtype, const void* q, const void* k_pool, const void* v_pool,
              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
              int max_context_len, int num_seqs, int num_heads, int head_dim, int block_size,
              int num_blocks, float scale, int dtype, void* workspace, size_t workspace_bytes,
              int partition_size, int32_t* err_flag, void* stream);

/*
 * Bytes of device workspace pa_decode_grouped needs for these sizes
 * (partition_size 0 = the automatic choice above).  0 on bad arguments.
 */
size_t pa_decode_grouped_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                         int partition_size);

/*
 * pa_decode_grouped -- pa_decode for a batch in which groups of sequences
 * share the blocks of a common prefix: the parallel samples or the beams of
 * one prompt ([summary] section 6, parallel sampling (Figure 9) and beam
 * search (Figure 10); [blog] "Prefix Sharing").  The outputs are those of pa_decode (the same
 * equation; the rounding order differs).  Each shared prefix is read from the
 * pool once for its whole group instead of once per sequence.
 * Arguments are those of pa_decode, plus:
 * group_start: device int32 [num_groups + 1]; group g is sequences
 *   group_start[g] .. group_start[g+1] - 1 (at most 8, at least 1), so groups
 *   are disjoint ranges of the batch in order; a sequence outside every group
 *   is decoded on its own.
 * group_prefix: device int32 [num_groups], a multiple of 16; the tokens
 *   [0, group_prefix[g]) of every member of group g are the same K/V: every
 *   member's table holds the first member's block ids over those tokens'
 *   blocks, and the prefix is at most every member's context length.  A
 *   group that breaks a rule (or whose range or size is out of bounds) sets
 *   PA_FLAG_BAD_GROUP and its members are decoded on their own; the results
 *   are still correct.  pa_alloc_prefix_groups computes groups from the host
 *   allocator's tables.
 * num_groups: >= 0 (0 = pa_decode).
 * workspace: at least pa_decode_grouped_workspace_bytes(...) bytes.
 * Launches on `stream`: the planning kernel (as in pa_decode; it also
 *   validates the groups and lists every sequence's own tokens past its
 *   group's prefix), then the group kernel, persistent, whose warps take
 *   first the prefix units (group, head, partition of the prefix: each
 *   16-token tile's K and V are multiplied with all the group's queries on
 *   the tensor cores) and then the listed items (one sequence, one head);
 *   the partitions of each (sequence, head) are merged by log-sum-exp as in
 *   pa_decode.
 */
int pa_decode_grouped(void* out, int out_dtype, const void* q, const void* k_pool, const void* v_pool,
                      const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                      int max_context_len, int num_seqs, int num_heads, int head_dim, int block_size,
                      int num_blocks, float scale, int dtype, const int32_t* group_start,
                      const int32_t* group_prefix, int num_groups, void* workspace, size_t workspace_bytes,
                      int partition_size, int32_t* err_flag, void* stream);

/*
 * pa_decode_static_scratch -- pa_decode without any device allocation by
 * anyone.  The paper has no counterpart: this is an interface of this
 * library only.
 *
 * pa_decode needs a few megabytes of device scratch (the work list and the
 * split-KV partials) that its caller normally allocates.  Some callers cannot
 * do that: a plugin that is handed only its input and output buffers by a
 * host framework owning all device memory, or code on a latency-critical path
 * where cudaMalloc / cudaFree would implicitly synchronise the device.  This
 * entry point takes the same arguments as pa_decode minus the workspace and
 * uses instead a fixed array of PA_DECODE_STATIC_SCRATCH_BYTES (16 MiB) that
 * lives in the library's device code and stays resident on every GPU that
 * loads the library until the process exits.
 *  - Limit: if pa_decode_workspace_bytes() for these sizes exceeds
 *    PA_DECODE_STATIC_SCRATCH_BYTES, it returns PA_ERR_WORKSPACE and launches
 *    nothing (the LLaMA-13B-shaped batch of 64 sequences x 40 heads with
 *    contexts up to 2048 needs about 5.3 MiB; 256 x 32 heads with contexts up
 *    to 16384 does not fit and must use pa_decode).
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  Nothing is allocated, then or later.
 *  - Every call on a device shares the one array and leaves its contents
 *    behind; no initial contents are needed (each call's planning kernel
 *    resets the counters it uses).  Calls that can overlap on the GPU (other
 *    streams, other threads) race on the array: serialise them.
 */
#define PA_DECODE_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
int pa_decode_static_scratch(void* out, int out_dtype, const void* q, const void* k_pool, const void* v_pool,
                             const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                             int max_context_len, int num_seqs, int num_heads, int head_dim, int block_size,
                             int num_blocks, float scale, int dtype, int partition_size, int32_t* err_flag,
                             void* stream);

/*
 * pa_prefill_chunk -- causal attention of prefill chunks over paged K/V.
 * [cb] "Chunked prefill": a long prompt is split into chunks processed over
 * several steps; [summary] section 4 equation, causal j <= i.
 *   chunk c holds query rows cu_q_lens[c] .. cu_q_lens[c+1]-1 of q; its row i
 *   sits at position ctx_before[c] + i of sequence c (block_tables row c) and
 *   attends positions 0 .. ctx_before[c] + i.  The chunk's own K/V must already
 *   be in the pools (pa_reshape_and_cache).
 * q, out: device [total_q][num_heads][head_dim]; q in `dtype`, out in `out_dtype`.
 * cu_q_lens: device int32 [num_chunks + 1], cu_q_lens[0] == 0, non-decreasing.
 * ctx_before: device int32 [num_chunks].
 * total_q: number of rows of q and out (== cu_q_lens[num_chunks]).
 * max_q_len: host upper bound of any chunk's length (sizes the work list).
 * Requires head_dim 64 or 128 and block_size a multiple of 16 (up to 65536).  Runs on the tensor cores (tcgen05.mma, accumulators
 * in tensor memory, tiles moved by TMA).  A chunk whose context runs past
 * its table sets PA_FLAG_BAD_LENGTH and is skipped; a table entry outside the
 * pool sets PA_FLAG_BAD_BLOCK and its tokens are left out.
 * Persistent grid (one CTA per SM).  A kernel launched behind it with
 * programmatic stream serialization may start while it runs and must wait
 * (griddepcontrol.wait) before reading its output.
 */
int pa_prefill_chunk(void* out, int out_dtype, const void* q, const int32_t* cu_q_lens,
                     const int32_t* ctx_before, const void* k_pool, const void* v_pool,
                     const int32_t* block_tables, int max_blocks_per_seq, int num_chunks, int total_q,
                     int max_q_len, int num_heads, int head_dim, int block_size, int num_blocks, float scale,
                     int dtype, int32_t* err_flag, void* stream);

/*
 * pa_mixed_step -- one step of a mixed batch: decode of num_seqs sequences
 * and prefill of num_chunks chunks over the same pools, run concurrently.
 * [cb] "Chunked prefill" and its scheduler: a step's token budget holds the
 * running requests' decode tokens and prefill chunks together and runs them
 * as one forward pass.
 *  - dec_* and the decode arguments are those of pa_decode (partition size
 *    chosen automatically); pf_* and the chunk arguments those of
 *    pa_prefill_chunk; pools, num_heads, head_dim, block_size, num_blocks,
 *    scale, dtype and err_flag are shared.
 *  - On `stream`: the decode's planning kernel, then the prefill's persistent
 *    grid on at most `prefill_sms` SMs (<= 0: PA_MIXED_PREFILL_SHARE percent
 *    of them), then the decode kernel as a programmatic dependent of the
 *    prefill: it starts as soon as the prefill's CTAs are resident and fills
 *    the remaining SMs.  Work queued on `stream` afterwards sees both outputs.
 *  - Outputs: the same values as pa_decode and pa_prefill_chunk give.
 *  - All arguments of both parts are checked before anything is launched.
 *    With no chunks it is pa_decode; with no sequences, pa_prefill_chunk.
 */
#define PA_MIXED_PREFILL_SHARE 45
int pa_mixed_step(void* dec_out, int dec_out_dtype, const void* dec_q, const int32_t* dec_block_tables,
                  int dec_max_blocks_per_seq, const int32_t* context_lens, int max_context_len, int num_seqs,
                  void* workspace, size_t workspace_bytes, void* pf_out, int pf_out_dtype, const void* pf_q,
                  const int32_t* cu_q_lens, const int32_t* ctx_before, const int32_t* pf_block_tables,
                  int pf_max_blocks_per_seq, int num_chunks, int total_q, int max_q_len, const void* k_pool,
                  const void* v_pool, int num_heads, int head_dim, int block_size, int num_blocks, float scale,
                  int dtype, int prefill_sms, int32_t* err_flag, void* stream);

/*
 * Decode graphs -- pa_decode recorded once per padded batch shape and
 * replayed.  [cb] "CUDA 그래프": a step's CPU work (batch assembly, kernel
 * dispatch) is removed by recording the GPU work once and replaying it for
 * batches of the same shape; because the shape changes every step, the query
 * count and the KV length are padded up to multiples of fixed intervals, the
 * recorded graphs are cached by padded shape, and a new shape triggers a new
 * recording.
 *
 * The graphs read and write caller-owned STATIC device buffers given at
 * creation, sized for the largest padded batch:
 *   q_buf, out_buf  [S_max][num_heads][head_dim]   (q in dtype, out in out_dtype)
 *   tables_buf      int32 [S_max][max_blocks_per_seq]
 *   ctx_buf         int32 [S_max]
 *   workspace       pa_decode_graphs_workspace_bytes(...) bytes, 16-byte aligned
 * with S_max = max_seqs rounded up to seq_interval.  The pools, scale, dtype
 * and err_flag are fixed at creation too.  Per step the caller writes rows
 * 0 .. num_seqs-1 of q_buf, tables_buf and ctx_buf (on the stream it passes
 * to _run, or before), then calls _run(num_seqs, max_context_len): the
 * shape is padded to (num_seqs up to a multiple of seq_interval,
 * max_context_len up to a multiple of kv_interval), ctx_buf rows num_seqs ..
 * padded-1 are zeroed on the stream (zero output rows), and the graph of that
 * padded shape is replayed on the stream -- recorded first, on a stream of the
 * object's own, if the shape is new.  Rows 0 .. num_seqs-1 of out_buf then
 * hold what pa_decode(..., num_seqs = padded, max_context_len = padded)
 * gives.  Shapes beyond the creation maxima: PA_ERR_INVALID_ARG.
 * The object holds host state only (no device memory); it is not thread-safe
 * and must be used on the device that was current at creation.
 */
typedef struct pa_decode_graphs pa_decode_graphs;
size_t pa_decode_graphs_workspace_bytes(int max_seqs, int num_heads, int head_dim, int max_context_len,
                                        int seq_interval, int kv_interval);
int pa_decode_graphs_create(void* out_buf, int out_dtype, const void* q_buf, const void* k_pool,
                            const void* v_pool, const int32_t* tables_buf, int max_blocks_per_seq,
                            int32_t* ctx_buf, int max_seqs, int max_context_len, int num_heads, int head_dim,
                            int block_size, int num_blocks, float scale, int dtype, void* workspace,
                            size_t workspace_bytes, int seq_interval, int kv_interval, int32_t* err_flag,
                            pa_decode_graphs** out);
int pa_decode_graphs_run(pa_decode_graphs* g, int num_seqs, int max_context_len, void* stream);
int pa_decode_graphs_count(const pa_decode_graphs* g); /* graphs recorded so far */
void pa_decode_graphs_destroy(pa_decode_graphs* g);

/*
 * Host-side validation of the inputs the kernels index with (a debug aid).
 * The kernels never trap on a bad block-table entry or length: they set a
 * PA_FLAG_* bit and skip the work.  These calls find the first bad entry
 * instead: they copy the tables and lengths to the host, SYNCHRONISE `stream`,
 * and check exactly the entries the kernels would read (the ceil(len / B)
 * entries of each row; [summary] section 4 block mapping).
 *  - decode: context_lens[s] in [0, max_context_len] and <= max_blocks_per_seq
 *    * block_size; entries 0 .. ceil(len/B)-1 of row s in [0, num_blocks).
 *  - prefill: cu_q_lens[0] == 0, cu_q_lens[num_chunks] == total_q, chunk
 *    lengths in [0, max_q_len], ctx_before[c] >= 0, ctx_before[c] + length
 *    within the table row, entries covering it in [0, num_blocks).
 * Return PA_OK or PA_ERR_BAD_INDEX; bad_out (int64[2], may be NULL) receives
 * (row, logical block) of the first bad entry, logical block -1 for a bad
 * length, (-1, -1) for bad cu_q_lens ends or when all is well.
 * With the environment variable PA_DEBUG set (not "0"), pa_decode,
 * pa_prefill_chunk and pa_mixed_step run these checks before launching and
 * return PA_ERR_BAD_INDEX (nothing launched, a line on stderr) on a bad entry.
 * Every GPU entry point also opens an NVTX range named after itself.
 */
int pa_check_decode_inputs(const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                           int num_seqs, int max_context_len, int block_size, int num_blocks, void* stream,
                           int64_t* bad_out);
int pa_check_prefill_inputs(const int32_t* cu_q_lens, const int32_t* ctx_before, const int32_t* block_tables,
                            int max_blocks_per_seq, int num_chunks, int total_q, int max_q_len, int block_size,
                            int num_blocks, void* stream, int64_t* bad_out);

/*
 * pa_selftest_wait_timeout -- exercises the bounded wait every kernel uses;
 * the paper has no counterpart.  One CTA copies 4 KiB from `src` (device,
 * 16-byte aligned) into shared memory with a bulk copy, then waits on an
 * mbarrier that nothing arrives at.  After the kernels' wait limit (1 s) the
 * wait gives up and sets PA_FLAG_TIMEOUT in *err_flag; the CTA then lets its
 * own copy land and exits normally, leaving the context usable.  result
 * (device int32[3]) receives: the wait's success (0 expected), whether the
 * copy landed (1), and the copy's last 32-bit word.
 */
int pa_selftest_wait_timeout(const void* src, int32_t* err_flag, int32_t* result, void* stream);

/*
 * pa_get_error -- synchronise `stream`, read the device error flag, clear it.
 * Returns PA_OK, PA_ERR_TIMEOUT (if PA_FLAG_TIMEOUT is set), PA_ERR_BAD_INDEX
 * (any other flag) or PA_ERR_CUDA.  If flags_out is non-null it receives the
 * raw flag bits.
 */
int pa_get_error(int32_t* err_flag, int32_t* flags_out, void* stream);

/*
 * pa_slot_mapping -- host-side slot computation for tokens of sequences whose
 * block tables the caller already holds (the allocator below does this itself
 * for the tokens it appends).  [summary] section 4 block mapping:
 *   slots_out[i] = table[seq_idx[i]][pos[i] / B] * B + pos[i] % B
 * All arrays are host memory; table is [num_rows][max_blocks_per_seq].
 * A position whose table entry is negative or beyond max_blocks_per_seq gives
 * PA_ERR_BAD_INDEX (slots before it are written).
 */
int pa_slot_mapping(const int32_t* table, int num_rows, int max_blocks_per_seq, int block_size,
                    const int32_t* seq_idx, const int32_t* pos, int n, int64_t* slots_out);

/* ---- host block allocator (no CUDA; never on the GPU path) ---------------------
 * The block manager of [blog] "アルゴリズムの擬似コード" and [summary] sections 5-6:
 *  - free list initialised to 0..N-1; a block is taken from its END (the first
 *    block handed out is N-1); taking from an empty list -> PA_ERR_NO_FREE_BLOCKS;
 *  - a taken block has reference count 1; releasing decrements; at 0 the block
 *    is appended to the free list;
 *  - append one token: no block yet -> take one; last block full -> take a new
 *    one; else last block shared (count > 1) -> copy-on-write: take a new block,
 *    record (old, new) as a copy pair, drop one reference of the old block and
 *    put the new block in its place.  The token's slot is (last block)*B + len%B.
 *  - fork: the child gets the parent's blocks and length; each block +1 reference;
 *  - free: releases the sequence's blocks in logical order.
 * A handle is not thread-safe; use one per thread or lock around it.
 */
typedef struct pa_alloc pa_alloc;

int pa_alloc_create(int num_blocks, int block_size, pa_alloc** out);
void pa_alloc_destroy(pa_alloc* a);

/*
 * Prefix caching ([cb] "Prefix 캐싱" and "제거" (eviction)): requests whose
 * prompts share a prefix share the blocks that hold it.
 *  - PA_ALLOC_PREFIX_CACHE in pa_alloc_create_ex's flags turns it on (without
 *    it the calls below behave like add_seq / append_slots and reuse nothing).
 *  - A sequence created by pa_alloc_add_seq_prefix and extended only through
 *    pa_alloc_append_tokens has known token ids.  Each of its blocks that
 *    becomes full is keyed by its whole prefix (the ids from position 0 to the
 *    block's end) unless that prefix already has a block.
 *  - pa_alloc_add_seq_prefix(tokens[0..n)) walks the prompt's full blocks from
 *    the first: while the block's prefix has a cached block, that block joins
 *    the new sequence (+1 reference).  *n_reused_tokens = the tokens covered
 *    (a multiple of B): their K/V are already in the pool, so the prefill
 *    starts after them; the remaining prompt tokens are appended with
 *    pa_alloc_append_tokens.
 *  - A block whose last reference goes keeps its content and key
 *    ("initialized") and still matches.  When a block must be taken and no
 *    block without content is free, the most recently freed initialized block
 *    loses its key and is taken.  pa_alloc_num_free counts both kinds.
 *  - pa_alloc_append_slots on such a sequence (ids unknown) ends its caching.
 *  - Keys are 128-bit chained fingerprints of the prefix ids; a match also
 *    compares the block's own ids.
 */
#define PA_ALLOC_PREFIX_CACHE 1
int pa_alloc_create_ex(int num_blocks, int block_size, int flags, pa_alloc** out);
int pa_alloc_add_seq_prefix(pa_alloc* a, int seq_id, const int32_t* tokens, int n_tokens, int* n_reused_tokens);
/* pa_alloc_append_slots with the appended tokens' ids (token_ids int32 [n]). */
int pa_alloc_append_tokens(pa_alloc* a, const int* seq_ids, const int32_t* token_ids, int n, int64_t* slots_out,
                           int32_t* copy_pairs_out, int* n_pairs_out);
/* Blocks holding a cache entry, and how many of them are free (initialized). */
int pa_alloc_prefix_stats(const pa_alloc* a, int* cached_blocks, int* initialized_free_blocks);
/* New empty sequence.  PA_ERR_INVALID_ARG if seq_id exists or is negative. */
int pa_alloc_add_seq(pa_alloc* a, int seq_id);
/* child shares all of parent's blocks.  PA_ERR_INVALID_ARG if parent missing / child exists. */
int pa_alloc_fork(pa_alloc* a, int parent, int child);
/*
 * One new token for each of the n distinct listed sequences, in list order.
 * slots_out: int64 [n].  copy_pairs_out: int32 [2*n] capacity; receives the
 * (src, dst) copy-on-write pairs in order, their count in *n_pairs_out.
 * All-or-nothing: PA_ERR_NO_FREE_BLOCKS leaves the allocator unchanged.
 */
int pa_alloc_append_slots(pa_alloc* a, const int* seq_ids, int n, int64_t* slots_out,
                          int32_t* copy_pairs_out, int* n_pairs_out);
int pa_alloc_free_seq(pa_alloc* a, int seq_id);
/* Copy seq's block ids into out[0..cap); *n_blocks and *seq_len receive the sizes
 * (PA_ERR_INVALID_ARG if cap is too small; sizes are still reported). */
int pa_alloc_block_table(const pa_alloc* a, int seq_id, int32_t* out, int cap, int* n_blocks, int* seq_len);
/* Fill rows of a padded table: row i = seq_ids[i]'s blocks, padded with -1 up to
 * max_blocks_per_seq; ctx_lens_out[i] = its length (either output may be NULL). */
int pa_alloc_block_tables(const pa_alloc* a, const int* seq_ids, int n, int max_blocks_per_seq,
                          int32_t* tables_out, int32_t* ctx_lens_out);
/* Groups for pa_decode_grouped over the batch seq_ids[0..n) in that order:
 * runs of consecutive sequences (at most max_group, 1..8) whose tables start
 * with the same block.  A run grows while the next sequence shares at least
 * its first full block with the run's first sequence; its prefix is, in
 * tokens, the leading blocks that every member holds in common with the first
 * and has filled (length >= (b + 1) * block_size), rounded down to a multiple
 * of 16; a run of one has prefix 0.  Writes group_start_out[0..G] (host int32,
 * room for n + 1) and group_prefix_out[0..G) (room for n), *num_groups_out =
 * G.  PA_ERR_INVALID_ARG for an unknown id or bad sizes. */
int pa_alloc_prefix_groups(const pa_alloc* a, const int* seq_ids, int n, int max_group, int32_t* group_start_out,
                           int32_t* group_prefix_out, int* num_groups_out);
int pa_alloc_num_free(const pa_alloc* a);
/* Reference count of block_id (-1 if out of range). */
int pa_alloc_ref(const pa_alloc* a, int block_id);
/* Number of live sequences. */
int pa_alloc_num_seqs(const pa_alloc* a);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
