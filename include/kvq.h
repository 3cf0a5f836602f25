/*
 * kvq.h -- C ABI of the GB300 (sm_103a) quantized paged-KV attention library.
 *
 * The library implements the hot path described on three pages about
 * vLLM's quantized KV cache (prhub.com.cn summaries of vLLM pull requests):
 *
 *   [P1] vllm PR 39445 "CPU 后端新增 FP8 KV 缓存量化支持": an fp8 KV cache;
 *        entry points cpu_attn_reshape_and_cache / cpu_attention_with_kv_cache
 *        that take kv_cache_dtype, k_scale and v_scale (Breakdown items 1-4).
 *   [P2] vllm PR 50194 "修复 CPU FP8 注意力调度器临时缓冲区大小计算错误":
 *        get_scheduler_metadata must size its tiles and scratch from the KV
 *        cache element size, not the query's (Motivation, Key source snippet).
 *   [P3] vllm PR 38378 "为 Triton 注意力后端引入 KV 缓存按令牌头 INT8/FP8 量化":
 *        int8 / fp8 per-(token, head) dynamic absmax scales stored inline in a
 *        padded head row (Breakdown item 3, Risks).
 *
 * Conventions for every call:
 *   - Device pointers point to memory of the CUDA device that is current on
 *     the calling thread; host pointers are named *_host.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Kernels are enqueued on it; calls do not synchronise, so a
 *     kernel fault surfaces at the caller's next stream synchronisation.
 *   - The caller owns every buffer it passes.  The library owns only the
 *     kvq_sched_t objects it creates (freed with kvq_sched_destroy).  No call
 *     except kvq_get_scheduler_metadata allocates device memory.
 *   - Every call returns KVQ_OK (0) or a negative KVQ_E_* status; no call
 *     throws, exits or prints.  Arguments are checked on the host before any
 *     launch; a call that returns an error has enqueued nothing.
 *   - bf16 tensors are IEEE bfloat16 bit patterns (uint16), little endian.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of the ABI are exported even when the library is built with
 * hidden default visibility. */
#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

/* ---- status codes ---------------------------------------------------- */
#define KVQ_OK 0
#define KVQ_E_INVALID_ARG (-1)      /* a pointer, size, stride or value is invalid */
#define KVQ_E_UNSUPPORTED (-2)      /* dtype / head_dim / GQA ratio not built      */
#define KVQ_E_SCHED_MISMATCH (-3)   /* sched built for other dtype/heads/head_dim  */
#define KVQ_E_WORKSPACE_TOO_SMALL (-4)
#define KVQ_E_CUDA (-5)             /* a CUDA runtime call or launch failed        */
#define KVQ_E_NO_MEMORY (-6)        /* host or device allocation failed            */
#define KVQ_E_TIMEOUT (-7)          /* a kernel gave up a bounded wait (see below) */

/* ---- KV cache data types -------------------------------------------------
 * 0..2 keep the kv_cache_dtype indices printed in [P2]'s source snippet
 * ("0 = kAuto, 1 = kFp8E4M3, 2 = kFp8E5M2"); 3 and 4 are [P3]'s modes.
 *
 *   KVQ_AUTO                 bf16 cache, row = 2*D bytes (no quantisation)
 *   KVQ_FP8_E4M3             OCP E4M3FN codes, per-tensor scale, row = D bytes
 *   KVQ_FP8_E5M2             OCP E5M2 codes, per-tensor scale, row = D bytes
 *   KVQ_INT8_PER_TOKEN_HEAD  int8 codes + inline fp32 scale, row = D+16 bytes
 *   KVQ_FP8_PER_TOKEN_HEAD   E4M3FN codes + inline fp32 scale, row = D+16 bytes
 *   KVQ_FP8_E5M2_PER_TOKEN_HEAD  E5M2 codes + inline fp32 scale, row = D+16
 *                            bytes: [P3]'s per-token-head scaling with the
 *                            other fp8 format (its Risks name other scale
 *                            granularities as the next modes)
 *
 * Per-token-head row layout: [D codes][scale: little-endian fp32][12 zero
 * bytes]; the 16-byte pad keeps every row 16-byte aligned.
 */
typedef enum {
  KVQ_AUTO = 0,
  KVQ_FP8_E4M3 = 1,
  KVQ_FP8_E5M2 = 2,
  KVQ_INT8_PER_TOKEN_HEAD = 3,
  KVQ_FP8_PER_TOKEN_HEAD = 4,
  KVQ_FP8_E5M2_PER_TOKEN_HEAD = 5
} kvq_dtype_t;

/* Opaque schedule (work list + sizes), owned by the library. */
typedef struct kvq_sched kvq_sched_t;

/* Parse a kv_cache_dtype string.  Accepts "auto" (the default of [P2]
 * Breakdown item 2), "fp8" (alias of fp8_e4m3), "fp8_e4m3", "fp8_e5m2",
 * "int8_per_token_head", "fp8_per_token_head", "fp8_e5m2_per_token_head".
 * s == NULL or "" reads as
 * "auto".  Unknown strings: KVQ_E_INVALID_ARG. */
KVQ_API int kvq_parse_kv_cache_dtype(const char* s, kvq_dtype_t* out);

/* Bytes of one (token, kv_head) cache row: 2*D (AUTO), D (per-tensor fp8)
 * or D+16 (per-token-head).  [P3] Risks: the per-token-head scale is stored
 * inline by padding the head size (here by 16 bytes: the fp32 scale and 12
 * zero bytes, so every row stays 16-byte aligned); [P1] Risks: an fp8 row
 * is half the bytes of a bf16 one.  head_dim must be a positive multiple
 * of 16; KVQ_E_INVALID_ARG otherwise, or for an unknown dtype. */
KVQ_API int kvq_cache_row_bytes(kvq_dtype_t dtype, int head_dim, size_t* out);

/* reshape_and_cache -- quantise new K/V tokens into the paged caches.
 * [P1] Breakdown item 1 (the reshape kernel writing the fp8 cache) and
 * Key files (cpu_attn_reshape_and_cache); [P3] Breakdown item 3
 * (_reshape_cache_per_token_head: dynamic per-(token, head) absmax scale).
 *
 *   key, value        device bf16 [num_tokens, num_heads_kv, head_dim]; heads
 *                     and dims contiguous; token stride given in elements
 *                     (key_stride_tok, value_stride_tok >= Hkv*D, multiples
 *                     of 8); base pointers 16-byte aligned.
 *   key_cache,        device uint8 [num_blocks, block_size, num_heads_kv, row]
 *   value_cache       with row = kvq_cache_row_bytes(dtype, head_dim);
 *                     16-byte aligned.
 *   slot_mapping      device int64 [num_tokens]: token t goes to block
 *                     slot/block_size, position slot%block_size.  Slots < 0
 *                     or >= num_blocks*block_size are skipped (nothing is
 *                     written for that token).
 *   dtype             any kvq_dtype_t.
 *   k_scale, v_scale  per-tensor scales (fp8_e4m3 / fp8_e5m2): code =
 *                     fp8(x / scale) with a correctly rounded fp32 division,
 *                     round-to-nearest-even and saturation to +-448 (e4m3) /
 *                     +-57344 (e5m2).  Must be finite and > 0 for those
 *                     dtypes; ignored otherwise.
 * Per-token-head: s = amax/qmax in fp32 (qmax 127 for int8, 448 for fp8
 * e4m3, 57344 for fp8 e5m2),
 * code = Q(x / s) (int8: round half to even, clamp [-128,127]); s == 0 gives
 * zero codes.  Inputs must be finite.  num_tokens == 0 is a no-op. */
KVQ_API int kvq_reshape_and_cache(const void* key, const void* value,
                          int64_t num_tokens, int64_t key_stride_tok,
                          int64_t value_stride_tok, int num_heads_kv,
                          int head_dim, void* key_cache, void* value_cache,
                          int64_t num_blocks, int block_size,
                          const int64_t* slot_mapping, kvq_dtype_t dtype,
                          float k_scale, float v_scale, void* stream);

/* get_scheduler_metadata -- plan one attention call (host only).
 * [P2] Breakdown item 1 and Key source snippet: the scheduler takes
 * kv_cache_dtype so that its tile and scratch sizes come from the KV cache
 * element size that the kernels use.
 *
 *   num_req                 requests in the batch (>= 0)
 *   heads_q, heads_kv       heads_q % heads_kv == 0
 *   head_dim                64, 128 or 256
 *   seq_lens_host           host int32 [num_req]: kv length L of each request
 *   query_start_loc_host    host int32 [num_req+1], non-decreasing, [0] == 0;
 *                           request r has Q = qsl[r+1]-qsl[r] <= L queries,
 *                           the last Q positions of its L-token context.
 *   causal, window          window > 0 keeps keys with p - j < window (the
 *                           query's own position included); window <= 0 is
 *                           off.  A window needs causal != 0.
 *   dtype                   the KV cache dtype the attention call will read.
 *   out                     receives a new schedule (free: kvq_sched_destroy)
 *   workspace_bytes         receives the scratch size the attention call
 *                           needs (may be 0); must not be NULL.
 * The schedule holds its plan in pinned host memory and reserves a device
 * buffer for it on the current device (both pooled: after the first few
 * schedules no call allocates).  This call does not touch the device
 * otherwise and does not synchronise: the first attention call made with
 * the schedule uploads the plan with an asynchronous copy on that call's
 * stream, ahead of its kernels.  Requests with at most 16
 * (query, head) rows per kv head (decodes) form row tiles whose 16-token KV
 * chunks are cut into equal contiguous segments, one per warp, so long
 * contexts are split along the KV axis and merged.  Requests with more rows
 * (prefills) form 128-row tiles for the tensor-core prefill kernel. */
KVQ_API int kvq_get_scheduler_metadata(int num_req, int heads_q, int heads_kv,
                               int head_dim, const int32_t* seq_lens_host,
                               const int32_t* query_start_loc_host, int causal,
                               int window, kvq_dtype_t dtype,
                               kvq_sched_t** out, size_t* workspace_bytes);

/* attention_with_kv_cache -- varlen causal GQA attention over the paged
 * caches, dequantisation fused into the tiles, online softmax.
 * [P1] Breakdown items 2-3 (tile GEMMs with fused fp8 dequantisation,
 * cpu_attention_with_kv_cache) and Risks (scale folding); [P2] Key source
 * snippet (causal, window_size, soft_cap, paged blocks, use_alibi,
 * use_sink); [P3] Breakdown item 3 (_prepare_kv_tile: per-token-head
 * dequantisation in the tile).
 *
 *   sched                   from kvq_get_scheduler_metadata.
 *   heads_q, heads_kv,      what the caller believes the caches and q hold;
 *   head_dim, dtype         they, causal and window must equal the values
 *                           the schedule was built for, else
 *                           KVQ_E_SCHED_MISMATCH.  (The bug of [P2]: tiles
 *                           sized for one KV element size, run on another.)
 *                           Every dtype is supported, KVQ_AUTO (bf16 rows)
 *                           included.
 *   q                       device bf16 [sum Q, heads_q, head_dim], contiguous,
 *                           16-byte aligned.
 *   key_cache, value_cache  as written by kvq_reshape_and_cache.
 *   query_start_loc,        device int32 copies of the arrays given to the
 *   seq_lens                scheduler (same values).
 *   block_table             device int32 [num_req, block_table_stride]:
 *                           logical block i of request r lives in physical
 *                           block block_table[r*stride + i].  Entries outside
 *                           [0, num_blocks) read as empty (masked) keys.
 *   block_size, num_blocks  cache geometry; block_size a multiple of 16,
 *                           num_blocks * block_size < 2^31.
 *   sm_scale                score scale (typically 1/sqrt(head_dim)).
 *   soft_cap                > 0: z <- soft_cap * tanh(z / soft_cap) after
 *                           sm_scale; <= 0: off.
 *   alibi_slopes            device fp32 [heads_q] or NULL: z <- z + slope_h *
 *                           (j - p) for key j and query position p, after
 *                           the soft cap (use_alibi of [P2]).
 *   sinks                   device fp32 [heads_q] or NULL: one extra logit
 *                           s_h per q head in the softmax normaliser, with
 *                           no value: o = sum_j e^z_j v_j / (e^s_h +
 *                           sum_j e^z_j) (use_sink of [P2]).
 *   k_scale, v_scale        per-tensor scales (per-tensor fp8 only), folded
 *                           into the scores and the output.
 *   out                     device bf16 [sum Q, heads_q, head_dim].
 *   workspace               device scratch of >= the scheduler's
 *                           workspace_bytes (256-byte aligned; may be NULL
 *                           when that is 0).  Calls sharing one workspace
 *                           or one schedule must be ordered on one stream.
 * Query row i of a request sits at position L - Q + i; key j is visible iff
 * (!causal || j <= p) and (window <= 0 || p - j < window).  The call
 * launches the prefill kernel (if the schedule has prefill tiles), the decode
 * kernel of each row-tile class, and the merge of the cut decode tiles (the
 * schedule's num_kernel_launches), in that order on `stream`.  A kernel that
 * gives up one of its bounded waits writes NaN rows and sets the schedule's
 * error word (kvq_sched_check_device). */
KVQ_API int kvq_attention_with_kv_cache(const kvq_sched_t* sched, int heads_q,
                                int heads_kv, int head_dim, kvq_dtype_t dtype,
                                const void* q,
                                const void* key_cache, const void* value_cache,
                                const int32_t* query_start_loc,
                                const int32_t* seq_lens,
                                const int32_t* block_table,
                                int block_table_stride, int block_size,
                                int64_t num_blocks, float sm_scale, int causal,
                                int window, float soft_cap,
                                const float* alibi_slopes, const float* sinks,
                                float k_scale, float v_scale, void* out,
                                void* workspace, size_t workspace_bytes,
                                void* stream);

/* attention_with_kv_cache_static_scratch -- the same attention for callers
 * that cannot allocate device memory (no cudaMalloc in their context: a
 * serving loop whose device heap is owned by a memory pool or allocator
 * hook).  It takes no workspace: the split-KV partials go to a fixed
 * KVQ_STATIC_SCRATCH_BYTES array of device memory that the library reserves
 * on every device it is loaded on, held until the process exits.  There is
 * no counterpart on the pages this library follows; it is an interface
 * addition.
 *   Arguments, layouts, ownership and checks are those of
 *   kvq_attention_with_kv_cache without workspace / workspace_bytes.  A
 *   schedule needing more scratch than KVQ_STATIC_SCRATCH_BYTES
 *   (kvq_sched_get_info's workspace_bytes) is refused with
 *   KVQ_E_WORKSPACE_TOO_SMALL before anything is enqueued.
 *   The call allocates nothing.  The first call on each device looks up the
 *   array's device address (cudaGetSymbolAddress); make that first call
 *   before any stream capture.
 *   All calls on a device share the one array and it keeps the last call's
 *   contents: calls that may overlap on the GPU (other streams, other host
 *   threads) race on it; order them on one stream. */
#define KVQ_STATIC_SCRATCH_BYTES (16u << 20)
KVQ_API int kvq_attention_with_kv_cache_static_scratch(
    const kvq_sched_t* sched, int heads_q, int heads_kv, int head_dim, kvq_dtype_t dtype,
    const void* q, const void* key_cache, const void* value_cache,
    const int32_t* query_start_loc, const int32_t* seq_lens, const int32_t* block_table,
    int block_table_stride, int block_size, int64_t num_blocks, float sm_scale, int causal,
    int window, float soft_cap, const float* alibi_slopes, const float* sinks, float k_scale,
    float v_scale, void* out, void* stream);

/* decode_step -- one serving step of a decode batch in ONE kernel launch:
 * the step's new K/V rows are quantised into the caches (exactly as
 * kvq_reshape_and_cache), the work plan is built on the device from the
 * device's query_start_loc / seq_lens (no host scheduler, no host copy of
 * the lengths), and causal split-KV attention runs over the caches (exactly
 * as kvq_attention_with_kv_cache).  [P2] Key source snippet
 * (get_scheduler_metadata feeding the attention, enable_kv_split) and
 * Breakdown item 1 (the schedule sized from the KV element size); [P1]
 * Breakdown items 1-3 (reshape_and_cache, then the attention).  Because
 * nothing of the plan lives on the host, a step captured in a CUDA graph
 * replays correctly with other lengths, new tokens and block tables, within
 * the capacities its workspace was sized for.
 *
 *   num_req, heads_q, heads_kv, head_dim, dtype   as for the other calls.
 *   key, value, num_new_tokens, key_stride_tok, value_stride_tok,
 *   slot_mapping            the step's new rows, as for kvq_reshape_and_cache
 *                           (num_new_tokens may be 0).
 *   key_cache, value_cache, num_blocks, block_size   the paged caches.
 *   q, query_start_loc,     as for kvq_attention_with_kv_cache (device);
 *   seq_lens, block_table,  every request must have 1 <= Q <= max_query_len
 *   block_table_stride      queries (Q = 0: skipped) and Q <= L; its table
 *                           row holds ceil(L / block_size) entries (entries
 *                           beyond block_table_stride, or outside the pool,
 *                           read as masked keys).
 *   max_query_len           host bound on Q; max_query_len * heads_q /
 *                           heads_kv must be <= 16 (decode rows), else
 *                           KVQ_E_UNSUPPORTED.  A request whose device Q
 *                           breaks the bound is skipped and flags the error
 *                           word (kvq_decode_step_check: KVQ_E_INVALID_ARG).
 *   sm_scale, window, soft_cap, alibi_slopes, sinks, k_scale, v_scale
 *                           as for kvq_attention_with_kv_cache (causal).
 *   out                     device bf16 [sum Q, heads_q, head_dim].
 *   workspace               device scratch of >= the size
 *                           kvq_decode_step_workspace_size gives for the
 *                           same num_req, shape, dtype, max_query_len and
 *                           ALiBi setting, 256-byte aligned, ZERO-FILLED
 *                           before its first use (e.g. cudaMemsetAsync);
 *                           every call leaves it ready for the next.  Calls
 *                           sharing a workspace must be ordered on one stream.
 * The kernel is a cooperative launch (all its CTAs resident at once, one
 * grid-wide barrier between the cache write and the attention), followed
 * on the stream by the merge of the tiles it cut among warps (a kernel of
 * its own, launched as a programmatic dependent); the barrier
 * wait is bounded (about a second) and a timeout flags the error word
 * (kvq_decode_step_check: KVQ_E_TIMEOUT).  Allocates nothing. */
KVQ_API int kvq_decode_step(int num_req, int heads_q, int heads_kv, int head_dim,
                            kvq_dtype_t dtype, const void* key, const void* value,
                            int64_t num_new_tokens, int64_t key_stride_tok,
                            int64_t value_stride_tok, const int64_t* slot_mapping,
                            void* key_cache, void* value_cache, int64_t num_blocks,
                            int block_size, const void* q, const int32_t* query_start_loc,
                            const int32_t* seq_lens, const int32_t* block_table,
                            int block_table_stride, int max_query_len, float sm_scale,
                            int window, float soft_cap, const float* alibi_slopes,
                            const float* sinks, float k_scale, float v_scale, void* out,
                            void* workspace, size_t workspace_bytes, void* stream);

/* No counterpart on the pages (their steps start from device tensors).  One
 * decode step from host memory to host memory, for a serving loop whose
 * step inputs and result live on the host: brings in_bytes from host_in to
 * dev_in, runs kvq_decode_step with the arguments after out_bytes -- its
 * device pointers (key, value, slot_mapping, q, query_start_loc, seq_lens,
 * block_table, ...) may point into dev_in --, copies the first out_bytes of
 * `out` to host_out, and waits for the stream.  When the device addresses
 * host_in (cudaHostGetDevicePointer succeeds: pinned memory, or any host
 * memory on systems whose GPU reads pageable memory) and both it and dev_in
 * are 16-byte aligned, the fused kernel does the copy: the
 * cache write and the plan read their inputs from host_in directly and the
 * kernel's other CTAs copy host_in to dev_in before its grid barrier (no
 * separate copy to wait for); otherwise one cudaMemcpyAsync on `stream`
 * comes first.  Either way dev_in holds host_in's bytes after the call.
 * host_in and host_out should be pinned (page-locked) for the copies to be
 * asynchronous; out_bytes must not exceed the output's size.  in_bytes /
 * out_bytes may be 0 (no copy).  With out NULL the step
 * writes its output straight into host_out (pinned host memory the device
 * addresses; out_bytes is then ignored): the rows cross to the host as the
 * kernels store them, with no copy after the step.  Errors: those of
 * kvq_decode_step (nothing is copied back then), KVQ_E_INVALID_ARG for a
 * NULL buffer with a nonzero size or an out NULL whose host_out the device
 * cannot address, KVQ_E_CUDA for a failed copy or wait.  Allocates nothing. */
KVQ_API int kvq_decode_step_host_io(const void* host_in, void* dev_in, size_t in_bytes,
                                    void* host_out, size_t out_bytes, int num_req, int heads_q,
                                    int heads_kv, int head_dim, kvq_dtype_t dtype, const void* key,
                                    const void* value, int64_t num_new_tokens,
                                    int64_t key_stride_tok, int64_t value_stride_tok,
                                    const int64_t* slot_mapping, void* key_cache,
                                    void* value_cache, int64_t num_blocks, int block_size,
                                    const void* q, const int32_t* query_start_loc,
                                    const int32_t* seq_lens, const int32_t* block_table,
                                    int block_table_stride, int max_query_len, float sm_scale,
                                    int window, float soft_cap, const float* alibi_slopes,
                                    const float* sinks, float k_scale, float v_scale, void* out,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* No counterpart on the pages.  kvq_decode_step_host_io's work (without the
 * final wait) captured once in a CUDA graph, for a serving loop that runs
 * the same step on the same buffers every step: each
 * kvq_decode_step_graph_launch replays it on `stream` and waits, so a step
 * costs one graph launch instead of the call's several launches.  The
 * caller rewrites host_in between launches (new rows, lengths, tables and
 * slots within the capacities given here: num_req, max_query_len, the
 * table's width); the plan lives on the device, so the replay follows.
 * Arguments as kvq_decode_step_host_io's, minus the stream.  Unless
 * in_bytes is 0, the fused kernel must be able to stage host_in (memory the
 * device addresses, 16-byte aligned, as is dev_in): otherwise
 * KVQ_E_UNSUPPORTED.  host_out must be pinned.
 * Every buffer must stay allocated, in place, until the graph is destroyed.
 * Errors: those of kvq_decode_step_host_io (nothing is created then),
 * KVQ_E_NO_MEMORY, KVQ_E_CUDA for a failed capture.  Allocates the graph,
 * its executable form and a private capture stream; *graph NULL on error. */
typedef struct kvq_step_graph kvq_step_graph_t;
KVQ_API int kvq_decode_step_graph_create(const void* host_in, void* dev_in, size_t in_bytes,
                                         void* host_out, size_t out_bytes, int num_req,
                                         int heads_q, int heads_kv, int head_dim,
                                         kvq_dtype_t dtype, const void* key, const void* value,
                                         int64_t num_new_tokens, int64_t key_stride_tok,
                                         int64_t value_stride_tok, const int64_t* slot_mapping,
                                         void* key_cache, void* value_cache, int64_t num_blocks,
                                         int block_size, const void* q,
                                         const int32_t* query_start_loc, const int32_t* seq_lens,
                                         const int32_t* block_table, int block_table_stride,
                                         int max_query_len, float sm_scale, int window,
                                         float soft_cap, const float* alibi_slopes,
                                         const float* sinks, float k_scale, float v_scale,
                                         void* out, void* workspace, size_t workspace_bytes,
                                         kvq_step_graph_t** graph);
/* Replay a captured step on `stream` and wait for it.  KVQ_E_INVALID_ARG for
 * a NULL graph, KVQ_E_CUDA for a failed launch or wait; the step's own
 * errors (device lengths beyond the capacities, a barrier timeout) go to the
 * workspace's error word, as kvq_decode_step's (kvq_decode_step_check). */
KVQ_API int kvq_decode_step_graph_launch(kvq_step_graph_t* graph, void* stream);
/* Free a captured step (NULL is a no-op); no launch of it may be pending. */
KVQ_API void kvq_decode_step_graph_destroy(kvq_step_graph_t* graph);

/* Workspace bytes of kvq_decode_step for these arguments on the current
 * device ([P2] Breakdown item 1: scratch sized from the KV element size and
 * the tile geometry).  use_alibi: whether alibi_slopes will be non-NULL.
 * Errors as kvq_decode_step's shape checks. */
KVQ_API int kvq_decode_step_workspace_size(int num_req, int heads_q, int heads_kv, int head_dim,
                                           kvq_dtype_t dtype, int max_query_len, int use_alibi,
                                           size_t* workspace_bytes);

/* No counterpart on the pages.  Read, and clear, a decode_step workspace's
 * error word: KVQ_E_TIMEOUT (the grid barrier gave up), KVQ_E_INVALID_ARG
 * (a request's device lengths broke the bounds) or KVQ_OK.  Blocks until
 * the device is idle. */
KVQ_API int kvq_decode_step_check(const void* workspace);

/* Free a schedule (NULL is a no-op).  No counterpart on the pages (their
 * schedule is a torch tensor that the garbage collector frees); it is the
 * C ABI's ownership rule for the object get_scheduler_metadata returns.
 * Its pinned plan image and device buffer go back to small library pools
 * that later schedules reuse (no cudaMalloc / cudaHostAlloc per step), so
 * destroy a schedule only once the attention calls that use it have
 * completed on the device, as for any memory the caller frees. */
KVQ_API void kvq_sched_destroy(kvq_sched_t* sched);

/* Summary of a schedule, for tests and benchmarks.  [P2] Breakdown item 1:
 * the sizes the scheduler derived from the KV element size (kv_elem_bytes,
 * row_bytes, workspace and shared-memory bytes) are the ones the kernels
 * run with.  Returns KVQ_E_INVALID_ARG for a NULL argument. */
typedef struct {
  int num_req, heads_q, heads_kv, head_dim;
  int dtype;                   /* kvq_dtype_t the schedule was built for      */
  int kv_elem_bytes;           /* bytes per cached K/V element (1 or 2)       */
  int row_bytes;               /* bytes per (token, kv_head) cache row        */
  int causal, window;
  int64_t num_tiles;           /* row tiles: <= 16 (query, head) rows of a kv head */
  int64_t num_pieces;          /* tile pieces (a tile cut among warps)        */
  int64_t num_merge_items;     /* tiles cut into more than one piece          */
  int64_t num_chunks;          /* 16-token KV chunks streamed in total        */
  int64_t num_decode_warps;    /* warps the chunk sequence is cut among       */
  int64_t max_splits;          /* most pieces of one tile                     */
  int64_t total_query_tokens;
  size_t workspace_bytes;
  size_t decode_smem_bytes;    /* dynamic shared memory per decode CTA        */
  size_t decode_chunk_bytes;   /* K+V bytes a warp streams per 16-token chunk */
  int64_t num_prefill_tiles;   /* 128-row tiles of the tensor-core prefill
                                  (CTA pairs: list entries, empty partners
                                  included; see kvq_plan_prefill_tile_t) */
  size_t prefill_smem_bytes;   /* dynamic shared memory per prefill CTA       */
  int64_t num_kernel_launches; /* kernels one attention call launches         */
  int64_t prefill_cta_group;   /* CTAs per prefill tile MMA: 1, or 2 for CTA
                                  pairs (a build option)                      */
} kvq_sched_info_t;

KVQ_API int kvq_sched_get_info(const kvq_sched_t* sched, kvq_sched_info_t* out);

/* ---- the plan, for tests and tools (host copies; no device access) --------
 * [P2] Breakdown item 1: the schedule is the single source of the tile and
 * scratch sizes the kernels run with; these calls expose it for checking.
 *
 * A decode piece is a run of consecutive 16-token chunks of one row tile
 * (<= 16 packed rows of one kv head), streamed by one warp.  The pieces of a
 * launch class lie end to end in its flat chunk sequence, which is cut into
 * contiguous segments, one per warp (stream-K: segment w starts at
 * floor(w * chunks / warps)); a tile cut by a segment boundary has several
 * pieces, whose partial rows a merge item combines.  The tiles are in
 * (request, kv head) order when a cache row is a whole number of 128-byte
 * lines; otherwise in head lockstep (lockstep[c] == 1): kv-head-major order,
 * a warp count that is a multiple of the kv heads (Hkv), every head's run cut
 * at the same chunks, and segment h * (warps / Hkv) + v on warp v * Hkv + h,
 * so the warps reading neighbouring heads' rows of the same tokens -- which
 * share 128-byte lines -- are neighbours and run side by side. */
typedef struct {
  int32_t launch;          /* decode launch class: 0 (tiles of <= 8 rows) or 1 */
  int32_t req, kv_head, row0, nrows;
  int32_t part;            /* first partial row of the piece in the workspace; -1: writes out */
  int32_t merge;           /* merge item of a cut tile; -1: not cut */
  int32_t key_lo, key_hi;  /* keys some row of the tile can see: [key_lo, key_hi) */
  int32_t flat0;           /* the piece's first position in its class's chunk sequence */
  int32_t chunk0;          /* that chunk's 16-token index within the request */
  int32_t nchunks;         /* chunks in the piece */
} kvq_plan_piece_t;

typedef struct {
  int32_t req, kv_head, row0, nrows;
  int32_t part;            /* partial row of (split 0, row 0); split s row n at part + s*nrows + n */
  int32_t nsplits;
} kvq_plan_merge_t;

/* A prefill tile.  Quantised caches at head_dim 128 and 256 run the prefill
 * on CTA pairs: entries 2i and 2i + 1 of the list are then two consecutive
 * row tiles of one (request, kv head), whose MMAs (M = 256) share each KV
 * tile, or a last tile and an empty partner (nrows 0, the same key range). */
typedef struct {
  int32_t req, kv_head, row0, nrows;  /* up to 128 packed rows of one kv head */
  int32_t key_lo, key_hi;             /* keys some row of the tile can see */
} kvq_plan_prefill_tile_t;

typedef struct {
  int64_t num_pieces, num_merges, num_prefill_tiles;
  int64_t num_chunks[2];   /* per decode launch class */
  int32_t num_warps[2];    /* per decode launch class */
  int32_t lockstep[2];     /* per class: 1 if cut in head lockstep (see above) */
} kvq_plan_sizes_t;

KVQ_API int kvq_sched_get_plan_sizes(const kvq_sched_t* sched, kvq_plan_sizes_t* out);

/* Copy the plan: pieces (class 0 then class 1, each in flat order), the
 * first piece of every warp's segment (class 0's warps then class 1's, as
 * indices into `pieces`; -1 for an empty segment), merge items and prefill
 * tiles (in launch order).  Any array may be NULL; otherwise its capacity
 * must hold the count from kvq_sched_get_plan_sizes (warps: num_warps[0] +
 * num_warps[1]), else KVQ_E_INVALID_ARG and nothing is written. */
KVQ_API int kvq_sched_export_plan(const kvq_sched_t* sched, kvq_plan_piece_t* pieces,
                                  int64_t pieces_cap, int32_t* warp_first_piece,
                                  int64_t warps_cap, kvq_plan_merge_t* merges,
                                  int64_t merges_cap, kvq_plan_prefill_tile_t* tiles,
                                  int64_t tiles_cap);

/* No counterpart on the pages (their kernels have no bounded waits).
 * Read, and clear, the schedule's device error word: KVQ_E_TIMEOUT if a
 * kernel run with this schedule gave up waiting for the tensor core (a
 * bounded wait of about a second; the kernel then released its tensor
 * memory and wrote NaN into the output rows of its tile); in the
 * bounds-checked build (libkvq_checked.so, compiled with KVQ_CHECKED=1)
 * KVQ_E_INVALID_ARG if a kernel found an index it derived from a device
 * array (query_start_loc row offsets, block-table positions) outside its
 * array and skipped the access; else KVQ_OK.
 * The attention calls return before their kernels run, so they cannot
 * report this themselves: a caller that does not read the error word sees
 * such a failure as NaN rows.  Blocks until the device is idle. */
KVQ_API int kvq_sched_check_device(const kvq_sched_t* sched);

/* Short English description of a status code (static storage; never NULL:
 * unknown codes give "unknown status").  No counterpart on the pages: the
 * C ABI returns status codes where their C++ entry points raise. */
KVQ_API const char* kvq_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
