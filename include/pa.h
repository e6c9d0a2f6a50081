/*
 * pa.h -- C ABI of the paged-KV attention library (libpa.so), sm_103a.
 *
 * Three operations make up the hot path of attention over a paged KV cache:
 *
 *   pa_reshape_and_cache  write new K/V rows into the physical block pool
 *                         through slot_mapping;
 *   pa_decode             one query token per sequence against its blocks,
 *                         online softmax, split-KV log-sum-exp combine;
 *   pa_prefill_varlen     causal attention for cu_seqlens-packed queries
 *                         against the paged cache.
 *
 * pa_decode_write is one decode step as one call (the write, then the
 * decode, overlapped); pa_decode_plan sizes pa_decode's workspace;
 * pa_decode_static_ws is pa_decode without a caller-supplied workspace.
 * pa_reshape_and_cache_int8 / pa_decode_int8 / pa_decode_write_int8 are the
 * write, the decode and the step over INT8 pools, the _fp8 calls the same
 * over FP8 (E4M3) pools; pa_copy_blocks copies whole blocks (copy-on-write).
 *
 * Sources (web pages on paged KV caches, cited by page and section):
 *   [SKILL] cannbot-skills "model-infer-kvcache" skill page: §3.1 physical
 *           layout and logical mapping, §3.3 slot_mapping, §3.4
 *           actual_seq_lengths, §3.6 data flow, App. C sparse_mode, App. E
 *           prefill vs decode parameters.
 *   [MHPQ]  "Paged KV Cache and Packed Sequence in cann-recipes-infer":
 *           §3.3 the paged_attention operator's parameters.
 *   [LQNN]  "Paged KV Cache is infrastructure, not a renamed cache": §3.1
 *           cu_seqlens, §4.4 packed attention, §4.5 cache update, §5.1 pitch.
 *   [VLLM]  "vLLM on CANN": PagedKVCache.read_kv and the block-wise online
 *           softmax of its attention kernel.
 *   [ATB]   "Ascend CANN ATB KV Cache and PagedAttention": the shared page
 *           pool and copy-on-write of a shared page ("page update race").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is caller-owned DEVICE memory on the current
 *    CUDA device unless stated otherwise.  The library never allocates,
 *    frees, synchronises, or reads device memory on the host; every kernel is
 *    enqueued on `stream` (a cudaStream_t passed as void*; NULL = the legacy
 *    default stream) and the call returns before it runs.
 *  - Strides are in ELEMENTS.  Element type is fp16 or bf16 (`dtype`); every
 *    K/V/Q/out pointer must be 16-byte aligned and every row stride a
 *    multiple of 8 elements.  The 8-bit (INT8 / FP8) calls keep fp16/bf16
 *    queries, outputs and new K/V rows; only their pools hold one-byte codes.
 *    pa_copy_blocks copies bytes and takes no element type.
 *  - Cache layout ([SKILL] §3.1): key_cache and value_cache are separate,
 *    contiguous [num_blocks, block_size, num_kv_heads, head_dim] pools.  A
 *    physical slot s addresses row s of the pool viewed as
 *    [num_blocks * block_size, num_kv_heads, head_dim], i.e. block
 *    s / block_size, offset s % block_size.
 *  - block_table is int32 [num_seqs, block_table_stride]; entry [b, i] is the
 *    physical block of logical block i of sequence b ([SKILL] §3.1-3.2).
 *    Only the first ceil(context_len / block_size) entries of a row are
 *    read; max_blocks_per_seq (<= block_table_stride) bounds the capacity.
 *  - Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *  - `scale` multiplies q.k and has NO default: the pages warn that a
 *    silently defaulted 1.0 corrupts results ([SKILL] App. A).
 *  - Host-detectable argument errors return a pa_status and enqueue nothing.
 *    Data-dependent errors found on the device (a bad slot, block id,
 *    cu_seqlens entry or context length) skip the affected unit of work and
 *    OR a PA_DEVERR_* bit into *d_error when d_error is non-NULL (an int32 in
 *    device memory the caller zeroes and reads).  No kernel traps, asserts or
 *    waits without a bound: a pipeline wait that exceeds its iteration limit
 *    sets PA_DEVERR_TIMEOUT and the block returns.
 *  - Outputs of sequences with context_len == 0, and of causal rows that see
 *    no key, are written as zeros ([MHPQ] §3.3: all-zero context lengths
 *    give an all-zero output).
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_ABI_VERSION 1

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_NULL = 1,        /* a required pointer is NULL                      */
  PA_ERR_SHAPE = 2,       /* inconsistent or negative sizes / strides        */
  PA_ERR_UNSUPPORTED = 3, /* valid but not built (head_dim, block_size, ...)  */
  PA_ERR_ALIGN = 4,       /* pointer not 16-byte aligned or stride not x8    */
  PA_ERR_WORKSPACE = 5,   /* workspace missing or smaller than required      */
  PA_ERR_CUDA = 6         /* a CUDA runtime call failed (pa_last_cuda_error) */
} pa_status;

typedef enum pa_dtype { PA_F16 = 0, PA_BF16 = 1 } pa_dtype;

/* Bits OR-ed into *d_error by the kernels. */
#define PA_DEVERR_SLOT 1       /* slot_mapping entry >= num_blocks*block_size */
#define PA_DEVERR_BLOCK_ID 2   /* block_table / block_mapping entry outside
                                  [0, num_blocks)                            */
#define PA_DEVERR_CU_SEQLENS 4 /* cu_seqlens not a prefix sum of the batch    */
#define PA_DEVERR_CONTEXT 8    /* context_len < 0, > capacity or > host hint  */
#define PA_DEVERR_TIMEOUT 16   /* a bounded pipeline wait gave up             */
#define PA_DEVERR_SCALE 32     /* an 8-bit pool's scale not positive finite   */

/* ABI version the library was built with (PA_ABI_VERSION). */
int32_t pa_abi_version(void);

/* Static, human-readable name of a status code. */
const char *pa_status_string(pa_status status);

/* cudaError_t of the most recent PA_ERR_CUDA on the calling thread (0 if
 * none). */
int32_t pa_last_cuda_error(void);

/*
 * pa_reshape_and_cache -- write this step's K/V rows into the pools.
 *
 * Defines ([SKILL] §3.3, App. D; [LQNN] §4.5): for each token t in
 * [0, num_tokens) with s = slot_mapping[t]:
 *     s <  0                     -> nothing is written (padding token);
 *     s >= num_blocks*block_size -> nothing is written, PA_DEVERR_SLOT;
 *     otherwise key_cache row s   = key[t]   (bit copy, all heads),
 *               value_cache row s = value[t].
 *
 *   key, value      [num_tokens, num_kv_heads, head_dim]; token t starts at
 *                   element t * kv_row_stride (heads contiguous, so K and V
 *                   may be views into an interleaved QKV buffer).
 *   key_cache,
 *   value_cache     pools as described above; written, never read.
 *   slot_mapping    int64 [num_tokens].  Duplicate non-negative slots in one
 *                   call are a caller error (which row wins is unspecified).
 *   d_error         nullable device int32, see above.
 * Requirements: num_kv_heads * head_dim * 2 bytes a multiple of 16.
 * num_tokens == 0 enqueues nothing and returns PA_OK.
 */
pa_status pa_reshape_and_cache(const void *key, const void *value,
                               int64_t kv_row_stride, void *key_cache,
                               void *value_cache, const int64_t *slot_mapping,
                               int32_t num_tokens, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size,
                               int64_t num_blocks, pa_dtype dtype,
                               int32_t *d_error, void *stream);

/*
 * pa_decode_plan -- the split-KV plan pa_decode will use.
 *
 * Long contexts are split into pieces; each piece's softmax state (max, sum,
 * unnormalised output) is combined by log-sum-exp ([SKILL] §3.1; the pages'
 * split-KV partitions).  A non-zero partition_size must be a positive
 * multiple of 16: every (sequence, KV head) is cut into partitions of that
 * many tokens and *partition_size_out returns it.  partition_size == 0 is the
 * automatic plan: the balanced split, which cuts the batch's whole token
 * stream into equal shares, one per worker of the decode grid (so no worker
 * waits on a long sequence while others idle); *partition_size_out is then 0.
 * (The automatic plan falls back to fixed partitions sized from
 * max_context_len, the batch shape and the SM count when the batch's token
 * count does not fit in int32.)  *workspace_bytes_out is the device
 * workspace pa_decode needs (0 when no context can be split).  Host-only;
 * enqueues nothing.
 */
pa_status pa_decode_plan(int32_t num_seqs, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim,
                         int32_t max_context_len, int32_t partition_size,
                         int32_t *partition_size_out,
                         size_t *workspace_bytes_out);

/*
 * pa_decode -- paged attention for one query token per sequence.
 *
 * Defines ([SKILL] §3.1, §3.6, App. C sparse_mode 0; [MHPQ] §3.3; [VLLM]):
 * for sequence b, query head h, KV head g = h / (Hq/Hkv), L = context_lens[b]
 *     K_j = key_cache[block_table[b, j / block_size], j % block_size, g, :]
 *     V_j likewise from value_cache,   j = 0 .. L-1 (no mask)
 *     out[b, h, :] = sum_j softmax_j(scale * q[b, h, :] . K_j) V_j,
 * accumulated in fp32 and rounded to dtype (nearest-even); 0 when L == 0.
 * context_lens counts the token written this step ([SKILL] §3.6:
 * actual_seq_lengths_kv = kv_len + 1), so write first, then decode.
 *
 *   out             [num_seqs, num_q_heads, head_dim], row stride
 *                   out_row_stride (elements between sequences).
 *   query           [num_seqs, num_q_heads, head_dim], row stride
 *                   q_row_stride.
 *   block_table     int32 [num_seqs, block_table_stride].
 *   context_lens    int32 [num_seqs].
 *   max_context_len host upper bound of context_lens (the pages'
 *                   max_context_len); sizes the grid.  A larger device value
 *                   is clamped to it and flagged PA_DEVERR_CONTEXT.
 *   partition_size  as for pa_decode_plan (0 = auto).
 *   workspace       device scratch of at least the planned bytes, 256-byte
 *                   aligned; may be NULL when the plan needs 0 bytes.
 * Supported: head_dim 64 or 128; num_q_heads / num_kv_heads in 1..8;
 * block_size 8, 16, 32, 64 or 128.
 */
pa_status pa_decode(void *out, int64_t out_row_stride, const void *query,
                    int64_t q_row_stride, const void *key_cache,
                    const void *value_cache, const int32_t *block_table,
                    int64_t block_table_stride, int32_t max_blocks_per_seq,
                    const int32_t *context_lens, int32_t num_seqs,
                    int32_t num_q_heads, int32_t num_kv_heads,
                    int32_t head_dim, int32_t block_size, int64_t num_blocks,
                    float scale, int32_t max_context_len,
                    int32_t partition_size, void *workspace,
                    size_t workspace_bytes, pa_dtype dtype, int32_t *d_error,
                    void *stream);

/*
 * pa_prefill_varlen -- causal attention for packed variable-length queries.
 *
 * Defines ([LQNN] §3.1, §4.4; [SKILL] App. C sparse_mode 3, App. E): the
 * queries of sequence b are rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of
 * `query` (q_b rows), and its keys are the first L_b = context_lens[b]
 * positions of its paged cache (write them first with pa_reshape_and_cache).
 * Row i of sequence b (query head h, KV head g) attends keys
 *     j <= L_b - q_b + i   when causal (the last query sees every key;
 *                          with L_b == q_b this is the plain lower
 *                          triangle of each sequence, never across
 *                          sequences),
 *     j <  L_b             when not causal,
 * with the same softmax and rounding as pa_decode.  Rows with no visible key
 * are written as zeros.
 *
 *   out, query      [total_q, num_q_heads, head_dim] with row strides
 *                   out_row_stride / q_row_stride.
 *   cu_seqlens_q    int32 [num_seqs + 1]: 0, then the running sum of q_b,
 *                   ending at total_q ([LQNN] §3.1 / §3.3 assert).
 *   context_lens    int32 [num_seqs].
 *   total_q         host copy of cu_seqlens_q[num_seqs].
 *   max_seqlen_q    host upper bound of q_b (the pages'
 *                   max_seqlen_in_batch); with total_q it sizes the grid.
 *   max_context_len host upper bound of context_lens.
 * Device checks: a cu_seqlens_q that is not a non-decreasing prefix sum
 * ending at total_q, or a q_b above max_seqlen_q, sets
 * PA_DEVERR_CU_SEQLENS and the offending sequences are skipped.
 * Supported: head_dim 64 or 128; num_q_heads % num_kv_heads == 0; block_size 16,
 * 32, 64 or 128.
 * Work is handed out to the CTAs through one of 256 counters kept in the
 * library's device memory, taken round robin per call; it needs no
 * workspace.  Calls may overlap on the GPU (different streams) as long as
 * fewer than 256 of them are in flight at once.
 */
pa_status pa_prefill_varlen(void *out, int64_t out_row_stride,
                            const void *query, int64_t q_row_stride,
                            const void *key_cache, const void *value_cache,
                            const int32_t *block_table,
                            int64_t block_table_stride,
                            int32_t max_blocks_per_seq,
                            const int32_t *cu_seqlens_q,
                            const int32_t *context_lens, int32_t num_seqs,
                            int32_t total_q, int32_t max_seqlen_q,
                            int32_t max_context_len, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int64_t num_blocks,
                            float scale, int32_t causal, pa_dtype dtype,
                            int32_t *d_error, void *stream);

/*
 * pa_decode_write -- one decode step: the new tokens' cache write, then the
 * decode that reads them.
 *
 * Defines ([SKILL] §3.6 decode data flow: write the step's K/V through
 * slot_mapping, then attend with actual_seq_lengths_kv = kv_len + 1;
 * [LQNN] §4.1–4.7 the decode loop): exactly
 *     pa_reshape_and_cache(key, value, kv_row_stride, key_cache, value_cache,
 *                          slot_mapping, num_new_tokens, ...);
 *     pa_decode(out, ..., key_cache, value_cache, block_table, ...);
 * on `stream`, with the same arguments, meanings, layouts and device error
 * bits as those two calls (key/value: [num_new_tokens, num_kv_heads,
 * head_dim] rows at kv_row_stride elements apart).  Every argument of both
 * is checked before either is enqueued.  What the pair does not allow: the
 * decode kernel reads context_lens, block_table and query, and builds its
 * schedule, while the write is still running, waiting for the write only
 * before its first K/V load -- so the write's time is hidden behind the
 * decode's start-up.  num_new_tokens == 0 is a plain pa_decode.
 */
pa_status pa_decode_write(void *out, int64_t out_row_stride,
                          const void *query, int64_t q_row_stride,
                          const void *key, const void *value,
                          int64_t kv_row_stride, void *key_cache,
                          void *value_cache, const int64_t *slot_mapping,
                          int32_t num_new_tokens, const int32_t *block_table,
                          int64_t block_table_stride,
                          int32_t max_blocks_per_seq,
                          const int32_t *context_lens, int32_t num_seqs,
                          int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, int32_t block_size,
                          int64_t num_blocks, float scale,
                          int32_t max_context_len, int32_t partition_size,
                          void *workspace, size_t workspace_bytes,
                          pa_dtype dtype, int32_t *d_error, void *stream);

/*
 * pa_debug_set_wait_limit_ns -- a testing aid; the pages have no
 * counterpart.
 *
 * Sets the bound, in nanoseconds, of every pipeline wait (one warp waiting
 * for another's data or buffer) in the kernels launched after the call,
 * from any thread; 0 restores the default of 2 s.  A wait that runs out
 * sets PA_DEVERR_TIMEOUT and its block returns, after waiting (with the full
 * 2 s bound) for the copies it has in flight and freeing its tensor memory.
 * A short bound lets a test run that recovery path without any fault: the
 * outputs of launches whose waits ran out are unspecified, and the launches
 * after them must be unaffected.
 */
void pa_debug_set_wait_limit_ns(uint64_t ns);

/*
 * pa_decode_static_ws -- pa_decode for callers that cannot allocate.
 *
 * The pages have no counterpart to this entry point; it is a convenience of
 * this library.  pa_decode needs a caller-supplied device workspace whenever
 * a sequence spans several split-KV partitions.  Some callers cannot provide
 * one: code that must not call cudaMalloc (for example while recording work
 * for later replay, or in a loop with a fixed memory budget), a plug-in
 * whose host framework owns every device allocation, or a plain C caller
 * without a device allocator.  This variant computes exactly what pa_decode
 * computes (same arguments, minus workspace/workspace_bytes) with its
 * workspace in a fixed array of PA_STATIC_WORKSPACE_BYTES inside the
 * library's device image, so it allocates nothing.
 *
 *  - Every GPU that loads the library holds the array until the process
 *    exits.
 *  - The first call on each device (with that device current) looks up the
 *    array's device address once; make that first call before any stream
 *    capture.  A failed lookup returns PA_ERR_CUDA.
 *  - partition_size == 0 uses pa_decode's automatic plan, lengthened (fewer
 *    partitions) until its workspace fits the array; an explicit
 *    partition_size whose workspace does not fit returns PA_ERR_WORKSPACE.
 *    So does a shape that would fit only with partitions too long for the
 *    decode kernel's shared memory (their block ids; many sequences of
 *    long contexts at block_size 8 or 16): use pa_decode with a workspace.
 *  - A failed lookup is recorded for pa_last_cuda_error().
 *  - All calls on a device share the array and leave their partial results
 *    in it (nothing in it has to start at zero).  Calls that may overlap on
 *    the GPU race on it: order them on one stream.
 */
#define PA_STATIC_WORKSPACE_BYTES (16u << 20) /* 16 MiB */

pa_status pa_decode_static_ws(void *out, int64_t out_row_stride,
                              const void *query, int64_t q_row_stride,
                              const void *key_cache, const void *value_cache,
                              const int32_t *block_table,
                              int64_t block_table_stride,
                              int32_t max_blocks_per_seq,
                              const int32_t *context_lens, int32_t num_seqs,
                              int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t block_size,
                              int64_t num_blocks, float scale,
                              int32_t max_context_len, int32_t partition_size,
                              pa_dtype dtype, int32_t *d_error, void *stream);

/*
 * INT8 KV pools.
 *
 * The pages list the fused attention operator's quantised-KV parameters --
 * one dequantisation scale for the key and one for the value ([SKILL] App.
 * A) -- and name an INT8 KV cache among its advanced features ([SKILL]
 * "advanced features"), without printing the formula.  This library's
 * reading: one fp32 scale per KV head for K (k_scale[g]) and one for V
 * (v_scale[g]); a value x is stored as the int8 code
 *     c = round-half-to-even(x / scale), clamped to [-127, 127]
 * with the division and the rounding in fp32 (IEEE round to nearest), a NaN
 * input stored as 0, and it is read back as c * scale.  The pools are
 * [num_blocks, block_size, num_kv_heads, head_dim] int8; everything else is
 * as for the 16-bit calls.  Halving the pool's bytes halves what a decode
 * step reads.
 *
 * A scale that is not a positive finite number sets PA_DEVERR_SCALE; the
 * write then stores code 0 for that head, and the decode gives that head's
 * queries a zero output.
 */

/*
 * pa_reshape_and_cache_int8 -- pa_reshape_and_cache into INT8 pools.
 *
 *   key, value      [num_tokens, num_kv_heads, head_dim] fp16/bf16 (dtype),
 *                   token t at element t * kv_row_stride.
 *   key_cache,
 *   value_cache     int8 pools; written, never read.
 *   k_scale,
 *   v_scale         device fp32 [num_kv_heads]; read, never written.
 * Requirements: num_kv_heads * head_dim a multiple of 16 (16-byte int8 rows
 * of the pool) and kv_row_stride * 2 bytes a multiple of 16.
 */
pa_status pa_reshape_and_cache_int8(const void *key, const void *value,
                                    int64_t kv_row_stride, void *key_cache,
                                    void *value_cache, const int64_t *slot_mapping,
                                    int32_t num_tokens, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t block_size,
                                    int64_t num_blocks, const float *k_scale,
                                    const float *v_scale, pa_dtype dtype,
                                    int32_t *d_error, void *stream);

/*
 * pa_decode_int8 -- pa_decode over INT8 pools.
 *
 * out[b, h, :] = sum_j softmax_j(scale * q . (k_scale[g] * Kc_j))
 *                      (v_scale[g] * Vc_j)
 * with Kc_j, Vc_j the int8 codes of key/value row j of KV head g.  The
 * scores and the weighted sum are accumulated in fp32 from the codes widened
 * exactly to fp16 and the query rounded to fp16 (its nearest fp16 value; a
 * query beyond the fp16 range is not supported); the K scale multiplies the
 * scores and the V scale the output.  query / out are fp16 or bf16 (dtype).
 * Workspace: as pa_decode_plan reports for the same shape.
 * Supported: head_dim 128; num_q_heads / num_kv_heads in 1..8; block_size 8,
 * 16, 32, 64 or 128.
 */
pa_status pa_decode_int8(void *out, int64_t out_row_stride, const void *query,
                         int64_t q_row_stride, const void *key_cache,
                         const void *value_cache, const int32_t *block_table,
                         int64_t block_table_stride, int32_t max_blocks_per_seq,
                         const int32_t *context_lens, int32_t num_seqs,
                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int64_t num_blocks, const float *k_scale,
                         const float *v_scale, float scale, int32_t max_context_len,
                         int32_t partition_size, void *workspace,
                         size_t workspace_bytes, pa_dtype dtype, int32_t *d_error,
                         void *stream);

/*
 * pa_decode_write_int8 -- one decode step over INT8 pools in one call:
 * pa_reshape_and_cache_int8(key, value, ..., slot_mapping, num_new_tokens,
 * k_scale, v_scale), then pa_decode_int8 over the updated pools, overlapped
 * like pa_decode_write (the decode reads everything but the K/V codes while
 * the write runs).  Every argument is checked before anything is enqueued;
 * arguments, requirements and errors are those of the two calls.
 */
pa_status pa_decode_write_int8(void *out, int64_t out_row_stride, const void *query,
                               int64_t q_row_stride, const void *key, const void *value,
                               int64_t kv_row_stride, void *key_cache, void *value_cache,
                               const int64_t *slot_mapping, int32_t num_new_tokens,
                               const int32_t *block_table, int64_t block_table_stride,
                               int32_t max_blocks_per_seq, const int32_t *context_lens,
                               int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size, int64_t num_blocks,
                               const float *k_scale, const float *v_scale, float scale,
                               int32_t max_context_len, int32_t partition_size,
                               void *workspace, size_t workspace_bytes, pa_dtype dtype,
                               int32_t *d_error, void *stream);

/*
 * FP8 KV pools.
 *
 * The same per-KV-head scales as the INT8 pools, with codes in the OCP FP8
 * E4M3 format (1 sign, 4 exponent bits of bias 7, 3 fraction bits;
 * exponent 0 subnormal; S.1111.111 NaN; no infinities, largest finite 448).
 * A value x is stored as the E4M3 value nearest to x / scale (the division
 * in fp32, ties to the even code, saturating at +-448; a NaN input is
 * stored as 0) and read back as value(code) * scale.  Pools are
 * [num_blocks, block_size, num_kv_heads, head_dim] bytes; the three calls
 * below are the FP8 counterparts of the INT8 calls above, with the same
 * arguments, requirements (head_dim 128 for the decode) and errors.  NaN
 * codes never come from the write; rows past a sequence's context may hold
 * any byte.
 */
pa_status pa_reshape_and_cache_fp8(const void *key, const void *value, int64_t kv_row_stride,
                                   void *key_cache, void *value_cache,
                                   const int64_t *slot_mapping, int32_t num_tokens,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                   int64_t num_blocks, const float *k_scale,
                                   const float *v_scale, pa_dtype dtype, int32_t *d_error,
                                   void *stream);

pa_status pa_decode_fp8(void *out, int64_t out_row_stride, const void *query,
                        int64_t q_row_stride, const void *key_cache, const void *value_cache,
                        const int32_t *block_table, int64_t block_table_stride,
                        int32_t max_blocks_per_seq, const int32_t *context_lens,
                        int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, int32_t block_size, int64_t num_blocks,
                        const float *k_scale, const float *v_scale, float scale,
                        int32_t max_context_len, int32_t partition_size, void *workspace,
                        size_t workspace_bytes, pa_dtype dtype, int32_t *d_error,
                        void *stream);

pa_status pa_decode_write_fp8(void *out, int64_t out_row_stride, const void *query,
                              int64_t q_row_stride, const void *key, const void *value,
                              int64_t kv_row_stride, void *key_cache, void *value_cache,
                              const int64_t *slot_mapping, int32_t num_new_tokens,
                              const int32_t *block_table, int64_t block_table_stride,
                              int32_t max_blocks_per_seq, const int32_t *context_lens,
                              int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t block_size, int64_t num_blocks,
                              const float *k_scale, const float *v_scale, float scale,
                              int32_t max_context_len, int32_t partition_size,
                              void *workspace, size_t workspace_bytes, pa_dtype dtype,
                              int32_t *d_error, void *stream);

/*
 * pa_copy_blocks -- copy whole blocks of both pools (copy-on-write).
 *
 * Defines ([ATB] "page update race": before a request appends K/V to a page
 * that other requests share, a free page is taken and the whole page is
 * copied into it; the page table then points at the copy): for each pair p
 * in [0, num_pairs) with src = block_mapping[2p], dst = block_mapping[2p+1]:
 *     both in [0, num_blocks) -> block dst of key_cache and of value_cache
 *                                receives block src, bit for bit;
 *     otherwise               -> nothing is copied for p, PA_DEVERR_BLOCK_ID.
 * Choosing the pairs (reference counts, the free page, the block-table
 * update) is the caller's policy.
 *
 *   key_cache,
 *   value_cache     pools of num_blocks blocks of block_bytes bytes each, of
 *                   any element type (16-bit or INT8 pools alike).
 *   block_mapping   int64 [num_pairs][2] device array of (src, dst).  A dst
 *                   that is also some pair's src, or named by two pairs, is a
 *                   caller error (the result is unspecified); src == dst
 *                   leaves the block as it is.
 *   d_error         nullable device int32, see above.
 * Requirements: block_bytes a positive multiple of 16; the pools 16-byte and
 * block_mapping 8-byte aligned.  num_pairs == 0 enqueues nothing.
 */
pa_status pa_copy_blocks(void *key_cache, void *value_cache, int64_t block_bytes,
                         int64_t num_blocks, const int64_t *block_mapping,
                         int32_t num_pairs, int32_t *d_error, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
