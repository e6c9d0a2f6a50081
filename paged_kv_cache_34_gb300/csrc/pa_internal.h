// pa_internal.h -- launcher interface between the C ABI shim (pa_api.cu) and
// the kernels.  Arguments arrive here already validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

struct ReshapeArgs {
  const void *key;
  const void *value;
  int64_t row_stride_bytes;  // between consecutive tokens of key / value
  void *key_cache;
  void *value_cache;
  const int64_t *slot_mapping;
  int32_t num_tokens;
  int64_t row_bytes;  // Hkv * D * 2
  int64_t num_slots;  // num_blocks * block_size
  int32_t *d_error;
  int num_sms;
  // 8-bit pools: the inputs are `dtype` (fp16/bf16), the pools INT8 codes
  // (or, with fp8, E4M3 codes) under the per-KV-head scales; row_bytes
  // counts the 16-bit input row.
  bool int8 = false;
  bool fp8 = false;
  pa_dtype dtype = PA_F16;
  int32_t head_dim = 0;
  const float *k_scale = nullptr, *v_scale = nullptr;
};
cudaError_t launch_reshape_and_cache(const ReshapeArgs &a, cudaStream_t stream);

struct CopyBlocksArgs {
  void *key_cache;
  void *value_cache;
  int64_t block_bytes;  // one block of one pool, a multiple of 16
  int64_t num_blocks;
  const int64_t *block_mapping;  // [num_pairs][2] (src, dst)
  int32_t num_pairs;
  int32_t *d_error;
  int num_sms;
};
cudaError_t launch_copy_blocks(const CopyBlocksArgs &a, cudaStream_t stream);

// Decode tiling shared by the planner and the kernels.
constexpr int kDecodeWarps = 4;     // consumer warps (independent workers) per CTA
constexpr int kDecodeCtasPerSm = 2;  // resident decode CTAs per SM
constexpr int kDecodeSub = 16;      // tokens per worker per pipeline stage
constexpr int kDecodeChunkCap = 2048;  // balanced schedule: most tokens per chunk
constexpr int kDecodeSliceHeads = 16;  // most query heads one K/V read serves

// The query heads of one KV head (the GQA group, G of them) are served in
// slices of at most kDecodeSliceHeads heads: one K/V read serves a whole
// slice (one or two 8-head column groups of the score tile), and a KV head
// with more query heads is read once per slice.  A decode unit is one
// (sequence, slice); a sequence has num_kv_heads * nc units.
struct DecodeSlices {
  int ng;  // 8-head column groups per slice (1 or 2)
  int hs;  // query heads per slice (the last slice may hold fewer)
  int nc;  // slices per KV head
};
inline DecodeSlices decode_slices(int group) {
  DecodeSlices s;
  s.hs = group < kDecodeSliceHeads ? group : kDecodeSliceHeads;
  s.ng = s.hs > 8 ? 2 : 1;
  s.nc = (group + s.hs - 1) / s.hs;
  return s;
}

// Balanced decode schedule sizes, shared by the planner and the launcher:
// the grid (CTAs) and the most pieces (workspace rows per slice head) the
// split can produce for max_context_len; `units` = decode units per sequence.
struct DecodeBalance {
  int grid, workers;
  int64_t pieces;  // units + chunks
};
inline DecodeBalance decode_balance(int num_seqs, int units, int max_ctx, int num_sms) {
  DecodeBalance d;
  const int64_t t_max = static_cast<int64_t>(num_seqs) * units * ((max_ctx + 15) / 16) * 16;
  int64_t grid = (t_max / kDecodeSub + kDecodeWarps - 1) / kDecodeWarps;
  if (grid > static_cast<int64_t>(kDecodeCtasPerSm) * num_sms)
    grid = static_cast<int64_t>(kDecodeCtasPerSm) * num_sms;
  if (grid < 1) grid = 1;
  d.grid = static_cast<int>(grid);
  d.workers = d.grid * kDecodeWarps;
  const int64_t per = static_cast<int64_t>(d.workers) * kDecodeChunkCap;
  const int64_t k = t_max > 0 ? (t_max + per - 1) / per : 1;
  const int64_t chunks = k * d.workers;
  d.pieces = static_cast<int64_t>(num_seqs) * units + chunks;
  return d;
}

struct DecodeArgs {
  void *out;
  int64_t out_row_stride;  // elements between sequences
  const void *query;
  int64_t q_row_stride;
  const int32_t *block_table;
  int64_t block_table_stride;
  int32_t capacity;  // max_blocks_per_seq * block_size, clamped to int32
  const int32_t *context_lens;
  int32_t num_seqs, num_q_heads, num_kv_heads, head_dim, block_size;
  int64_t num_blocks;
  float scale_log2;  // scale * log2(e)
  int32_t max_context_len, partition_size, num_partitions;  // partition_size 0: balanced
  int grid;        // decode CTAs
  bool merge;      // launch the merge kernel
  float *ws_o;     // fixed: [S, Hq, num_partitions, D]; balanced: [pieces, G, D]
  float *ws_ml;    // same rows, 2 floats: max (log2 units), sum
  int32_t *ws_pref;  // balanced: [S + 1] prefix sums for the merge kernel
  // The previous kernel in the stream is this library's cache write, which
  // writes only K/V pool rows: the decode kernel may read everything else
  // before waiting for it.
  bool after_write = false;
  // The one-call step: the decode launch also writes num_new tokens' K/V
  // rows (new_k / new_v, new_stride elements apart) into the pools at
  // slot_mapping, and takes each sequence's newest row from the token
  // written to it.
  int32_t num_new = 0;
  const void *new_k = nullptr, *new_v = nullptr;
  int64_t new_stride = 0;
  const int64_t *slot_mapping = nullptr;
  void *k_pool = nullptr, *v_pool = nullptr;
  DecodeSlices slices;
  int32_t *d_error;
  pa_dtype dtype;
  // pool maps: box (64 elements | head_dim codes, 1, box_rows), swizzled
  CUtensorMap tm_k, tm_v;
  int box_rows;
  int num_sms;
  bool kv_int8 = false;  // one-byte pools with per-KV-head scales
  bool kv_fp8 = false;   // ... holding E4M3 codes rather than INT8
  const float *k_scale = nullptr, *v_scale = nullptr;
  uint64_t wait_ns = 0;  // bound of a pipeline wait (see pipeline_wait_ns)
};
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream);
// Records a failed CUDA call for pa_last_cuda_error() (this thread).
void record_cuda_error(cudaError_t e);
// Bound of the kernels' pipeline waits for the next launches: 2 s, unless a
// test shortened it through pa_debug_set_wait_limit_ns.
uint64_t pipeline_wait_ns();
size_t decode_smem_bytes(int head_dim, int num_seqs, int partition_size, int block_size,
                         bool kv_int8 = false);

struct PrefillArgs {
  void *out;
  int64_t out_row_stride;
  const void *query;
  int64_t q_row_stride;
  const int32_t *block_table;
  int64_t block_table_stride;
  int32_t capacity;
  const int32_t *cu_seqlens_q;
  const int32_t *context_lens;
  int32_t num_seqs, total_q, max_seqlen_q, max_context_len;
  int32_t num_q_heads, num_kv_heads, head_dim, block_size;
  int64_t num_blocks;
  float scale_log2;
  int32_t causal;
  int32_t *d_error;
  pa_dtype dtype;
  // Query heads packed into a tile's rows (a power of two dividing 128 and
  // the GQA group, or 1); tm_q's box is 64 x packed_heads x 128 / packed_heads.
  int packed_heads = 1;
  CUtensorMap tm_q, tm_k, tm_v;
  int num_sms;
  uint64_t wait_ns = 0;  // bound of a pipeline wait (see pipeline_wait_ns)
};
// The query heads a prefill tile packs: the whole GQA group when it is a
// power of two up to 128 (and the packed rows of the longest sequence fit in
// int32), else 1.
inline int prefill_packed_heads(int group, int max_seqlen_q) {
  if (group < 1 || group > 128 || (group & (group - 1)) != 0) return 1;
  if (static_cast<int64_t>(max_seqlen_q) * group > 0x3fffffff) return 1;
  return group;
}
cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream);

}  // namespace pa
