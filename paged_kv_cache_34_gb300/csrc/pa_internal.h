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
};
cudaError_t launch_reshape_and_cache(const ReshapeArgs &a, cudaStream_t stream);

// Decode tiling shared by the planner and the kernels.
constexpr int kDecodeWarps = 4;     // consumer warps (independent workers) per CTA
constexpr int kDecodeSub = 16;      // tokens per worker per pipeline stage
constexpr int kDecodeMaxGroup = 8;  // query heads per KV head

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
  int32_t max_context_len, partition_size, num_partitions;
  float *ws_o;   // [S, Hq, num_partitions, D]      (num_partitions > 1)
  float *ws_ml;  // [S, Hq, num_partitions, 2]      (max in log2 units, sum)
  int32_t *d_error;
  pa_dtype dtype;
  CUtensorMap tm_k, tm_v;  // pool maps, box (64, 1, box_rows), 128B swizzle
  int box_rows;
  int num_sms;
};
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream);
size_t decode_smem_bytes(int head_dim, int num_seqs, int partition_size, int block_size);

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
  CUtensorMap tm_q, tm_k, tm_v;
  int num_sms;
};
cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream);

}  // namespace pa
