// pa_api.cu -- the extern "C" entry points declared in include/pa.h.
//
// Host-side only: argument validation, the split-KV plan, TMA tensor-map
// encoding, and kernel launches on the caller's stream.  Nothing here
// allocates device memory, synchronises, or reads device data.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace {

thread_local int32_t g_last_cuda_error = 0;

pa_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int32_t>(e);
  return PA_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- device properties, cached per device ---------------------------------
constexpr int kMaxDevices = 64;
int g_num_sms[kMaxDevices] = {0};

cudaError_t current_num_sms(int *out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices && g_num_sms[dev] > 0) {
    *out = g_num_sms[dev];
    return cudaSuccess;
  }
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices) g_num_sms[dev] = n;
  *out = n;
  return cudaSuccess;
}

// ---- cuTensorMapEncodeTiled through the runtime's driver entry point -----
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

// A 3-D map over rows of `heads` x `head_dim` 16-bit elements:
//   dim0 = head_dim (contiguous), dim1 = heads, dim2 = rows,
// with `row_stride` elements between rows; box (64, 1, box_rows) and
// 128-byte swizzle (the box's 64 elements are exactly one 128-byte line).
// A pool viewed as [rows, heads, head_dim] for TMA: boxes of 128 bytes of one
// head's row (64 16-bit elements, or 128 int8 codes) by box_rows rows, with
// the 128-byte swizzle the kernels' shared-memory reads expect.
// One-byte pools: boxes of one head's whole row (head_dim codes), with the
// 64-byte swizzle at head_dim 64.
bool encode_rows_map(CUtensorMap *map, const void *base, pa_dtype dtype, int head_dim,
                     int heads, int64_t rows, int64_t row_stride, int box_rows,
                     bool int8 = false, int box_heads = 1) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t eb = int8 ? 1 : 2;  // element bytes
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * eb,
                                 static_cast<cuuint64_t>(row_stride) * eb};
  const cuuint32_t box[3] = {int8 ? static_cast<cuuint32_t>(head_dim) : 64u,
                             static_cast<cuuint32_t>(box_heads),
                             static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = int8               ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapSwizzle sw =
      int8 && head_dim == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  CUresult r = enc(map, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool valid_block_size(int bs) { return bs == 8 || bs == 16 || bs == 32 || bs == 64 || bs == 128; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The automatic plan is the balanced split, as long as its positions fit in
// int32 (else fixed partitions sized by plan_partition); `units` = decode
// units (KV-head slices) per sequence.
bool use_balanced(int num_seqs, int units, int max_ctx, int partition_size) {
  if (partition_size != 0 || max_ctx <= 0) return false;
  const int64_t t = static_cast<int64_t>(num_seqs) * units * ((max_ctx + 15) / 16) * 16;
  return t < (1LL << 30);
}

// Fixed split-KV plan.  Auto: every worker warp (kDecodeWarps per CTA,
// kDecodeCtasPerSm CTAs per SM) should get about eight items of the largest possible batch, so the static
// item schedule balances; a partition is at least 64 tokens (128 when eight
// query heads share a KV head) so the partial states stay a few percent of the
// K/V bytes.
int plan_partition(int num_seqs, int num_q_heads, int num_kv_heads, int max_ctx,
                   int partition_size, int num_sms) {
  if (partition_size > 0) return partition_size;
  const long units = static_cast<long>(num_seqs > 0 ? num_seqs : 1) * num_kv_heads *
                     pa::decode_slices(num_q_heads / num_kv_heads).nc;
  const long target_items =
      static_cast<long>(num_sms) * pa::kDecodeCtasPerSm * pa::kDecodeWarps * 8;
  long P = (units * max_ctx + target_items - 1) / target_items;
  P = ((P + pa::kDecodeSub - 1) / pa::kDecodeSub) * pa::kDecodeSub;
  const long pmin = (num_q_heads / num_kv_heads) > 4 ? 128 : 64;
  if (P < pmin) P = pmin;
  if (P > (1 << 20)) P = 1 << 20;
  return static_cast<int>(P);
}

}  // namespace

namespace pa {
void record_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int32_t>(e); }

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
uint64_t pipeline_wait_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
}  // namespace pa

extern "C" {

int32_t pa_abi_version(void) { return PA_ABI_VERSION; }

int32_t pa_last_cuda_error(void) { return g_last_cuda_error; }

void pa_debug_set_wait_limit_ns(uint64_t ns) {
  pa::g_wait_ns.store(ns ? ns : pa::kDefaultWaitNs, std::memory_order_relaxed);
}

const char *pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_NULL: return "PA_ERR_NULL: a required pointer is NULL";
    case PA_ERR_SHAPE: return "PA_ERR_SHAPE: inconsistent sizes or strides";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: configuration not built";
    case PA_ERR_ALIGN: return "PA_ERR_ALIGN: pointer not 16-byte aligned or stride not x8";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing or too small";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: a CUDA runtime call failed";
  }
  return "unknown pa_status";
}

}  // extern "C"

namespace {

// Validates a cache write and fills its launch arguments; enqueues nothing.
// *empty is set when there is nothing to write.
pa_status prepare_write(const void *key, const void *value, int64_t kv_row_stride,
                        void *key_cache, void *value_cache, const int64_t *slot_mapping,
                        int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                        int32_t block_size, int64_t num_blocks, pa_dtype dtype, int32_t *d_error,
                        pa::ReshapeArgs *out, bool *empty) {
  *empty = true;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks < 0)
    return PA_ERR_SHAPE;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (!key_cache || !value_cache) return PA_ERR_NULL;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !slot_mapping) return PA_ERR_NULL;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (kv_row_stride < row) return PA_ERR_SHAPE;
  if ((row * 2) % 16 != 0 || kv_row_stride % 8 != 0) return PA_ERR_ALIGN;
  if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache))
    return PA_ERR_ALIGN;
  pa::ReshapeArgs a;
  a.key = key;
  a.value = value;
  a.row_stride_bytes = kv_row_stride * 2;
  a.key_cache = key_cache;
  a.value_cache = value_cache;
  a.slot_mapping = slot_mapping;
  a.num_tokens = num_tokens;
  a.row_bytes = row * 2;
  a.num_slots = num_blocks * block_size;
  a.d_error = d_error;
  a.num_sms = 0;  // filled in at launch
  *out = a;
  *empty = false;
  return PA_OK;
}

// The write into 8-bit pools (INT8, or E4M3 with fp8).
pa_status write_8bit(const void *key, const void *value, int64_t kv_row_stride, void *key_cache,
                     void *value_cache, const int64_t *slot_mapping, int32_t num_tokens,
                     int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                     int64_t num_blocks, const float *k_scale, const float *v_scale,
                     pa_dtype dtype, int32_t *d_error, void *stream, bool fp8) {
  pa::ReshapeArgs w;
  bool empty = true;
  const pa_status st = prepare_write(key, value, kv_row_stride, key_cache, value_cache,
                                     slot_mapping, num_tokens, num_kv_heads, head_dim, block_size,
                                     num_blocks, dtype, d_error, &w, &empty);
  if (st != PA_OK) return st;
  if (!k_scale || !v_scale) return PA_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(k_scale) | reinterpret_cast<uintptr_t>(v_scale)) & 3u)
    return PA_ERR_ALIGN;
  // int8 pool rows in 16-byte chunks, a chunk within one head
  if (head_dim % 16 != 0) return PA_ERR_ALIGN;
  if (empty) return PA_OK;
  w.int8 = true;
  w.fp8 = fp8;
  w.dtype = dtype;
  w.head_dim = head_dim;
  w.k_scale = k_scale;
  w.v_scale = v_scale;
  cudaError_t e = current_num_sms(&w.num_sms);
  if (e != cudaSuccess) return cuda_fail(e);
  e = pa::launch_reshape_and_cache(w, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

pa_status pa_reshape_and_cache(const void *key, const void *value, int64_t kv_row_stride,
                               void *key_cache, void *value_cache,
                               const int64_t *slot_mapping, int32_t num_tokens,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int64_t num_blocks, pa_dtype dtype, int32_t *d_error,
                               void *stream) {
  pa::ReshapeArgs w;
  bool empty = true;
  const pa_status st = prepare_write(key, value, kv_row_stride, key_cache, value_cache,
                                     slot_mapping, num_tokens, num_kv_heads, head_dim, block_size,
                                     num_blocks, dtype, d_error, &w, &empty);
  if (st != PA_OK || empty) return st;
  cudaError_t e = current_num_sms(&w.num_sms);
  if (e != cudaSuccess) return cuda_fail(e);
  e = pa::launch_reshape_and_cache(w, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_copy_blocks(void *key_cache, void *value_cache, int64_t block_bytes,
                         int64_t num_blocks, const int64_t *block_mapping, int32_t num_pairs,
                         int32_t *d_error, void *stream) {
  if (num_pairs < 0 || num_blocks < 0 || block_bytes <= 0) return PA_ERR_SHAPE;
  if (!key_cache || !value_cache) return PA_ERR_NULL;
  if (block_bytes % 16 != 0 || !aligned16(key_cache) || !aligned16(value_cache))
    return PA_ERR_ALIGN;
  if (num_pairs == 0) return PA_OK;
  if (!block_mapping) return PA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(block_mapping) & 7u) return PA_ERR_ALIGN;
  pa::CopyBlocksArgs a;
  a.key_cache = key_cache;
  a.value_cache = value_cache;
  a.block_bytes = block_bytes;
  a.num_blocks = num_blocks;
  a.block_mapping = block_mapping;
  a.num_pairs = num_pairs;
  a.d_error = d_error;
  cudaError_t e = current_num_sms(&a.num_sms);
  if (e != cudaSuccess) return cuda_fail(e);
  e = pa::launch_copy_blocks(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_reshape_and_cache_int8(const void *key, const void *value, int64_t kv_row_stride,
                                    void *key_cache, void *value_cache,
                                    const int64_t *slot_mapping, int32_t num_tokens,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                    int64_t num_blocks, const float *k_scale,
                                    const float *v_scale, pa_dtype dtype, int32_t *d_error,
                                    void *stream) {
  return write_8bit(key, value, kv_row_stride, key_cache, value_cache, slot_mapping, num_tokens,
                    num_kv_heads, head_dim, block_size, num_blocks, k_scale, v_scale, dtype,
                    d_error, stream, false);
}

pa_status pa_reshape_and_cache_fp8(const void *key, const void *value, int64_t kv_row_stride,
                                   void *key_cache, void *value_cache,
                                   const int64_t *slot_mapping, int32_t num_tokens,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                   int64_t num_blocks, const float *k_scale,
                                   const float *v_scale, pa_dtype dtype, int32_t *d_error,
                                   void *stream) {
  return write_8bit(key, value, kv_row_stride, key_cache, value_cache, slot_mapping, num_tokens,
                    num_kv_heads, head_dim, block_size, num_blocks, k_scale, v_scale, dtype,
                    d_error, stream, true);
}

pa_status pa_decode_plan(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t max_context_len, int32_t partition_size,
                         int32_t *partition_size_out, size_t *workspace_bytes_out) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_context_len < 0 || partition_size < 0)
    return PA_ERR_SHAPE;
  if (partition_size % pa::kDecodeSub != 0) return PA_ERR_SHAPE;
  int sms = 0;
  cudaError_t e = current_num_sms(&sms);
  if (e != cudaSuccess) return cuda_fail(e);
  size_t ws = 0;
  int P = 0;
  if (num_q_heads % num_kv_heads != 0) return PA_ERR_SHAPE;
  const pa::DecodeSlices sl = pa::decode_slices(num_q_heads / num_kv_heads);
  if (use_balanced(num_seqs, num_kv_heads * sl.nc, max_context_len, partition_size)) {
    // Balanced split (P reported as 0): pieces x (heads per slice) rows of
    // partial state, plus the per-sequence prefix sums for the merge kernel.
    const pa::DecodeBalance d =
        pa::decode_balance(num_seqs, num_kv_heads * sl.nc, max_context_len, sms);
    const size_t rows = static_cast<size_t>(d.pieces) * sl.hs;
    ws = align256(rows * head_dim * sizeof(float)) + align256(rows * 2 * sizeof(float)) +
         align256((static_cast<size_t>(num_seqs) + 1) * sizeof(int32_t));
  } else {
    P = plan_partition(num_seqs, num_q_heads, num_kv_heads, max_context_len, partition_size,
                       sms);
    const int64_t nparts = max_context_len > 0 ? (max_context_len + P - 1) / P : 1;
    if (nparts > 1) {
      const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * nparts;
      ws = align256(rows * head_dim * sizeof(float)) + align256(rows * 2 * sizeof(float));
    }
  }
  if (partition_size_out) *partition_size_out = P;
  if (workspace_bytes_out) *workspace_bytes_out = ws;
  return PA_OK;
}

}  // extern "C"

namespace {

// pa_decode, optionally preceded by the step's cache write `write` (launched
// first, after every check has passed, so an error enqueues nothing).
pa_status decode_call(void *out, int64_t out_row_stride, const void *query, int64_t q_row_stride,
                      const void *key_cache, const void *value_cache, const int32_t *block_table,
                      int64_t block_table_stride, int32_t max_blocks_per_seq,
                      const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                      int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                      int64_t num_blocks, float scale, int32_t max_context_len,
                      int32_t partition_size, void *workspace, size_t workspace_bytes,
                      pa_dtype dtype, int32_t *d_error, void *stream,
                      const pa::ReshapeArgs *write, const float *k_scale = nullptr,
                      const float *v_scale = nullptr, bool fp8 = false) {
  const bool int8 = k_scale != nullptr || v_scale != nullptr;
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq < 0 || max_context_len < 0 ||
      partition_size < 0)
    return PA_ERR_SHAPE;
  if (num_q_heads % num_kv_heads != 0) return PA_ERR_SHAPE;
  if (block_table_stride < max_blocks_per_seq) return PA_ERR_SHAPE;
  if (!isfinite(scale)) return PA_ERR_SHAPE;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (!valid_block_size(block_size)) return PA_ERR_UNSUPPORTED;
  if (num_blocks * block_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (partition_size % pa::kDecodeSub != 0) return PA_ERR_SHAPE;
  if (num_seqs == 0) {  // nothing to attend: only the step's write, if any
    if (!write) return PA_OK;
    pa::ReshapeArgs w = *write;
    cudaError_t e = current_num_sms(&w.num_sms);
    if (e == cudaSuccess) e = pa::launch_reshape_and_cache(w, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
  }
  if (!out || !query || !key_cache || !value_cache || !block_table || !context_lens)
    return PA_ERR_NULL;
  const int64_t qrow = static_cast<int64_t>(num_q_heads) * head_dim;
  if (q_row_stride < qrow || out_row_stride < qrow) return PA_ERR_SHAPE;
  if (q_row_stride % 8 || out_row_stride % 8) return PA_ERR_ALIGN;
  if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache))
    return PA_ERR_ALIGN;
  if (int8) {
    if (!k_scale || !v_scale) return PA_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(k_scale) | reinterpret_cast<uintptr_t>(v_scale)) & 3u)
      return PA_ERR_ALIGN;
  }

  int32_t P = 0;
  size_t need = 0;
  pa_status st = pa_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                                partition_size, &P, &need);
  if (st != PA_OK) return st;
  const bool balanced = P == 0;
  const int32_t nparts = balanced ? 0 : (max_context_len > 0 ? (max_context_len + P - 1) / P : 1);
  if (need > 0 && (!workspace || workspace_bytes < need ||
                   (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return PA_ERR_WORKSPACE;

  pa::DecodeArgs a;
  a.out = out;
  a.out_row_stride = out_row_stride;
  a.query = query;
  a.q_row_stride = q_row_stride;
  a.block_table = block_table;
  a.block_table_stride = block_table_stride;
  const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * block_size;
  a.capacity = static_cast<int32_t>(cap > INT32_MAX ? INT32_MAX : cap);
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.max_context_len = max_context_len;
  a.partition_size = P;
  a.num_partitions = nparts;
  a.ws_o = nullptr;
  a.ws_ml = nullptr;
  a.ws_pref = nullptr;
  a.slices = pa::decode_slices(num_q_heads / num_kv_heads);
  const int units = num_kv_heads * a.slices.nc;  // decode units per sequence
  cudaError_t e = current_num_sms(&a.num_sms);
  if (e != cudaSuccess) return cuda_fail(e);
  if (balanced) {
    const pa::DecodeBalance d = pa::decode_balance(num_seqs, units, max_context_len, a.num_sms);
    a.grid = d.grid;
    a.merge = true;
    const size_t rows = static_cast<size_t>(d.pieces) * a.slices.hs;
    char *w = static_cast<char *>(workspace);
    a.ws_o = reinterpret_cast<float *>(w);
    w += align256(rows * head_dim * sizeof(float));
    a.ws_ml = reinterpret_cast<float *>(w);
    w += align256(rows * 2 * sizeof(float));
    a.ws_pref = reinterpret_cast<int32_t *>(w);
  } else {
    // Items are at most S * units * partitions; kDecodeCtasPerSm CTAs per SM,
    // kDecodeWarps workers each.
    const int64_t items = static_cast<int64_t>(num_seqs) * units * nparts;
    int64_t grid = (items + pa::kDecodeWarps - 1) / pa::kDecodeWarps;
    if (grid > static_cast<int64_t>(pa::kDecodeCtasPerSm) * a.num_sms)
      grid = static_cast<int64_t>(pa::kDecodeCtasPerSm) * a.num_sms;
    if (grid < 1) grid = 1;
    a.grid = static_cast<int>(grid);
    a.merge = nparts > 1;
    if (need > 0) {
      const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * nparts;
      a.ws_o = static_cast<float *>(workspace);
      a.ws_ml = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                          align256(rows * head_dim * sizeof(float)));
    }
  }
  a.d_error = d_error;
  a.dtype = dtype;
  a.wait_ns = pa::pipeline_wait_ns();
  a.box_rows = block_size < pa::kDecodeSub ? block_size : pa::kDecodeSub;
  // The item schedule keeps per-sequence prefix sums in shared memory.
  if (pa::decode_smem_bytes(head_dim, num_seqs, P, block_size, int8) > 227 * 1024)
    return PA_ERR_UNSUPPORTED;
  const int64_t rows = num_blocks * block_size;
  const int64_t row_stride = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (!encode_rows_map(&a.tm_k, key_cache, dtype, head_dim, num_kv_heads, rows, row_stride,
                       a.box_rows, int8) ||
      !encode_rows_map(&a.tm_v, value_cache, dtype, head_dim, num_kv_heads, rows, row_stride,
                       a.box_rows, int8))
    return cuda_fail(cudaErrorInvalidValue);
  a.kv_int8 = int8;
  a.kv_fp8 = int8 && fp8;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  if (write && (!balanced || int8)) {
    // Fixed partitions or one-byte pools: the write is its own launch; the
    // decode kernel reads context_lens, block_table and the query at once
    // and waits for the write (programmatic dependent launch) only before
    // its first K/V load.
    pa::ReshapeArgs w = *write;
    w.num_sms = a.num_sms;
    e = pa::launch_reshape_and_cache(w, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    a.after_write = true;
  } else if (write) {
    // 16-bit pools, balanced schedule: the step's cache write runs inside
    // the decode launch.
    a.num_new = write->num_tokens;
    a.new_k = write->key;
    a.new_v = write->value;
    a.new_stride = write->row_stride_bytes / 2;
    a.slot_mapping = write->slot_mapping;
    a.k_pool = write->key_cache;
    a.v_pool = write->value_cache;
  }
  e = pa::launch_decode(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

pa_status pa_decode(void *out, int64_t out_row_stride, const void *query, int64_t q_row_stride,
                    const void *key_cache, const void *value_cache, const int32_t *block_table,
                    int64_t block_table_stride, int32_t max_blocks_per_seq,
                    const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                    int64_t num_blocks, float scale, int32_t max_context_len,
                    int32_t partition_size, void *workspace, size_t workspace_bytes,
                    pa_dtype dtype, int32_t *d_error, void *stream) {
  return decode_call(out, out_row_stride, query, q_row_stride, key_cache, value_cache,
                     block_table, block_table_stride, max_blocks_per_seq, context_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                     max_context_len, partition_size, workspace, workspace_bytes, dtype, d_error,
                     stream, nullptr);
}

pa_status pa_decode_int8(void *out, int64_t out_row_stride, const void *query,
                         int64_t q_row_stride, const void *key_cache, const void *value_cache,
                         const int32_t *block_table, int64_t block_table_stride,
                         int32_t max_blocks_per_seq, const int32_t *context_lens,
                         int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, int64_t num_blocks,
                         const float *k_scale, const float *v_scale, float scale,
                         int32_t max_context_len, int32_t partition_size, void *workspace,
                         size_t workspace_bytes, pa_dtype dtype, int32_t *d_error,
                         void *stream) {
  if (!k_scale || !v_scale) return PA_ERR_NULL;
  return decode_call(out, out_row_stride, query, q_row_stride, key_cache, value_cache,
                     block_table, block_table_stride, max_blocks_per_seq, context_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                     max_context_len, partition_size, workspace, workspace_bytes, dtype, d_error,
                     stream, nullptr, k_scale, v_scale);
}

pa_status pa_decode_fp8(void *out, int64_t out_row_stride, const void *query,
                        int64_t q_row_stride, const void *key_cache, const void *value_cache,
                        const int32_t *block_table, int64_t block_table_stride,
                        int32_t max_blocks_per_seq, const int32_t *context_lens,
                        int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, int32_t block_size, int64_t num_blocks,
                        const float *k_scale, const float *v_scale, float scale,
                        int32_t max_context_len, int32_t partition_size, void *workspace,
                        size_t workspace_bytes, pa_dtype dtype, int32_t *d_error,
                        void *stream) {
  if (!k_scale || !v_scale) return PA_ERR_NULL;
  return decode_call(out, out_row_stride, query, q_row_stride, key_cache, value_cache,
                     block_table, block_table_stride, max_blocks_per_seq, context_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                     max_context_len, partition_size, workspace, workspace_bytes, dtype, d_error,
                     stream, nullptr, k_scale, v_scale, true);
}

pa_status pa_decode_write(void *out, int64_t out_row_stride, const void *query,
                          int64_t q_row_stride, const void *key, const void *value,
                          int64_t kv_row_stride, void *key_cache, void *value_cache,
                          const int64_t *slot_mapping, int32_t num_new_tokens,
                          const int32_t *block_table, int64_t block_table_stride,
                          int32_t max_blocks_per_seq, const int32_t *context_lens,
                          int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, int32_t block_size, int64_t num_blocks, float scale,
                          int32_t max_context_len, int32_t partition_size, void *workspace,
                          size_t workspace_bytes, pa_dtype dtype, int32_t *d_error,
                          void *stream) {
  pa::ReshapeArgs w;
  bool empty = true;
  const pa_status st = prepare_write(key, value, kv_row_stride, key_cache, value_cache,
                                     slot_mapping, num_new_tokens, num_kv_heads, head_dim,
                                     block_size, num_blocks, dtype, d_error, &w, &empty);
  if (st != PA_OK) return st;
  return decode_call(out, out_row_stride, query, q_row_stride, key_cache, value_cache,
                     block_table, block_table_stride, max_blocks_per_seq, context_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                     max_context_len, partition_size, workspace, workspace_bytes, dtype, d_error,
                     stream, empty ? nullptr : &w);
}

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
                               int32_t *d_error, void *stream) {
  if (!k_scale || !v_scale) return PA_ERR_NULL;
  pa::ReshapeArgs w;
  bool empty = true;
  const pa_status st = prepare_write(key, value, kv_row_stride, key_cache, value_cache,
                                     slot_mapping, num_new_tokens, num_kv_heads, head_dim,
                                     block_size, num_blocks, dtype, d_error, &w, &empty);
  if (st != PA_OK) return st;
  w.int8 = true;
  w.dtype = dtype;
  w.head_dim = head_dim;
  w.k_scale = k_scale;
  w.v_scale = v_scale;
  return decode_call(out, out_row_stride, query, q_row_stride, key_cache, value_cache,
                     block_table, block_table_stride, max_blocks_per_seq, context_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                     max_context_len, partition_size, workspace, workspace_bytes, dtype, d_error,
                     stream, empty ? nullptr : &w, k_scale, v_scale);
}

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
                              int32_t *d_error, void *stream) {
  if (!k_scale || !v_scale) return PA_ERR_NULL;
  pa::ReshapeArgs w;
  bool empty = true;
  const pa_status st = prepare_write(key, value, kv_row_stride, key_cache, value_cache,
                                     slot_mapping, num_new_tokens, num_kv_heads, head_dim,
                                     block_size, num_blocks, dtype, d_error, &w, &empty);
  if (st != PA_OK) return st;
  w.int8 = true;
  w.fp8 = true;
  w.dtype = dtype;
  w.head_dim = head_dim;
  w.k_scale = k_scale;
  w.v_scale = v_scale;
  return decode_call(out, out_row_stride, query, q_row_stride, key_cache, value_cache,
                     block_table, block_table_stride, max_blocks_per_seq, context_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                     max_context_len, partition_size, workspace, workspace_bytes, dtype, d_error,
                     stream, empty ? nullptr : &w, k_scale, v_scale, true);
}

pa_status pa_prefill_varlen(void *out, int64_t out_row_stride, const void *query,
                            int64_t q_row_stride, const void *key_cache,
                            const void *value_cache, const int32_t *block_table,
                            int64_t block_table_stride, int32_t max_blocks_per_seq,
                            const int32_t *cu_seqlens_q, const int32_t *context_lens,
                            int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
                            int32_t max_context_len, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int64_t num_blocks, float scale, int32_t causal, pa_dtype dtype,
                            int32_t *d_error, void *stream) {
  if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || max_context_len < 0 ||
      num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_blocks <= 0 || max_blocks_per_seq < 0)
    return PA_ERR_SHAPE;
  if (num_q_heads % num_kv_heads != 0) return PA_ERR_SHAPE;
  if (block_table_stride < max_blocks_per_seq) return PA_ERR_SHAPE;
  if (!isfinite(scale)) return PA_ERR_SHAPE;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (!(block_size == 16 || block_size == 32 || block_size == 64 || block_size == 128))
    return PA_ERR_UNSUPPORTED;
  if (num_blocks * block_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_q == 0) return PA_OK;
  if (!out || !query || !key_cache || !value_cache || !block_table || !cu_seqlens_q ||
      !context_lens)
    return PA_ERR_NULL;
  const int64_t qrow = static_cast<int64_t>(num_q_heads) * head_dim;
  if (q_row_stride < qrow || out_row_stride < qrow) return PA_ERR_SHAPE;
  if (q_row_stride % 8 || out_row_stride % 8) return PA_ERR_ALIGN;
  if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache))
    return PA_ERR_ALIGN;

  pa::PrefillArgs a;
  a.out = out;
  a.out_row_stride = out_row_stride;
  a.query = query;
  a.q_row_stride = q_row_stride;
  a.block_table = block_table;
  a.block_table_stride = block_table_stride;
  const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * block_size;
  a.capacity = static_cast<int32_t>(cap > INT32_MAX ? INT32_MAX : cap);
  a.cu_seqlens_q = cu_seqlens_q;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.total_q = total_q;
  a.max_seqlen_q = max_seqlen_q;
  a.max_context_len = max_context_len;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.causal = causal ? 1 : 0;
  a.d_error = d_error;
  a.dtype = dtype;
  a.wait_ns = pa::pipeline_wait_ns();
  cudaError_t e = current_num_sms(&a.num_sms);
  if (e != cudaSuccess) return cuda_fail(e);
  const int64_t kv_rows = num_blocks * block_size;
  const int64_t kv_stride = static_cast<int64_t>(num_kv_heads) * head_dim;
  const int box = block_size;  // one box per block
  // The query tile is 128 rows: 128 / pg tokens x the pg query heads of one
  // KV head, the heads of a token adjacent.
  a.packed_heads = pa::prefill_packed_heads(num_q_heads / num_kv_heads, max_seqlen_q);
  if (!encode_rows_map(&a.tm_q, query, dtype, head_dim, num_q_heads, total_q, q_row_stride,
                       128 / a.packed_heads, false, a.packed_heads) ||
      !encode_rows_map(&a.tm_k, key_cache, dtype, head_dim, num_kv_heads, kv_rows, kv_stride,
                       box) ||
      !encode_rows_map(&a.tm_v, value_cache, dtype, head_dim, num_kv_heads, kv_rows, kv_stride,
                       box))
    return cuda_fail(cudaErrorInvalidValue);
  e = pa::launch_prefill(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // extern "C"
