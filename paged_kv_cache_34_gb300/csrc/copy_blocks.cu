// copy_blocks.cu -- copy-on-write of whole blocks of the K and V pools.
//
// Operation (coreui.cn "Ascend CANN ATB KV Cache and PagedAttention", the
// "page update race" section: before a request appends K/V to a page that
// other requests share, it takes a free page and copies the whole page into
// it): for each pair p, block block_mapping[2p + 1] of the K pool and of the
// V pool receives block block_mapping[2p], bit for bit.  A pair naming a
// block outside the pool copies nothing and is reported.
//
// Design: pure HBM copy, element type irrelevant.  A work unit is one 16 KB
// slice of one block of one pool; CTAs walk the units with a grid stride and
// every thread moves four 16-byte vectors, all four loads in flight before
// the stores.  A block is contiguous, so loads and stores coalesce fully.
// Loads are coherent (the pools are written in the same launch) and do not
// allocate in L1.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyVec = 4;                                 // 16-byte vectors per thread
constexpr int64_t kSliceVec = kCopyThreads * kCopyVec;      // 16-byte vectors per unit
constexpr int kCopyCtasPerSm = 8;

__device__ __forceinline__ uint4 ld_stream_v4(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(
    uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache, int64_t block_vec,
    int64_t num_blocks, const int64_t *__restrict__ block_mapping, int32_t num_pairs,
    int64_t slices, int32_t *err) {
  griddep_wait();  // the pools and the mapping may come from the kernel before
  griddep_launch_dependents();
  const int64_t per_pair = 2 * slices;  // K slices, then V slices
  const int64_t units = static_cast<int64_t>(num_pairs) * per_pair;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int64_t pair = u / per_pair;
    const int64_t r = u - pair * per_pair;
    const bool is_v = r >= slices;
    const int64_t slice = is_v ? r - slices : r;
    const int64_t src = __ldg(block_mapping + 2 * pair);
    const int64_t dst = __ldg(block_mapping + 2 * pair + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (r == 0 && threadIdx.x == 0) raise_error(err, PA_DEVERR_BLOCK_ID);
      continue;
    }
    uint4 *pool = is_v ? value_cache : key_cache;
    const int64_t off = slice * kSliceVec;
    const uint4 *s = pool + src * block_vec + off;
    uint4 *d = pool + dst * block_vec + off;
    const int64_t n = block_vec - off < kSliceVec ? block_vec - off : kSliceVec;
    uint4 v[kCopyVec];
#pragma unroll
    for (int k = 0; k < kCopyVec; ++k) {
      const int64_t i = threadIdx.x + k * kCopyThreads;
      if (i < n) v[k] = ld_stream_v4(s + i);
    }
#pragma unroll
    for (int k = 0; k < kCopyVec; ++k) {
      const int64_t i = threadIdx.x + k * kCopyThreads;
      if (i < n) d[i] = v[k];
    }
  }
}

}  // namespace

cudaError_t launch_copy_blocks(const CopyBlocksArgs &a, cudaStream_t stream) {
  const int64_t block_vec = a.block_bytes / 16;
  const int64_t slices = (block_vec + kSliceVec - 1) / kSliceVec;
  const int64_t units = static_cast<int64_t>(a.num_pairs) * 2 * slices;
  if (units == 0) return cudaSuccess;
  const int64_t max_ctas = static_cast<int64_t>(a.num_sms) * kCopyCtasPerSm;
  const int grid = static_cast<int>(units < max_ctas ? units : max_ctas);
  return launch_pdl(copy_blocks_kernel, dim3(grid), dim3(kCopyThreads), 0, stream,
                    static_cast<uint4 *>(a.key_cache), static_cast<uint4 *>(a.value_cache),
                    block_vec, a.num_blocks, a.block_mapping, a.num_pairs, slices, a.d_error);
}

}  // namespace pa
