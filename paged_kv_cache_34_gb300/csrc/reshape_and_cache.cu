// reshape_and_cache.cu -- write new K/V rows into the paged pool.
//
// Operation (cannbot-skills "model-infer-kvcache" skill page, §3.3
// slot_mapping and App. D; lqnn.cn article §4.5 cache update): token t's K
// and V rows (all KV heads, head_dim contiguous) are copied bit for bit to
// row slot_mapping[t] of the pool viewed as [num_blocks*block_size, Hkv, D];
// that row is block slot / block_size, offset slot % block_size.  A negative
// slot writes nothing; a slot past the pool is skipped and reported.
//
// Design: pure HBM copy.  One CTA walks tokens with a grid stride; its threads
// move the token's row in 16-byte vectors (read-only non-allocating loads,
// ordinary stores), K and V interleaved so each thread keeps four
// independent 16-byte loads in flight before storing.  Destination rows are
// contiguous (Hkv*D*2 bytes), so stores coalesce fully, as the pages note.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__device__ __forceinline__ uint4 ld_nc_v4(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const uint4 *__restrict__ key, const uint4 *__restrict__ value, int64_t row_stride_vec,
    uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache,
    const int64_t *__restrict__ slot_mapping, int32_t num_tokens, int32_t row_vec,
    int64_t num_slots, int32_t *err) {
  griddep_wait();  // inputs may come from the kernel just before this one
  griddep_launch_dependents();
  for (int64_t t = blockIdx.x; t < num_tokens; t += gridDim.x) {
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (threadIdx.x == 0) raise_error(err, PA_DEVERR_SLOT);
      continue;
    }
    const uint4 *ks = key + t * row_stride_vec;
    const uint4 *vs = value + t * row_stride_vec;
    uint4 *kd = key_cache + slot * row_vec;
    uint4 *vd = value_cache + slot * row_vec;
    int i = threadIdx.x;
    for (; i + (int)blockDim.x < row_vec; i += 2 * blockDim.x) {
      const uint4 k0 = ld_nc_v4(ks + i), k1 = ld_nc_v4(ks + i + blockDim.x);
      const uint4 v0 = ld_nc_v4(vs + i), v1 = ld_nc_v4(vs + i + blockDim.x);
      kd[i] = k0;
      kd[i + blockDim.x] = k1;
      vd[i] = v0;
      vd[i + blockDim.x] = v1;
    }
    if (i < row_vec) {
      const uint4 k0 = ld_nc_v4(ks + i), v0 = ld_nc_v4(vs + i);
      kd[i] = k0;
      vd[i] = v0;
    }
  }
}

// The write into 8-bit pools (INT8 or, with FP8, E4M3 codes).
template <class E, bool FP8>
__global__ void __launch_bounds__(256) reshape_and_cache_int8_kernel(
    const uint4 *__restrict__ key, const uint4 *__restrict__ value, int64_t row_stride_vec,
    uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache,
    const int64_t *__restrict__ slot_mapping, int32_t num_tokens, int32_t row_vec8,
    int32_t head_dim, int64_t num_slots, const float *__restrict__ k_scale,
    const float *__restrict__ v_scale, int32_t *err) {
  griddep_wait();  // inputs may come from the kernel just before this one
  griddep_launch_dependents();
  for (int64_t t = blockIdx.x; t < num_tokens; t += gridDim.x) {
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (threadIdx.x == 0) raise_error(err, PA_DEVERR_SLOT);
      continue;
    }
    // 16-byte output chunk i holds elements 16i .. 16i+15 of the row (one
    // head: head_dim is a multiple of 16), read as two 16-byte input vectors.
    const uint4 *ks = key + t * row_stride_vec;
    const uint4 *vs = value + t * row_stride_vec;
    uint4 *kd = key_cache + slot * row_vec8;
    uint4 *vd = value_cache + slot * row_vec8;
    for (int i = threadIdx.x; i < row_vec8; i += blockDim.x) {
      const int g = (i * 16) / head_dim;
      const float ksc = __ldg(k_scale + g), vsc = __ldg(v_scale + g);
      const uint4 k0 = ld_nc_v4(ks + 2 * i), k1 = ld_nc_v4(ks + 2 * i + 1);
      const uint4 v0 = ld_nc_v4(vs + 2 * i), v1 = ld_nc_v4(vs + 2 * i + 1);
      const bool good = scale_ok(ksc) && scale_ok(vsc);
      if (!good) raise_error(err, PA_DEVERR_SCALE);
      const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
      kd[i] = good ? quant16<E, FP8>(k0, k1, ksc) : zero;
      vd[i] = good ? quant16<E, FP8>(v0, v1, vsc) : zero;
    }
  }
}

cudaError_t launch_reshape_and_cache(const ReshapeArgs &a, cudaStream_t stream) {
  if (a.int8) {
    const int row_vec8 = static_cast<int>(a.row_bytes / 2 / 16);  // int8 row, 16-byte units
    int threads = 256;
    if (row_vec8 < 256) threads = ((row_vec8 + 31) / 32) * 32;
    const int64_t max_ctas = static_cast<int64_t>(a.num_sms) * 16;
    const int grid = static_cast<int>(a.num_tokens < max_ctas ? a.num_tokens : max_ctas);
    auto kernel = a.fp8 ? (a.dtype == PA_BF16 ? reshape_and_cache_int8_kernel<BF16, true>
                                              : reshape_and_cache_int8_kernel<F16, true>)
                        : (a.dtype == PA_BF16 ? reshape_and_cache_int8_kernel<BF16, false>
                                              : reshape_and_cache_int8_kernel<F16, false>);
    return launch_pdl(kernel, dim3(grid), dim3(threads), 0, stream,
                      static_cast<const uint4 *>(a.key), static_cast<const uint4 *>(a.value),
                      static_cast<int64_t>(a.row_stride_bytes / 16),
                      static_cast<uint4 *>(a.key_cache), static_cast<uint4 *>(a.value_cache),
                      a.slot_mapping, a.num_tokens, row_vec8, a.head_dim, a.num_slots, a.k_scale,
                      a.v_scale, a.d_error);
  }
  const int row_vec = static_cast<int>(a.row_bytes / 16);
  int threads = 256;
  if (row_vec < 256) threads = ((row_vec + 31) / 32) * 32;
  // Enough CTAs to cover the GPU several times over; each walks tokens.
  const int64_t max_ctas = static_cast<int64_t>(a.num_sms) * 16;
  const int grid = static_cast<int>(a.num_tokens < max_ctas ? a.num_tokens : max_ctas);
  return launch_pdl(reshape_and_cache_kernel, dim3(grid), dim3(threads), 0, stream,
                    static_cast<const uint4 *>(a.key), static_cast<const uint4 *>(a.value),
                    static_cast<int64_t>(a.row_stride_bytes / 16),
                    static_cast<uint4 *>(a.key_cache), static_cast<uint4 *>(a.value_cache),
                    a.slot_mapping, a.num_tokens, row_vec, a.num_slots, a.d_error);
}

}  // namespace pa
