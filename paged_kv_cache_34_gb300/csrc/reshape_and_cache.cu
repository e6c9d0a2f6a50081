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

// INT8 pools: each KV head's values are stored as round-half-even(x /
// scale) clamped to [-127, 127] (NaN -> 0), the division and the rounding in
// fp32 (cannbot-skills page, App. A quantised-KV scales; the formula is this
// library's reading).  A scale that is not a positive finite number stores 0
// and reports PA_DEVERR_SCALE.
__device__ __forceinline__ bool scale_ok(float s) { return s > 0.0f && s <= 3.4028234663852886e38f; }

__device__ __forceinline__ uint32_t code8(float x, float s) {
  if (x != x) return 0u;
  int c = __float2int_rn(__fdiv_rn(x, s));
  c = c > 127 ? 127 : (c < -127 ? -127 : c);
  return static_cast<uint32_t>(c) & 0xffu;
}

// FP8 pools: each value is stored as the nearest E4M3 value (ties to even,
// saturating at +-448) to x / scale, the division in fp32; NaN -> 0 (the same
// reading of the pages' quantised-KV scales, with the OCP E4M3 format).  Two
// values per conversion: `lo` in the low byte.
__device__ __forceinline__ uint32_t fp8_pair(float lo, float hi, float s) {
  const float a = lo != lo ? 0.0f : __fdiv_rn(lo, s);
  const float b = hi != hi ? 0.0f : __fdiv_rn(hi, s);
  uint16_t r;
  // the first source goes to the upper byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// 16 values (two 16-byte vectors of fp16/bf16 pairs) -> 16 codes.
template <class E, bool FP8>
__device__ __forceinline__ uint4 quant16(const uint4 &a, const uint4 &b, float s) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t out[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t w0 = w[2 * q], w1 = w[2 * q + 1];
    if constexpr (FP8) {
      out[q] = fp8_pair(E::lo(w0), E::hi(w0), s) | (fp8_pair(E::lo(w1), E::hi(w1), s) << 16);
    } else {
      out[q] = code8(E::lo(w0), s) | (code8(E::hi(w0), s) << 8) |
               (code8(E::lo(w1), s) << 16) | (code8(E::hi(w1), s) << 24);
    }
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
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
