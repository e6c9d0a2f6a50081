// pa_device.cuh -- device-side building blocks shared by the sm_103a kernels
// of the paged-KV attention library: the 16-bit element traits, the device
// error flag, bounded mbarrier waits, TMA tile loads, and the warp-level
// tensor-core fragments (ldmatrix / mma.sync / movmatrix) used by decode.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <utility>

#include "pa.h"

namespace pa {

// ---------------------------------------------------------------------------
// Element types
// ---------------------------------------------------------------------------
struct F16 {
  using T = __half;
  using T2 = __half2;
  static constexpr bool kBF16 = false;
  static __device__ __forceinline__ T from_float(float x) { return __float2half_rn(x); }
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  }
  // a += low half of w, b += high half, each widened exactly (mixed-precision
  // add.f32.f16: no separate unpacking instructions).
  static __device__ __forceinline__ void add_halves(uint32_t w, float &a, float &b) {
    asm("{\n\t.reg .b16 l16, h16;\n\tmov.b32 {l16, h16}, %2;\n\t"
        "add.rn.f32.f16 %0, l16, %0;\n\tadd.rn.f32.f16 %1, h16, %1;\n\t}"
        : "+f"(a), "+f"(b)
        : "r"(w));
  }
  static __device__ __forceinline__ float lo(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
  }
  static __device__ __forceinline__ float hi(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
  }
};
struct BF16 {
  using T = __nv_bfloat16;
  using T2 = __nv_bfloat162;
  static constexpr bool kBF16 = true;
  static __device__ __forceinline__ T from_float(float x) { return __float2bfloat16_rn(x); }
  static __device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  }
  static __device__ __forceinline__ void add_halves(uint32_t w, float &a, float &b) {
    asm("{\n\t.reg .b16 l16, h16;\n\tmov.b32 {l16, h16}, %2;\n\t"
        "add.rn.f32.bf16 %0, l16, %0;\n\tadd.rn.f32.bf16 %1, h16, %1;\n\t}"
        : "+f"(a), "+f"(b)
        : "r"(w));
  }
  static __device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
  static __device__ __forceinline__ float hi(uint32_t w) {
    return __uint_as_float(w & 0xffff0000u);
  }
};

// ---------------------------------------------------------------------------
// Host: lift a kernel's dynamic shared-memory limit to the device maximum,
// once per device.  The attribute call can wait for work in flight, so it
// must not run on every launch.
// ---------------------------------------------------------------------------
template <auto Kernel>
cudaError_t allow_dynamic_smem() {
  static int done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  int max_optin = 0;
  e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_optin);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = 1;
  return e;
}

// ---------------------------------------------------------------------------
// Device error flag (caller-owned int32, may be null)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void raise_error(int32_t *flag, int32_t bits) {
  if (flag) atomicOr(flag, bits);
}

// Context length as the kernels use it: a negative length, one beyond the
// block table's capacity, or one above the host's max_context_len hint is
// reported and treated as empty (the sequence's output is zero).
__device__ __forceinline__ int checked_context_len(int len, int capacity, int hint,
                                                   int32_t *err, bool report) {
  if (len < 0 || len > capacity || len > hint) {
    if (report) raise_error(err, PA_DEVERR_CONTEXT);
    return 0;
  }
  return len;
}

// ---------------------------------------------------------------------------
// One-byte pool codes: the write's quantiser (also used by the one-call
// decode step for the newest row, so both give the same codes)
// ---------------------------------------------------------------------------
// INT8 pools: each KV head's values are stored as round-half-even(x /
// scale) clamped to [-127, 127] (NaN -> 0), the division and the rounding in
// fp32 (cannbot-skills page, App. A quantised-KV scales; the formula is this
// library's reading).  A scale that is not a positive finite number stores 0
// and reports PA_DEVERR_SCALE.
__device__ __forceinline__ bool scale_ok(float s) { return s > 0.0f && s <= 3.4028234663852886e38f; }

// x / s rounded to nearest (ties to even) in fp32, for a positive finite s
// and its correctly rounded reciprocal r = RN(1/s): q0 = RN(x r) is within
// an ulp of x / s, the remainder x - q0 s is exact with one fused
// multiply-add, and RN(q0 + remainder * r) is then the correctly rounded
// quotient (Markstein's division theorem; P. Markstein, IBM J. Res. Dev.
// 34(1), 1990).  It holds while the quotient is a normal number; below that
// the result is still within the subnormal range, and an infinite first
// product is returned as is -- either way the codes built from it below are
// those of the exactly rounded quotient.  The result takes x's sign (s > 0),
// which a zero remainder step would otherwise lose for x = -0.
__device__ __forceinline__ float div_rn_recip(float x, float s, float r) {
  const float q0 = __fmul_rn(x, r);
  if (isinf(q0)) return q0;
  const float e = __fmaf_rn(-q0, s, x);
  return copysignf(__fmaf_rn(e, r, q0), x);
}

__device__ __forceinline__ uint32_t code8(float x, float s, float r) {
  if (x != x) return 0u;
  int c = __float2int_rn(div_rn_recip(x, s, r));
  c = c > 127 ? 127 : (c < -127 ? -127 : c);
  return static_cast<uint32_t>(c) & 0xffu;
}

// FP8 pools: each value is stored as the nearest E4M3 value (ties to even,
// saturating at +-448) to x / scale, the division in fp32; NaN -> 0 (the same
// reading of the pages' quantised-KV scales, with the OCP E4M3 format).  Two
// values per conversion: `lo` in the low byte.
__device__ __forceinline__ uint32_t fp8_pair(float lo, float hi, float s, float r) {
  const float a = lo != lo ? 0.0f : div_rn_recip(lo, s, r);
  const float b = hi != hi ? 0.0f : div_rn_recip(hi, s, r);
  uint16_t pair;
  // the first source goes to the upper byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(b), "f"(a));
  return pair;
}

// 16 values with the plain division, for a subnormal scale (outside the
// conditions of the reciprocal route above): kept out of line, it is never
// the common path.
template <class E, bool FP8>
__device__ __noinline__ uint4 quant16_div(uint4 a, uint4 b, float s) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t out[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float v[4] = {E::lo(w[2 * q]), E::hi(w[2 * q]), E::lo(w[2 * q + 1]), E::hi(w[2 * q + 1])};
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = v[k] != v[k] ? 0.0f : __fdiv_rn(v[k], s);
    if constexpr (FP8) {
      uint16_t lo, hi;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(v[1]), "f"(v[0]));
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(v[3]), "f"(v[2]));
      out[q] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    } else {
      uint32_t c4 = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        int c = __float2int_rn(v[k]);
        c = c > 127 ? 127 : (c < -127 ? -127 : c);
        c4 |= (static_cast<uint32_t>(c) & 0xffu) << (8 * k);
      }
      out[q] = c4;
    }
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// 16 values (two 16-byte vectors of fp16/bf16 pairs) -> 16 codes.
template <class E, bool FP8>
__device__ __forceinline__ uint4 quant16(const uint4 &a, const uint4 &b, float s) {
  if (!(s >= 1.17549435e-38f)) return quant16_div<E, FP8>(a, b, s);  // subnormal scale
  const float r = __frcp_rn(s);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t out[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t w0 = w[2 * q], w1 = w[2 * q + 1];
    if constexpr (FP8) {
      out[q] = fp8_pair(E::lo(w0), E::hi(w0), s, r) |
               (fp8_pair(E::lo(w1), E::hi(w1), s, r) << 16);
    } else {
      out[q] = code8(E::lo(w0), s, r) | (code8(E::hi(w0), s, r) << 8) |
               (code8(E::lo(w1), s, r) << 16) | (code8(E::hi(w1), s, r) << 24);
    }
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarriers, bounded waits
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Upper bound on any single pipeline wait.  Far above any legitimate wait
// (microseconds), far below a hung GPU: a wait that exceeds it reports
// PA_DEVERR_TIMEOUT and lets the block return.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Waits for the phase of `bar` with the given parity to complete.  Returns
// false if the bound was reached.  Pipeline waits take the launch's bound
// (kWaitLimitNs unless a test shortened it); waits for a block's own copies
// in flight before it leaves keep kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - start > limit_ns) return false;
  }
}

// 2^x on the special-function unit (PTX ex2.approx, flush-to-zero): the
// hardware instruction, not a library routine; 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// Packed fp32 pairs (sm_100-family f32x2 arithmetic)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) loads into shared memory
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of one box at coordinates (c0, c1, c2) (innermost first).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// 4-byte asynchronous global -> shared copies (no register staging).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_8(uint32_t dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
// 16-byte asynchronous global -> shared copy through L2 only.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Warp-level tensor-core fragments (decode)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                            uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                                  uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// Transposes an 8x8 b16 matrix held one 32-bit pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// D(16x8, f32) += A(16x16) * B(16x8), A row-major, B column-major.
template <bool kBF16>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (kBF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  The library's kernels are launched so that
// they may start while the previous kernel in the stream is still running;
// each one waits for that kernel's completion (and its memory) before it
// reads anything, and lets the next kernel start launching right away.
// Both are no-ops for a kernel launched the ordinary way.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Host: launch `kernel` with programmatic stream serialization allowed.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace pa
