// decode.cu -- paged attention for one query token per sequence.
//
// Operation (cannbot-skills "model-infer-kvcache" skill page §3.1 mapping,
// §3.6 decode data flow, App. C sparse_mode 0; mhpq.cn article §3.3
// paged_attention; "vLLM on CANN" block loop with online softmax): for
// sequence b, query head h and KV head g = h / G, the keys and values of
// logical positions 0..L-1 are read through block_table, and
//     out = sum_j softmax_j(scale * q . K_j) V_j.
//
// Design for sm_103a (the pages' Ascend kernels walk one page per step with
// a scalar online softmax; this keeps the block walk and the online softmax
// but is shaped for HBM bandwidth):
//
//  * Grid (partition, KV head, sequence).  A sequence's context is cut into
//    partitions of P tokens (split-KV); each CTA streams one partition of
//    one KV head and serves all G query heads of that KV head from the same
//    bytes (GQA sharing).  When a sequence spans several partitions each CTA
//    writes its softmax state (max, sum, unnormalised output) to workspace
//    and a combine kernel merges them by log-sum-exp.
//  * One producer warp stages the partition's block-table slice in shared
//    memory once, then issues TMA tile loads (128-byte swizzled, one box per
//    (block, D/64 half)) into a 3-stage ring of 64-token K/V chunks guarded
//    by mbarriers.  Two CTAs fit per SM, so six chunks are in flight.
//  * Four consumer warps each own 16 tokens of a chunk.  Scores are computed
//    transposed on the tensor cores -- S^T[16 tokens x 8 heads] =
//    K[16 x D] Q^T[D x 8] with mma.sync m16n8k16, fp32 accumulate -- so the G
//    heads fill the N=8 side and no rows are padding for G = 8.  The online
//    softmax runs on the fragments (warp-shuffle max over tokens), P^T is
//    formed with movmatrix, and O^T[D x 8] += V^T[D x 16] P^T[16 x 8] reads V
//    through ldmatrix.trans.  The partition's four warp states are merged in
//    shared memory at the end.
//  * Exponentials are base 2 with the scale pre-multiplied by log2(e).
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kThreads = (kDecodeWarps + 1) * 32;  // + producer warp
constexpr int kStages = 3;
constexpr int kHalfBytes = kDecodeChunk * 128;  // 64 tokens x 64 elements x 2 B

template <int D>
struct DecodeSmem {
  static constexpr int kHalves = D / 64;
  static constexpr int kStageBytes = 2 * kHalves * kHalfBytes;  // K + V
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kFlagOffset = kBarOffset + 2 * kStages * 8;
  static constexpr int kBlkOffset = kFlagOffset + 16;
  static int bytes(int max_blocks) { return 1024 + kBlkOffset + 4 * max_blocks; }
};

struct DecodeParams {
  void *out;
  int64_t out_row_stride;
  const void *q;
  int64_t q_row_stride;
  const int32_t *block_table;
  int64_t bt_stride;
  const int32_t *context_lens;
  int32_t capacity, max_ctx;
  int32_t hq, hkv, group, block_size;
  int64_t num_blocks;
  float scale_log2;
  int32_t partition_size, num_partitions;
  float *ws_o, *ws_ml;
  int32_t *err;
};

__device__ __forceinline__ float shfl_xor(float v, int m) {
  return __shfl_xor_sync(0xffffffffu, v, m);
}

template <class E, int D>
__device__ void write_empty_result(const DecodeParams &p, int b, int g, int part,
                                   int nparts_seq, int tid, int nthreads) {
  // A partition that contributes nothing: zeros in the output when it is the
  // sequence's only partition, otherwise a neutral softmax state.
  const int G = p.group;
  if (nparts_seq <= 1) {
    typename E::T *out = static_cast<typename E::T *>(p.out) + b * p.out_row_stride;
    for (int i = tid; i < G * D; i += nthreads)
      out[(g * G) * D + i] = E::from_float(0.f);
  } else {
    for (int i = tid; i < G * D; i += nthreads) {
      const int h = g * G + i / D, d = i % D;
      const int64_t row = (static_cast<int64_t>(b) * p.hq + h) * p.num_partitions + part;
      p.ws_o[row * D + d] = 0.f;
      if (d == 0) {
        p.ws_ml[row * 2 + 0] = -INFINITY;
        p.ws_ml[row * 2 + 1] = 0.f;
      }
    }
  }
}

template <class E, int D, int BOXR>
__global__ void __launch_bounds__(kThreads, 2)
    decode_partition_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv) {
  using S = DecodeSmem<D>;
  constexpr int NH = S::kHalves;
  constexpr int KSTEPS = D / 16;
  constexpr int BOXES = kDecodeChunk / BOXR;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::kBarOffset);
  uint64_t *empty = full + kStages;
  volatile int *s_flag = reinterpret_cast<volatile int *>(smem + S::kFlagOffset);
  int *s_blk = reinterpret_cast<int *>(smem + S::kBlkOffset);

  const int part = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = p.partition_size;
  const int L = checked_context_len(__ldg(p.context_lens + b), p.capacity, p.max_ctx, p.err,
                                    tid == 0 && part == 0 && g == 0);
  const int start = part * P;
  const int nparts_seq = (L + P - 1) / P;
  if (L == 0) {
    if (part == 0) write_empty_result<E, D>(p, b, g, part, 1, tid, kThreads);
    return;
  }
  if (start >= L) return;
  const int end = min(start + P, L);
  const int bs = p.block_size;
  const int first_lblk = start / bs;
  const int nblk = (end - 1) / bs - first_lblk + 1;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), kDecodeWarps);
    }
    s_flag[0] = 0;  // a bad block id in this partition
    s_flag[1] = 0;  // a wait gave up
    fence_barrier_init();
  }
  if (warp == kDecodeWarps) {
    if (lane == 0) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
    }
    const int32_t *bt = p.block_table + static_cast<int64_t>(b) * p.bt_stride + first_lblk;
    for (int i = lane; i < nblk; i += 32) {
      const int id = __ldg(bt + i);
      if (id < 0 || id >= p.num_blocks) {
        raise_error(p.err, PA_DEVERR_BLOCK_ID);
        s_flag[0] = 1;
      }
      s_blk[i] = id;
    }
  }
  __syncthreads();
  if (s_flag[0]) {
    write_empty_result<E, D>(p, b, g, part, nparts_seq, tid, kThreads);
    return;
  }

  const int ntok = end - start;
  const int nchunks = (ntok + kDecodeChunk - 1) / kDecodeChunk;

  // ------------------------------------------------------------ producer --
  if (warp == kDecodeWarps) {
    if (lane != 0) return;
    int issued = 0;
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % kStages;
      if (c >= kStages && !mbar_wait_bounded(smem_u32(empty + s), ((c / kStages) - 1) & 1)) {
        raise_error(p.err, PA_DEVERR_TIMEOUT);
        s_flag[1] = 1;
        break;
      }
      if (s_flag[1]) break;
      const int c0 = start + c * kDecodeChunk;
      int nbox = 0;
#pragma unroll
      for (int k = 0; k < BOXES; ++k) nbox += (c0 + k * BOXR < end) ? 1 : 0;
      const uint32_t bar = smem_u32(full + s);
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nbox * BOXR * 128 * NH * 2));
      const uint32_t kdst = smem_u32(smem + s * S::kStageBytes);
      const uint32_t vdst = kdst + NH * kHalfBytes;
      for (int k = 0; k < nbox; ++k) {
        const int j = c0 + k * BOXR;
        const int row = s_blk[j / bs - first_lblk] * bs + (j % bs);
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          tma_load_3d(kdst + h * kHalfBytes + k * BOXR * 128, &tmk, bar, h * 64, g, row);
          tma_load_3d(vdst + h * kHalfBytes + k * BOXR * 128, &tmv, bar, h * 64, g, row);
        }
      }
      ++issued;
    }
    // Do not leave while copies this CTA issued may still land.
    for (int c = issued - 1; c >= 0 && c >= issued - kStages; --c)
      mbar_wait_bounded(smem_u32(full + (c % kStages)), (c / kStages) & 1);
    return;
  }

  // ----------------------------------------------------------- consumers --
  const int G = p.group;
  const int qh = lane >> 2;  // head column this lane feeds to Q^T
  uint32_t qf[KSTEPS][2];
  {
    const typename E::T *qrow = static_cast<const typename E::T *>(p.q) +
                                b * p.q_row_stride + (g * G + qh) * D + 2 * (lane & 3);
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      qf[ks][0] = qh < G ? __ldg(reinterpret_cast<const uint32_t *>(qrow + ks * 16)) : 0u;
      qf[ks][1] = qh < G ? __ldg(reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8)) : 0u;
    }
  }
  float o[KSTEPS][4];
#pragma unroll
  for (int mt = 0; mt < KSTEPS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2(lane&3), +1
  const float sl = p.scale_log2;
  const int r0 = warp * 16;  // this warp's first row in a chunk
  const int mj = lane >> 3, mr = lane & 7;

  for (int c = 0; c < nchunks; ++c) {
    const int s = c % kStages;
    if (!mbar_wait_bounded(smem_u32(full + s), (c / kStages) & 1)) {
      raise_error(p.err, PA_DEVERR_TIMEOUT);
      s_flag[1] = 1;
      break;
    }
    const int j0 = start + c * kDecodeChunk + r0;
    if (j0 < end) {
      uint8_t *kst = smem + s * S::kStageBytes;
      const uint32_t kb = smem_u32(kst);
      const uint32_t vb = kb + NH * kHalfBytes;
      bool zeroed = false;
      if (j0 + 16 > end) {
        // Rows past the context may hold anything (even NaN); their weight is
        // zero, so make their V rows exact zeros before the P.V product.
        uint8_t *vrows = kst + NH * kHalfBytes;
        for (int i = lane; i < 16 * NH * 8; i += 32) {
          const int rr = i / (NH * 8), h = (i / 8) % NH, cc = i % 8;
          if (j0 + rr >= end)
            *reinterpret_cast<uint4 *>(vrows + h * kHalfBytes + (r0 + rr) * 128 + cc * 16) =
                make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
        zeroed = true;
      }
      // S^T = K Q^T for this warp's 16 tokens.
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        const int row = r0 + (mj & 1) * 8 + mr;
        const int c16 = ks * 2 + (mj >> 1);
        const uint32_t addr =
            kb + (c16 >> 3) * kHalfBytes + row * 128 + (((c16 & 7) ^ (row & 7)) << 4);
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4(addr, a0, a1, a2, a3);
        mma_16816<E::kBF16>(sc, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
      }
      const int t0 = j0 + (lane >> 2), t1 = t0 + 8;
      const float s00 = t0 < end ? sc[0] * sl : -INFINITY;
      const float s01 = t0 < end ? sc[1] * sl : -INFINITY;
      const float s10 = t1 < end ? sc[2] * sl : -INFINITY;
      const float s11 = t1 < end ? sc[3] * sl : -INFINITY;
      float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
      for (int m = 4; m < 32; m <<= 1) {
        mx0 = fmaxf(mx0, shfl_xor(mx0, m));
        mx1 = fmaxf(mx1, shfl_xor(mx1, m));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float cr0 = exp2f(m0 - mn0), cr1 = exp2f(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      // P is rounded to the input type for the tensor core; the row sums use
      // the same rounded values, so the output is an exact weighted mean of
      // V under the rounded weights.
      const uint32_t w0 = E::pack2(exp2f(s00 - mn0), exp2f(s01 - mn1));  // token t0
      const uint32_t w1 = E::pack2(exp2f(s10 - mn0), exp2f(s11 - mn1));  // token t1
      l0 = l0 * cr0 + (E::lo(w0) + E::lo(w1));
      l1 = l1 * cr1 + (E::hi(w0) + E::hi(w1));
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt) {
        o[mt][0] *= cr0;
        o[mt][1] *= cr1;
        o[mt][2] *= cr0;
        o[mt][3] *= cr1;
      }
      // P^T fragments (tokens x heads) from the S^T accumulator layout.
      const uint32_t pb0 = movmatrix_trans(w0);
      const uint32_t pb1 = movmatrix_trans(w1);
      // O^T += V^T P^T, one 16-wide slice of D at a time.
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt) {
        const int row = r0 + (mj >> 1) * 8 + mr;
        const int c16 = mt * 2 + (mj & 1);
        const uint32_t addr =
            vb + (c16 >> 3) * kHalfBytes + row * 128 + (((c16 & 7) ^ (row & 7)) << 4);
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4_trans(addr, a0, a1, a2, a3);
        mma_16816<E::kBF16>(o[mt], a0, a1, a2, a3, pb0, pb1);
      }
      if (zeroed) fence_proxy_async_smem();  // generic writes before the next TMA
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(empty + s));
  }

  // Row sums: combine the lanes that share a head.
#pragma unroll
  for (int m = 4; m < 32; m <<= 1) {
    l0 += shfl_xor(l0, m);
    l1 += shfl_xor(l1, m);
  }

  // Merge the four warps' states through shared memory (stage 0 is free:
  // every chunk has been consumed).
  named_barrier_sync(1, kDecodeWarps * 32);
  float *sO = reinterpret_cast<float *>(smem);           // [warp][8][D]
  float *sM = sO + kDecodeWarps * kDecodeMaxGroup * D;  // [warp][8]
  float *sL = sM + kDecodeWarps * kDecodeMaxGroup;      // [warp][8]
  {
    const int h0 = 2 * (lane & 3), h1 = h0 + 1;
    float *w = sO + warp * kDecodeMaxGroup * D;
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) {
      const int d0 = mt * 16 + (lane >> 2), d1 = d0 + 8;
      w[h0 * D + d0] = o[mt][0];
      w[h1 * D + d0] = o[mt][1];
      w[h0 * D + d1] = o[mt][2];
      w[h1 * D + d1] = o[mt][3];
    }
    if (lane < 4) {
      sM[warp * kDecodeMaxGroup + h0] = m0;
      sM[warp * kDecodeMaxGroup + h1] = m1;
      sL[warp * kDecodeMaxGroup + h0] = l0;
      sL[warp * kDecodeMaxGroup + h1] = l1;
    }
  }
  named_barrier_sync(1, kDecodeWarps * 32);
  for (int i = tid; i < G * D; i += kDecodeWarps * 32) {
    const int h = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, sM[w * kDecodeMaxGroup + h]);
    float acc = 0.f, l = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) {
        const float f = exp2f(sM[w * kDecodeMaxGroup + h] - M);
        acc += f * sO[(w * kDecodeMaxGroup + h) * D + d];
        l += f * sL[w * kDecodeMaxGroup + h];
      }
    }
    if (nparts_seq == 1) {
      typename E::T *out = static_cast<typename E::T *>(p.out) + b * p.out_row_stride;
      out[(g * G + h) * D + d] = E::from_float(l > 0.f ? acc / l : 0.f);
    } else {
      const int64_t row =
          (static_cast<int64_t>(b) * p.hq + g * G + h) * p.num_partitions + part;
      p.ws_o[row * D + d] = acc;
      if (d == 0) {
        p.ws_ml[row * 2 + 0] = M;
        p.ws_ml[row * 2 + 1] = l;
      }
    }
  }
}

// Merges the partitions of each (sequence, query head) by log-sum-exp:
//   M = max_p m_p,  w_p = 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p l_p.
template <class E, int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const DecodeParams p) {
  extern __shared__ float sw[];  // [num_partitions] weights
  __shared__ float red[D / 32];
  const int b = blockIdx.x / p.hq, h = blockIdx.x % p.hq;
  const int tid = threadIdx.x;
  const int L = checked_context_len(__ldg(p.context_lens + b), p.capacity, p.max_ctx, p.err, false);
  const int n = (L + p.partition_size - 1) / p.partition_size;
  if (n <= 1) return;
  const int64_t row0 = (static_cast<int64_t>(b) * p.hq + h) * p.num_partitions;
  const float *ml = p.ws_ml + row0 * 2;

  float mx = -INFINITY;
  for (int i = tid; i < n; i += D) mx = fmaxf(mx, ml[2 * i]);
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
  if ((tid & 31) == 0) red[tid >> 5] = mx;
  __syncthreads();
  float M = red[0];
#pragma unroll
  for (int w = 1; w < D / 32; ++w) M = fmaxf(M, red[w]);
  __syncthreads();

  float ls = 0.f;
  for (int i = tid; i < n; i += D) {
    const float m = ml[2 * i];
    const float w = (M == -INFINITY) ? 0.f : exp2f(m - M);
    sw[i] = w;
    ls += w * ml[2 * i + 1];
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, m);
  if ((tid & 31) == 0) red[tid >> 5] = ls;
  __syncthreads();
  float l = 0.f;
#pragma unroll
  for (int w = 0; w < D / 32; ++w) l += red[w];

  const float *po = p.ws_o + row0 * D + tid;
  float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
  int i = 0;
  for (; i + 4 <= n; i += 4) {
    acc0 += sw[i] * po[(i + 0) * D];
    acc1 += sw[i + 1] * po[(i + 1) * D];
    acc2 += sw[i + 2] * po[(i + 2) * D];
    acc3 += sw[i + 3] * po[(i + 3) * D];
  }
  for (; i < n; ++i) acc0 += sw[i] * po[i * D];
  const float acc = (acc0 + acc1) + (acc2 + acc3);
  typename E::T *out = static_cast<typename E::T *>(p.out) + b * p.out_row_stride + h * D;
  out[tid] = E::from_float(l > 0.f ? acc / l : 0.f);
}

template <class E, int D, int BOXR>
cudaError_t launch_typed(const DecodeArgs &a, const DecodeParams &p, cudaStream_t stream) {
  using S = DecodeSmem<D>;
  const int max_blocks = a.partition_size / a.block_size + 2;
  const int smem = S::bytes(max_blocks);
  auto kernel = decode_partition_kernel<E, D, BOXR>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_partitions, a.num_kv_heads, a.num_seqs);
  kernel<<<grid, kThreads, smem, stream>>>(p, a.tm_k, a.tm_v);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.num_partitions <= 1) return e;
  decode_combine_kernel<E, D><<<a.num_seqs * a.num_q_heads, D,
                                a.num_partitions * sizeof(float), stream>>>(p);
  return cudaGetLastError();
}

template <class E, int D>
cudaError_t launch_box(const DecodeArgs &a, const DecodeParams &p, cudaStream_t stream) {
  switch (a.box_rows) {
    case 8: return launch_typed<E, D, 8>(a, p, stream);
    case 16: return launch_typed<E, D, 16>(a, p, stream);
    case 32: return launch_typed<E, D, 32>(a, p, stream);
    case 64: return launch_typed<E, D, 64>(a, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream) {
  DecodeParams p;
  p.out = a.out;
  p.out_row_stride = a.out_row_stride;
  p.q = a.query;
  p.q_row_stride = a.q_row_stride;
  p.block_table = a.block_table;
  p.bt_stride = a.block_table_stride;
  p.context_lens = a.context_lens;
  p.capacity = a.capacity;
  p.max_ctx = a.max_context_len;
  p.hq = a.num_q_heads;
  p.hkv = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.scale_log2 = a.scale_log2;
  p.partition_size = a.partition_size;
  p.num_partitions = a.num_partitions;
  p.ws_o = a.ws_o;
  p.ws_ml = a.ws_ml;
  p.err = a.d_error;
  const bool bf = a.dtype == PA_BF16;
  if (a.head_dim == 128)
    return bf ? launch_box<BF16, 128>(a, p, stream) : launch_box<F16, 128>(a, p, stream);
  if (a.head_dim == 64)
    return bf ? launch_box<BF16, 64>(a, p, stream) : launch_box<F16, 64>(a, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
