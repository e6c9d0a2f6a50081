// prefill.cu -- causal attention for cu_seqlens-packed queries against the
// paged KV cache, on the sm_103a tensor cores (tcgen05 + TMEM, fed by TMA).
//
// Operation (lqnn.cn article §3.1 cu_seqlens and §4.4 packed attention;
// cannbot-skills "model-infer-kvcache" skill page App. C sparse_mode 3 and
// App. E): sequence b owns query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1
// and the first L_b keys of its paged cache; with q_b queries, row i sees
// keys j <= L_b - q_b + i (the last query sees every key), never another
// sequence's keys.
//
// Design (the pages build a per-sequence mask from cu_seqlens on Ascend;
// here nothing is masked outside the diagonal tile and nothing padded):
//  * CTA = (128-row query tile of one sequence, query head).  Tiles are
//    dealt heaviest-first (by tile index, i.e. by how many KV tiles the
//    causal row range needs) so long tails start early.
//  * Warp 4 (TMA): loads the Q tile once and streams 128-token K/V tiles
//    into a 2-stage ring; each K/V tile is gathered block by block through
//    block_table (one TMA box per block), with the 128-byte swizzle the MMA
//    descriptors expect.
//  * Warp 5 (MMA, one thread): S = Q K^T into a double-buffered TMEM tile
//    (M=128, N=128, K=16 x 8 instructions), then O += P V with V read
//    MN-major straight from its TMA tile.  S(kt+1) is issued before P(kt) is
//    ready, so the tensor core works while the softmax runs.
//  * Warps 0-3 (softmax, one thread per query row = TMEM lane): read S from
//    TMEM, mask only tiles that cross the causal edge or the context end,
//    exponentiate in base 2, and write P (bf16/fp16) to shared memory in the
//    swizzled K-major layout.  The running max is only raised -- and O in
//    TMEM rescaled -- when a row's max grows by more than 2^8, which keeps
//    every P <= 256 and the result exact up to rounding.
//  * Epilogue: O / l from TMEM to registers to global memory.
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {

namespace {

constexpr int kThreads = 192;             // warps 0-3 softmax, 4 TMA, 5 MMA
constexpr int kHalf = 128 * 128;          // 128 rows x 64 elements x 2 B
constexpr int kTile = 2 * kHalf;          // 128 x 128 tile, two 64-wide halves
constexpr int kQOff = 0;
constexpr int kKVOff = kTile;             // stage s: K at +s*2*kTile, V +kTile
constexpr int kPOff = kKVOff + 4 * kTile;
constexpr int kBarOff = kPOff + kTile;
enum { kQFull = 0, kKVFull = 1, kKVEmpty = 3, kSFull = 5, kSFree = 7, kPFull = 9, kPVDone = 10,
       kFin = 11, kNumBars = 12 };
constexpr int kMiscOff = kBarOff + kNumBars * 8;
constexpr int kSmemBytes = 1024 + kMiscOff + 64;
constexpr uint32_t kTmemCols = 512;       // S0 | S1 | O | unused
constexpr float kRescaleThreshold = 8.0f;  // log2 of the largest P allowed

struct PrefillParams {
  void *out;
  int64_t out_row_stride;
  const int32_t *block_table;
  int64_t bt_stride;
  const int32_t *cu;
  const int32_t *ctx;
  int32_t capacity, max_ctx;
  int32_t num_seqs, total_q, max_seqlen_q;
  int32_t hq, group, block_size;
  int64_t num_blocks;
  float scale_log2;
  int32_t causal;
  int32_t *err;
};

// Which (sequence, query tile) this CTA serves: slot x of the list ordered by
// tile index descending, sequences in order within one tile index.
__device__ void find_tile(const PrefillParams &p, int x, int lane, int *seq_out, int *tile_out) {
  const int max_tiles = (p.max_seqlen_q + 127) / 128;
  int rem = x;
  for (int i = max_tiles - 1; i >= 0; --i) {
    for (int c0 = 0; c0 < p.num_seqs; c0 += 32) {
      const int s = c0 + lane;
      bool has = false;
      if (s < p.num_seqs) {
        const int q = __ldg(p.cu + s + 1) - __ldg(p.cu + s);
        has = q >= 0 && q <= p.max_seqlen_q && (q + 127) / 128 > i;
      }
      unsigned bal = __ballot_sync(0xffffffffu, has);
      const int n = __popc(bal);
      if (rem < n) {
        for (int k = 0; k < rem; ++k) bal &= bal - 1;
        *seq_out = c0 + __ffs(bal) - 1;
        *tile_out = i;
        return;
      }
      rem -= n;
    }
  }
  *seq_out = -1;
  *tile_out = -1;
}

// cu_seqlens must start at 0, never decrease, end at total_q, and no
// sequence may exceed max_seqlen_q (which sized the grid).
__device__ void check_cu_seqlens(const PrefillParams &p, int lane) {
  bool bad = false;
  if (lane == 0) bad = __ldg(p.cu) != 0 || __ldg(p.cu + p.num_seqs) != p.total_q;
  for (int s = lane; s < p.num_seqs; s += 32) {
    const int q = __ldg(p.cu + s + 1) - __ldg(p.cu + s);
    bad |= q < 0 || q > p.max_seqlen_q;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) raise_error(p.err, PA_DEVERR_CU_SEQLENS);
}

template <class E>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmq,
                   const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kBarOff);
  volatile int *misc = reinterpret_cast<volatile int *>(smem + kMiscOff);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y;

  if (warp == 0) {
    int seq, tile;
    find_tile(p, blockIdx.x, lane, &seq, &tile);
    if (lane == 0) {
      misc[0] = seq;
      misc[1] = tile;
      misc[3] = 0;  // abort: some wait gave up
    }
    if (blockIdx.x == 0 && h == 0) check_cu_seqlens(p, lane);
  }
  if (warp == 1 && lane == 0) {
    // S-free and P-full collect one arrival per softmax warp.
    for (int i = 0; i < kNumBars; ++i)
      mbar_init(bar(i), (i == kSFree || i == kSFree + 1 || i == kPFull) ? 4 : 1);
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(const_cast<int *>(misc + 2)), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int seq = misc[0], tile = misc[1];
  const uint32_t tbase = static_cast<uint32_t>(misc[2]);

  int nkv = 0, q_start = 0, rows_valid = 0, L = 0, lim_base = 0, row0 = 0;
  if (seq >= 0) {
    q_start = __ldg(p.cu + seq);
    const int q_len = __ldg(p.cu + seq + 1) - q_start;
    L = checked_context_len(__ldg(p.ctx + seq), p.capacity, p.max_ctx, p.err,
                            tid == 0 && h == 0 && tile == 0);
    row0 = tile * 128;
    rows_valid = min(128, q_len - row0);
    lim_base = p.causal ? L - q_len : 0x3fffffff;  // row i sees keys <= lim_base + i
    int kv_end = L;
    if (p.causal) kv_end = min(L, L - q_len + row0 + 128);
    if (kv_end < 0) kv_end = 0;
    nkv = (kv_end + 127) / 128;
  }
  const int g = h / p.group;

  if (warp == 4) {
    // ----------------------------------------------------------- TMA --
    if (lane == 0 && nkv > 0) {
      tma_prefetch_desc(&tmq);
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
      const uint32_t qs = smem_u32(smem + kQOff);
      mbar_arrive_expect_tx(bar(kQFull), kTile);
      tma_load_3d(qs, &tmq, bar(kQFull), 0, h, q_start + row0);
      tma_load_3d(qs + kHalf, &tmq, bar(kQFull), 64, h, q_start + row0);
      const int bs = p.block_size;  // one TMA box per block (16..128 rows)
      const int boxr = bs;
      const int nbox = 128 / boxr;
      const int32_t *bt = p.block_table + static_cast<int64_t>(seq) * p.bt_stride;
      int issued = 0;
      for (int kt = 0; kt < nkv; ++kt) {
        const int st = kt & 1;
        if (kt >= 2 && !mbar_wait_bounded(bar(kKVEmpty + st), ((kt >> 1) - 1) & 1)) {
          raise_error(p.err, PA_DEVERR_TIMEOUT);
          misc[3] = 1;
          break;
        }
        if (misc[3]) break;
        const int j0 = kt * 128;
        int rows[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) rows[k] = -1;
        int n = 0;
        for (int k = 0; k < nbox; ++k) {
          const int j = j0 + k * boxr;
          if (j >= L) break;
          const int id = __ldg(bt + j / bs);
          if (id < 0 || id >= p.num_blocks) {
            raise_error(p.err, PA_DEVERR_BLOCK_ID);
            continue;
          }
          rows[k] = id * bs + (j % bs);
          ++n;
        }
        const uint32_t kd = smem_u32(smem + kKVOff + st * 2 * kTile);
        const uint32_t vd = kd + kTile;
        mbar_arrive_expect_tx(bar(kKVFull + st), static_cast<uint32_t>(n * boxr * 128 * 4));
        for (int k = 0; k < nbox; ++k) {
          if (rows[k] < 0) continue;
          const uint32_t off = k * boxr * 128;
          tma_load_3d(kd + off, &tmk, bar(kKVFull + st), 0, g, rows[k]);
          tma_load_3d(kd + kHalf + off, &tmk, bar(kKVFull + st), 64, g, rows[k]);
          tma_load_3d(vd + off, &tmv, bar(kKVFull + st), 0, g, rows[k]);
          tma_load_3d(vd + kHalf + off, &tmv, bar(kKVFull + st), 64, g, rows[k]);
        }
        ++issued;
      }
      // Do not leave while copies this CTA issued may still land.
      mbar_wait_bounded(bar(kQFull), 0);
      for (int kt = issued - 1; kt >= 0 && kt >= issued - 2; --kt)
        mbar_wait_bounded(bar(kKVFull + (kt & 1)), (kt >> 1) & 1);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ----------------------------------------------------------- MMA --
    if (lane == 0 && nkv > 0) {
      constexpr bool kBF = E::kBF16;
      const uint32_t id_qk = idesc_f16(kBF, 128, 128, false);
      const uint32_t id_pv = idesc_f16(kBF, 128, 128, true);
      const uint32_t qs = smem_u32(smem + kQOff);
      const uint32_t ps = smem_u32(smem + kPOff);
      const uint32_t t_o = tbase + 256;
      bool ok = mbar_wait_bounded(bar(kQFull), 0);
      auto issue_pv = [&](int kt) {
        const uint32_t vs = smem_u32(smem + kKVOff + (kt & 1) * 2 * kTile + kTile);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          umma_f16_ss(t_o, sdesc_sw128(ps + (k >> 2) * kHalf + (k & 3) * 32, 16, 1024),
                      sdesc_sw128(vs + k * 2048, kHalf, 1024), id_pv, (kt > 0 || k > 0) ? 1u : 0u);
        umma_commit(bar(kPVDone));
        umma_commit(bar(kKVEmpty + (kt & 1)));
      };
      for (int kt = 0; ok && kt < nkv; ++kt) {
        const int st = kt & 1;
        ok = mbar_wait_bounded(bar(kKVFull + st), (kt >> 1) & 1);
        if (ok && kt >= 2) ok = mbar_wait_bounded(bar(kSFree + st), ((kt >> 1) - 1) & 1);
        if (!ok) break;
        tc_fence_after();
        const uint32_t ks = smem_u32(smem + kKVOff + st * 2 * kTile);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          umma_f16_ss(tbase + st * 128,
                      sdesc_sw128(qs + (k >> 2) * kHalf + (k & 3) * 32, 16, 1024),
                      sdesc_sw128(ks + (k >> 2) * kHalf + (k & 3) * 32, 16, 1024), id_qk,
                      k > 0 ? 1u : 0u);
        umma_commit(bar(kSFull + st));
        if (kt >= 1) {
          ok = mbar_wait_bounded(bar(kPFull), (kt - 1) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_pv(kt - 1);
        }
      }
      if (ok) {
        ok = mbar_wait_bounded(bar(kPFull), (nkv - 1) & 1);
        if (ok) {
          tc_fence_after();
          issue_pv(nkv - 1);
        }
      }
      if (!ok) {
        raise_error(p.err, PA_DEVERR_TIMEOUT);
        misc[3] = 1;
      }
      // Every MMA issued above has completed once this barrier fires.
      umma_commit(bar(kFin));
      mbar_wait_bounded(bar(kFin), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- softmax --
    const int r = tid;  // query row in the tile == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const int lim = min(lim_base + row0 + r, L - 1);  // last visible key
    const float sl = p.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    uint8_t *prow = smem + kPOff + r * 128;
    for (int kt = 0; kt < nkv; ++kt) {
      const int sb = kt & 1;
      ok = mbar_wait_bounded(bar(kSFull + sb), (kt >> 1) & 1);
      if (!ok) break;
      tc_fence_after();
      float s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_addr + sb * 128 + c * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(v[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kSFree + sb));

      const int bound = lim - kt * 128;  // columns 0..bound are visible
      if (bound < 127) {
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = c <= bound ? s[c] : -INFINITY;
      }
      // Row max of the raw scores (scale > 0 keeps the order), as a tree.
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
      for (int c = 8; c < 128; ++c) mx[c & 7] = fmaxf(mx[c & 7], s[c]);
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl;
      const bool raise_max = mt > m_ref + kRescaleThreshold;
      const float m_new = raise_max ? mt : m_ref;
      const float corr = raise_max ? fast_exp2(m_ref - m_new) : 1.f;
      const float mu = m_new == -INFINITY ? 0.f : m_new;
      // p = 2^(s * scale*log2(e) - max).  P is rounded to the input type for
      // the tensor core; the row sum uses the same rounded values, so O / l is
      // an exact weighted mean of V under the rounded weights.
      uint32_t pw[64];
      float rsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        pw[c] = E::pack2(fast_exp2(fmaf(s[2 * c], sl, -mu)),
                         fast_exp2(fmaf(s[2 * c + 1], sl, -mu)));
        rsum[c & 3] += E::sum2(pw[c]);
      }
      const float rs = (rsum[0] + rsum[1]) + (rsum[2] + rsum[3]);
      if (kt >= 1) {
        // P(kt-1) has been consumed and O holds the sum through kt-1.
        ok = mbar_wait_bounded(bar(kPVDone), (kt - 1) & 1);
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, raise_max)) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            const uint32_t ta = tbase + lane_addr + 256 + c * 32;
            tmem_ld32(ta, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * corr);
            tmem_st32(ta, v);
          }
          tmem_wait_st();
        }
      }
      l = l * corr + rs;
      m_ref = m_new;

      if (kt == nkv - 1 && L < (kt + 1) * 128) {
        // Rows past the context end may hold anything (even NaN); their
        // weight is zero, so make their V rows exact zeros for the MMA.
        ok = mbar_wait_bounded(bar(kKVFull + (kt & 1)), (kt >> 1) & 1);
        if (!ok) break;
        uint8_t *vt = smem + kKVOff + (kt & 1) * 2 * kTile + kTile;
        const int first = L - kt * 128;
        for (int i = tid; i < (128 - first) * 16; i += 128) {
          const int row = first + i / 16, c16 = i % 16;
          *reinterpret_cast<uint4 *>(vt + (c16 >> 3) * kHalf + row * 128 + (c16 & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
      }
      // P row -> shared memory, K-major with the 128-byte swizzle.
#pragma unroll
      for (int c8 = 0; c8 < 16; ++c8) {
        const uint4 w = make_uint4(pw[c8 * 4 + 0], pw[c8 * 4 + 1], pw[c8 * 4 + 2], pw[c8 * 4 + 3]);
        *reinterpret_cast<uint4 *>(prow + (c8 >> 3) * kHalf + (((c8 & 7) ^ (r & 7)) << 4)) = w;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kPFull));
    }
    if (!ok) {
      raise_error(p.err, PA_DEVERR_TIMEOUT);
      misc[3] = 1;
    }
    // ------------------------------------------------------ epilogue --
    if (seq >= 0) {
      const bool have_o = ok && nkv > 0 && mbar_wait_bounded(bar(kPVDone), (nkv - 1) & 1);
      if (nkv > 0) tc_fence_after();
      const float inv_l = (have_o && l > 0.f) ? 1.f / l : 0.f;
      const int64_t grow = static_cast<int64_t>(q_start) + row0 + r;
      const bool store = r < rows_valid && grow >= 0 && grow < p.total_q;
      typename E::T *orow = static_cast<typename E::T *>(p.out) + grow * p.out_row_stride + h * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        if (have_o) {
          tmem_ld32(tbase + lane_addr + 256 + c * 32, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (store) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            const float *f = reinterpret_cast<const float *>(v) + q4 * 8;
            w.x = E::pack2(f[0] * inv_l, f[1] * inv_l);
            w.y = E::pack2(f[2] * inv_l, f[3] * inv_l);
            w.z = E::pack2(f[4] * inv_l, f[5] * inv_l);
            w.w = E::pack2(f[6] * inv_l, f[7] * inv_l);
            *reinterpret_cast<uint4 *>(orow + c * 32 + q4 * 8) = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream) {
  PrefillParams p;
  p.out = a.out;
  p.out_row_stride = a.out_row_stride;
  p.block_table = a.block_table;
  p.bt_stride = a.block_table_stride;
  p.cu = a.cu_seqlens_q;
  p.ctx = a.context_lens;
  p.capacity = a.capacity;
  p.max_ctx = a.max_context_len;
  p.num_seqs = a.num_seqs;
  p.total_q = a.total_q;
  p.max_seqlen_q = a.max_seqlen_q;
  p.hq = a.num_q_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.scale_log2 = a.scale_log2;
  p.causal = a.causal;
  p.err = a.d_error;
  // Query tiles: sum_b ceil(q_b / 128) is at most both bounds below.
  const int64_t max_tiles = (static_cast<int64_t>(a.max_seqlen_q) + 127) / 128;
  int64_t slots = (static_cast<int64_t>(a.total_q) + 127LL * a.num_seqs) / 128;
  if (slots > a.num_seqs * max_tiles) slots = a.num_seqs * max_tiles;
  if (slots <= 0) return cudaSuccess;
  if (slots > 0x7fffffff) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(slots), a.num_q_heads);
  cudaError_t e;
  if (a.dtype == PA_BF16) {
    e = allow_dynamic_smem<prefill_kernel<BF16>>();
    if (e != cudaSuccess) return e;
    prefill_kernel<BF16><<<grid, kThreads, kSmemBytes, stream>>>(p, a.tm_q, a.tm_k, a.tm_v);
  } else {
    e = allow_dynamic_smem<prefill_kernel<F16>>();
    if (e != cudaSuccess) return e;
    prefill_kernel<F16><<<grid, kThreads, kSmemBytes, stream>>>(p, a.tm_q, a.tm_k, a.tm_v);
  }
  return cudaGetLastError();
}

}  // namespace pa
