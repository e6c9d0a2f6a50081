// decode_kernel.cuh -- paged attention for one query token per sequence
// (kernel templates; the instantiations live in decode_*.cu, one translation
// unit per element type and pool format, so they compile in parallel).
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
//  * Work.  A unit is one (sequence, KV-head slice): a slice is the query
//    heads of one KV head, up to 16 of them, and every piece of work serves
//    all of a slice's heads from the same K/V bytes (GQA sharing).  A KV head
//    with more than 16 query heads is cut into slices of 16 that sit next
//    to each other in the schedule.  Two schedules cut the units into
//    pieces (split-KV):
//      - fixed partitions (a partition size is given): a unit's context is
//        cut into partitions of P tokens, the pages' scheme; worker w of W
//        takes items w, w+W, ... of the (sequence, slice, partition) list;
//      - balanced (automatic): the units' contexts, each rounded up to 16
//        tokens, are laid end to end and cut into equal chunks, one (or a
//        few) per worker, so every worker streams the same number of tokens
//        whatever the mix of lengths.  A chunk can hold the tail of one unit
//        and the head of the next.
//    A piece that is its unit's whole context writes the output directly;
//    otherwise it writes its softmax state (max, sum, unnormalised output)
//    to workspace and a merge kernel combines the pieces by log-sum-exp.
//  * Persistent CTAs, independent warps.  The grid is at most two CTAs per
//    SM.  Each of a CTA's four consumer warps is a worker with its own static
//    list of pieces, so no warp ever waits for another.  The lists come from
//    per-sequence prefix sums computed once per CTA from context_lens.
//  * One producer warp feeds all four workers through a 3-stage ring of
//    TMA tile loads (swizzled) guarded by mbarriers: each stage holds 16
//    tokens (32 for one-byte pools) of K and V for every worker, read block
//    by block through the block table.  Producer lane w walks worker w's
//    pieces with incremental (block, offset) counters, and the block ids of
//    the worker's next piece are copied into shared memory with cp.async
//    while its current piece streams, so no id lookup or division sits on
//    the load-issue path.
//  * Scores are computed transposed on the tensor cores -- S^T[16 tokens x 8
//    heads] = K[16 x D] Q^T[D x 8] with mma.sync m16n8k16, fp32 accumulate --
//    so the slice's heads fill the N side, 8 per column group (NG = 1 or 2
//    groups share every K fragment).  The online softmax runs on the
//    fragments (warp-shuffle max over tokens), P^T is formed with movmatrix,
//    and O^T[D x 8] += V^T[D x 16] P^T[16 x 8] reads V through ldmatrix.trans
//    (16-bit pools) or widens one-byte codes into fragments in registers.
//  * The one-call decode step: the same launch also writes the step's new
//    K/V rows into the pool (workers copy them before their first stage
//    lands), and the worker holding a sequence's newest row takes it from
//    the token that slot_mapping sends there, straight from the step's
//    input, so no read waits for the write.
//  * Exponentials are base 2 with the scale pre-multiplied by log2(e).
#pragma once

#include <math.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace dec {

constexpr int kWorkers = kDecodeWarps;
constexpr int kThreads = (kWorkers + 1) * 32;  // + producer warp
// The one-call step adds a writer warp; at most three warps per SM
// sub-partition either way (two CTAs per SM), so the register budget is the
// same.
constexpr int threads_for(bool wr) { return (kWorkers + (wr ? 2 : 1)) * 32; }
constexpr int kWriterWarp = kWorkers + 1;
constexpr uint32_t kTerminate = 0x100u;        // stage header: no more data

// A stage holds, per K and V, `kRegions` regions of kWorkers x kRows rows:
// 16-bit pools in 64-element halves (rows of 128 bytes, 128-byte swizzle),
// 16 rows per worker; one-byte pools in one region of whole rows (D bytes:
// 128-byte swizzle at D 128, 64-byte swizzle at D 64), 32 rows per worker.
template <int D, bool KV8 = false>
struct DecodeSmem {
  static constexpr int kStages = 3;
  static constexpr int kRows = KV8 ? 2 * kDecodeSub : kDecodeSub;  // per worker
  static constexpr int kRowBytes = KV8 ? D : 128;
  static constexpr int kRegionBytes = kWorkers * kRows * kRowBytes;
  static constexpr int kHalves = D / 64;
  static constexpr int kRegions = KV8 ? 1 : kHalves;
  static constexpr int kStageBytes = 2 * kRegions * kRegionBytes;  // K + V
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kHdrOffset = kBarOffset + 2 * kStages * 8;
  static constexpr int kAbortOffset = kHdrOffset + 32;  // after kStages (<= 8) headers
  // per worker (one-call step, 16-bit pools): the step's input K and V rows
  // of its piece's newest token, then that row's block id and token b's slot
  static constexpr int kNewOffset = kAbortOffset + 128;
  static constexpr int kNewMeta = KV8 ? 0 : 2 * D * 2;
  static constexpr int kNewBytes = KV8 ? 0 : kNewMeta + 16;
  static constexpr int kVarOffset = kNewOffset + kWorkers * kNewBytes;  // pref[S+1], len[S], ids
  static int bytes(int num_seqs, int max_ids) {
    return 1024 + kVarOffset + 4 * (2 * num_seqs + 1) + 4 * kWorkers * 2 * max_ids;
  }
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
  int32_t num_seqs, hq, hkv, group, block_size;
  int32_t nc, hs, vh;  // slices per KV head, heads per slice (rows per piece), units per sequence
  int32_t box_rows;    // TMA box height (block_size, at most 16)
  int64_t num_blocks;
  float scale_log2;
  int32_t partition_size, num_partitions, max_ids;
  int32_t balanced, chunk_cap, num_workers;  // balanced schedule (see above)
  float *ws_o, *ws_ml;
  int32_t *ws_pref;  // balanced: the prefix sums, for the merge kernel
  const float *k_scale, *v_scale;  // one-byte pools: per-KV-head dequantisation scales
  // The one-call step: nw new tokens (new_k / new_v [nw, Hkv, D] rows at
  // new_stride elements) are written to pool rows slot_mapping[t] (of
  // num_slots) in the same launch; a sequence's newest row is taken from
  // the token written to it.  nw = 0: a plain decode.
  int32_t nw;
  // Launched right after this step's cache write as its own kernel (the
  // two-launch step): only K/V pool rows can be that kernel's output, so
  // everything else is read at once and only the first K/V load waits.
  int32_t after_write;
  const void *new_k, *new_v;
  int64_t new_stride;
  const int64_t *slot_mapping;
  void *k_pool, *v_pool;
  int64_t num_slots;
  int32_t *err;
  uint64_t wait_ns;  // bound of a pipeline wait
};

// One piece of work: tokens [start, end) of unit (sequence b, slice g) whose
// context is L tokens.  `direct`: the piece is the unit's whole context and
// writes the output; else its softmax state goes to workspace rows
// prow + h * pstride for the slice's query heads h = 0..hs-1.
struct Item {
  int b, g, part, L, start, end;
  bool direct;
  int64_t prow;
  int pstride;
};

__host__ __device__ __forceinline__ int ceil16(int x) { return (x + 15) & ~15; }

// Balanced schedule: chunk size (in 16-rounded token-units) for T token-units
// over NW workers, each taking at most `cap` tokens per chunk (and then
// several chunks).  The decode and merge kernels must agree on it.
__host__ __device__ __forceinline__ int balanced_chunk(int T, int NW, int cap) {
  // 32-bit unsigned arithmetic is exact while T < 2^31 and NW * cap < 2^31
  // (no sum below exceeds 2^32).
  const uint32_t t = T > 0 ? static_cast<uint32_t>(T) : 0u;
  const uint32_t per = static_cast<uint32_t>(NW) * static_cast<uint32_t>(cap);
  const uint32_t k = t > 0 ? (t + per - 1) / per : 1u;
  const uint32_t kn = k * static_cast<uint32_t>(NW);
  const int c = ceil16(static_cast<int>((t + kn - 1) / kn));
  return c > 0 ? c : 16;
}

// What every role of a CTA needs to walk the schedule.
struct Sched {
  const int *pref;  // fixed: items before sequence b; balanced: token-units before b
  const int *len;   // checked context lengths
  int S, vh, hq, G, nc, hs, P, NP, NW;
  bool balanced;
  int total;      // fixed: items; balanced: token-units
  int C, chunks;  // balanced: chunk size and count
};

// First query head of slice g (unit numbering within a sequence) and the
// number of heads in it.
__device__ __forceinline__ int slice_head0(const Sched &sc, int g, int &nh) {
  const int kvh = sc.nc == 1 ? g : g / sc.nc;
  const int sl = g - kvh * sc.nc;
  nh = min(sc.hs, sc.G - sl * sc.hs);
  return kvh * sc.G + sl * sc.hs;
}

// Item i of the numbering given by the prefix sums `pref` (items of sequence
// b are pref[b] .. pref[b+1]-1, ordered by slice then partition).
__device__ __forceinline__ Item decode_item(int i, const Sched &sc) {
  int lo = 0, hi = sc.S;  // pref[lo] <= i < pref[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sc.pref[mid] <= i) lo = mid;
    else hi = mid;
  }
  Item m;
  m.b = lo;
  m.L = sc.len[lo];
  const int np = m.L > 0 ? (m.L + sc.P - 1) / sc.P : 1;
  const int rem = i - sc.pref[lo];
  m.g = rem / np;  // numbered by slice, then partition
  m.part = rem - m.g * np;
  m.start = m.part * sc.P;
  m.end = min(m.start + sc.P, m.L);
  if (m.end < m.start) m.end = m.start;
  return m;
}

// A worker's place in its piece list (fixed: next item index; balanced:
// current chunk and position in it).
struct Cursor {
  int i, x;
};
__device__ __forceinline__ Cursor first_cursor(const Sched &sc, int gw) {
  Cursor c;
  c.i = gw;
  c.x = sc.balanced ? gw * sc.C : 0;
  return c;
}

// The next piece of a worker's list; false at the end.  The fixed schedule
// also returns the (empty) items of empty sequences, end == start.
__device__ inline bool next_piece(const Sched &sc, Cursor &cu, Item &m) {
  if (!sc.balanced) {
    if (cu.i >= sc.total) return false;
    m = decode_item(cu.i, sc);
    cu.i += sc.NW;
    m.direct = (m.L > 0 ? (m.L + sc.P - 1) / sc.P : 1) == 1;
    int nh;
    const int h0 = slice_head0(sc, m.g, nh);
    m.prow = (static_cast<int64_t>(m.b) * sc.hq + h0) * sc.NP + m.part;
    m.pstride = sc.NP;
    return true;
  }
  while (cu.i < sc.chunks) {
    const int cend = min((cu.i + 1) * sc.C, sc.total);
    if (cu.x >= cend) {  // chunk done: this worker's next one
      cu.i += sc.NW;
      cu.x = cu.i * sc.C;
      continue;
    }
    // the unit (sequence b, slice g) holding position x: pref[b] <= x < pref[b+1]
    int lo = 0, hi = sc.S;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sc.pref[mid] <= cu.x) lo = mid;
      else hi = mid;
    }
    const int L = sc.len[lo];
    const int W = ceil16(L);
    const int rel = cu.x - sc.pref[lo];
    const int g = rel / W;
    const int t0 = rel - g * W;
    const int t1 = min(W, t0 + (cend - cu.x));
    cu.x += t1 - t0;
    if (t0 >= L) continue;  // only the rounding past the context end
    m.b = lo;
    m.g = g;
    m.L = L;
    m.part = cu.i;
    m.start = t0;
    m.end = min(t1, L);
    m.direct = t0 == 0 && t1 >= L;
    m.prow = (static_cast<int64_t>(lo) * sc.vh + g + cu.i) * sc.hs;
    m.pstride = 1;
    return true;
  }
  return false;
}

__device__ __forceinline__ float shfl_xor(float v, int m) {
  return __shfl_xor_sync(0xffffffffu, v, m);
}

// The query as the B operand of S^T = K Q^T, column group n of the slice
// (heads h0 + 8n + lane / 4): lane (head column, t = lane % 4) feeds k-step
// ks.  16-bit pools: elements 16ks + 2t, +1 and 16ks + 2t + 8, +9 (the
// ldmatrix order of K).  One-byte pools: elements (D/4)t + 4ks .. +3, the
// order in which the K fragments are widened -- a dot product over D takes
// any order both operands share.
template <class E, int D, bool KV8, int NG>
__device__ __forceinline__ void load_q(uint32_t (&qf)[NG][D / 16][2], const DecodeParams &p,
                                       int b, int h0, int nh, int lane) {
#pragma unroll
  for (int n = 0; n < NG; ++n) {
    const int qh = 8 * n + (lane >> 2);  // head column this lane feeds to Q^T
    const bool ok = qh < nh;
    const typename E::T *qrow = static_cast<const typename E::T *>(p.q) + b * p.q_row_stride +
                                (h0 + (ok ? qh : 0)) * D + (KV8 ? D / 4 : 2) * (lane & 3);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int e0 = KV8 ? 4 * ks : 16 * ks, e1 = KV8 ? 4 * ks + 2 : 16 * ks + 8;
      qf[n][ks][0] = ok ? __ldg(reinterpret_cast<const uint32_t *>(qrow + e0)) : 0u;
      qf[n][ks][1] = ok ? __ldg(reinterpret_cast<const uint32_t *>(qrow + e1)) : 0u;
    }
  }
}

// Widens four one-byte codes (one word) to two fp16 pairs exactly: lo gets
// bytes 0-1, hi bytes 2-3 (the lower byte in the lower half).  Every INT8
// code and every E4M3 value is an fp16 value.
//  INT8: with the sign bit flipped a code c is the byte u = c + 128; the
//    fp16 with bits 0x6400 | u is 1024 + u, and subtracting 1152 leaves c.
//  E4M3: the hardware converts two values per instruction.
template <bool FP8>
__device__ __forceinline__ void widen4(uint32_t w, uint32_t &lo, uint32_t &hi) {
  if constexpr (FP8) {
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"(static_cast<uint16_t>(w & 0xffffu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"(static_cast<uint16_t>(w >> 16)));
  } else {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(b) : "r"(u), "r"(0x64646464u));
    const __half2 off = __floats2half2_rn(1152.0f, 1152.0f);
    __half2 ha = __hsub2(*reinterpret_cast<__half2 *>(&a), off);
    __half2 hb = __hsub2(*reinterpret_cast<__half2 *>(&b), off);
    lo = *reinterpret_cast<uint32_t *>(&ha);
    hi = *reinterpret_cast<uint32_t *>(&hb);
  }
}

// Two code words a, b holding the same four elements of two tokens -> the
// fp16 pairs (a.byte i, b.byte i): e0 for i = 0, e1 for 1, e2 for 2, e3 for 3.
template <bool FP8>
__device__ __forceinline__ void widen_tokens(uint32_t a, uint32_t b, uint32_t &e0,
                                             uint32_t &e1, uint32_t &e2, uint32_t &e3) {
  uint32_t x, y;
  asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(x) : "r"(a), "r"(b));
  asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(y) : "r"(a), "r"(b));
  widen4<FP8>(x, e0, e1);
  widen4<FP8>(y, e2, e3);
}

// bf16 queries over one-byte pools run on the fp16 tensor-core path: each
// head's query is multiplied by the power of two 2^e that brings its largest
// magnitude into [2^14, 2^15) and rounded to fp16 -- exact for every element
// within 2^28 of that largest one (bf16 has 8 significant bits, fp16 11) --
// and the head's scores are multiplied back by 2^-e, so no query value
// leaves fp16's range.  Lane (head column, t) holds the pairs of load_q;
// qsc[n] receives 2^-e of the lane's head in column group n.
template <int D, int NG>
__device__ __forceinline__ void q_bf16_to_f16(uint32_t (&qf)[NG][D / 16][2],
                                              float (&qsc)[NG]) {
#pragma unroll
  for (int n = 0; n < NG; ++n) {
    float mx = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
      for (int j = 0; j < 2; ++j)
        mx = fmaxf(mx, fmaxf(fabsf(BF16::lo(qf[n][ks][j])), fabsf(BF16::hi(qf[n][ks][j]))));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));  // the head's four lanes
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    int e = 0;
    if (mx > 0.f) {
      const int ex = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 127;  // floor(log2)
      e = min(126, max(-126, 14 - ex));
    }
    const float f = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
      for (int j = 0; j < 2; ++j)
        qf[n][ks][j] = F16::pack2(BF16::lo(qf[n][ks][j]) * f, BF16::hi(qf[n][ks][j]) * f);
    qsc[n] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
  }
}

__device__ __forceinline__ void lds128(uint32_t addr, uint32_t (&w)[4]) {
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "r"(addr));
}
__device__ __forceinline__ void lds64(uint32_t addr, uint32_t &w0, uint32_t &w1) {
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(addr));
}

// Byte offset of 16-byte chunk c of stage row r (rows relative to a
// 1024-byte aligned region): 128-byte rows swizzle the chunk by r & 7,
// 64-byte rows (one-byte pools at D 64) by (r / 2) & 3, as TMA stores them.
template <int RP>
__device__ __forceinline__ uint32_t chunk_off(int r, int c) {
  if constexpr (RP == 128) return r * 128 + ((c ^ (r & 7)) << 4);
  else return r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
}

// KVF: the pool format -- 0 fp16/bf16 (as E), 1 INT8 codes, 2 FP8 (E4M3)
// codes.  NG: 8-head column groups per slice (1 or 2).  WR: the one-call
// step (the launch also writes the step's new rows); the plain decode is
// built without that code, which would otherwise cost it registers.
template <class E, int D, bool BAL, int KVF, int NG, bool WR>
__global__ void __launch_bounds__(threads_for(WR), kDecodeCtasPerSm)
    decode_persistent_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                             const __grid_constant__ CUtensorMap tmv) {
  constexpr bool KV8 = KVF != 0;  // one-byte codes, widened to fp16
  constexpr bool FP8 = KVF == 2;
  using M = std::conditional_t<KV8, F16, E>;  // the tensor cores' operand type
  constexpr bool BF = M::kBF16;
  constexpr bool QS = KV8 && E::kBF16;  // bf16 queries rescaled per head into fp16
  static_assert(!(WR && KV8), "the one-call step is built for 16-bit pools");
  using S = DecodeSmem<D, KV8>;
  constexpr int NH = S::kHalves;
  constexpr int NR = S::kRegions;
  constexpr int KSTEPS = D / 16;
  constexpr int NS = S::kStages;
  constexpr int ROWS = S::kRows;       // tokens per worker per stage
  constexpr int RB = S::kRegionBytes;  // one region of a stage
  constexpr int RP = S::kRowBytes;     // one stage row
  constexpr int NT = ROWS / 16;        // score tiles per stage
  constexpr int MAXBOX = ROWS / 8;     // most TMA boxes per worker per stage
  static_assert(NS <= 8, "stage headers");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::kBarOffset);
  uint64_t *empty = full + NS;
  volatile uint32_t *s_hdr = reinterpret_cast<volatile uint32_t *>(smem + S::kHdrOffset);
  volatile int *s_abort = reinterpret_cast<volatile int *>(smem + S::kAbortOffset);
  int *s_pref = reinterpret_cast<int *>(smem + S::kVarOffset);
  int *s_len = s_pref + p.num_seqs + 1;
  int *s_ids = s_len + p.num_seqs;  // [kWorkers][2][max_ids]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = p.partition_size;
  const int nseq = p.num_seqs;
  // Inputs come from earlier kernels (after a separate cache write, only its
  // K/V rows do: see after_write).
  if (!p.after_write) griddep_wait();
  griddep_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), kWorkers);
    }
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    // Items per sequence (checked context lengths) and their prefix sums.
    int carry = 0;
    for (int base = 0; base < nseq; base += 32) {
      const int b = base + lane;
      int items = 0;
      if (b < nseq) {
        const int L = checked_context_len(__ldg(p.context_lens + b), p.capacity, p.max_ctx,
                                          p.err, blockIdx.x == 0);
        s_len[b] = L;
        items = (BAL ? ceil16(L) : (L > 0 ? (L + P - 1) / P : 1)) * p.vh;
      }
      int incl = items;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (b < nseq) s_pref[b + 1] = carry + incl;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_pref[0] = 0;
  }
  if (warp == kWorkers && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  __syncthreads();

  Sched sc;
  sc.pref = s_pref;
  sc.len = s_len;
  sc.S = nseq;
  sc.vh = p.vh;
  sc.hq = p.hq;
  sc.G = p.group;
  sc.nc = p.nc;
  sc.hs = p.hs;
  sc.P = P;
  sc.NP = p.num_partitions;
  sc.NW = gridDim.x * kWorkers;
  sc.balanced = BAL;  // compile-time: each kernel carries one schedule's code
  sc.total = s_pref[nseq];
  sc.C = sc.balanced ? balanced_chunk(sc.total, sc.NW, p.chunk_cap) : 0;
  sc.chunks = sc.balanced ? (sc.total + sc.C - 1) / sc.C : 0;
  if (sc.balanced && blockIdx.x == 0 && p.ws_pref)
    for (int i = tid; i <= nseq; i += blockDim.x) p.ws_pref[i] = s_pref[i];
  const int bs = p.block_size;

  // The one-call step's cache write (16-bit pools), done by each CTA's
  // writer warp while the producer and the workers run: lane-global index i
  // covers 16-byte chunk i % C of token i / C's K and V rows (C chunks per
  // row, all KV heads), so each lane copies at most a chunk or two.  Slots
  // < 0 write nothing; slots past the pool are reported and skipped.
  auto write_new = [&]() {
    const int C = p.hkv * D / 8;
    const int64_t total = static_cast<int64_t>(p.nw) * C;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * 32;
#pragma unroll 1
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * 32 + lane; i < total; i += stride) {
      const int t = static_cast<int>(i / C), c = static_cast<int>(i - static_cast<int64_t>(t) * C);
      // the row's loads are issued with the slot's (their addresses do not
      // depend on it)
      const uint4 k = __ldg(reinterpret_cast<const uint4 *>(
                                static_cast<const typename E::T *>(p.new_k) + t * p.new_stride) +
                            c);
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(
                                static_cast<const typename E::T *>(p.new_v) + t * p.new_stride) +
                            c);
      const int64_t slot = __ldg(p.slot_mapping + t);
      if (slot < 0) continue;
      if (slot >= p.num_slots) {
        if (c == 0) raise_error(p.err, PA_DEVERR_SLOT);
        continue;
      }
      static_cast<uint4 *>(p.k_pool)[slot * C + c] = k;
      static_cast<uint4 *>(p.v_pool)[slot * C + c] = v;
    }
  };

  if constexpr (WR) {
    if (warp == kWriterWarp) {
      write_new();
      return;
    }
  }

  // ------------------------------------------------------------ producer --
  if (warp == kWorkers) {
    // Lane w (< 4) feeds worker w: it walks that worker's items block by
    // block, keeping the current item's position as (logical block, offset)
    // counters, and copies the block ids of the worker's next item into
    // shared memory with cp.async while the current item streams.  Lane 0
    // owns the stage barriers.  Lanes w + 4, w + 8, ... shadow worker w's
    // walk up to its first piece and help copy that piece's ids.
    const bool feeder = lane < kWorkers;
    const int wk = lane % kWorkers;
    const int boxr = p.box_rows;
    const int nbx = ROWS / boxr;  // boxes per worker per stage
    int cur = 0, endt = 0, gq = 0, sel = 0, lblk = 0, off = 0;
    int nstart = 0, nend = 0, ng = 0, nbuf = 0;
    bool act = false, have_next = false, want_next = false;
    Cursor pc = first_cursor(sc, blockIdx.x * kWorkers + wk);
    // Finds this worker's next piece with tokens (items of empty sequences
    // carry none: the worker writes their zeros itself) and starts copying
    // its block ids into buffer `buf`, ids k0, k0 + kstep, ... from this lane.
    auto prefetch = [&](int buf, int k0, int kstep) {
      Item m;
      have_next = false;
      while (next_piece(sc, pc, m)) {
        if (m.end <= m.start) continue;
        const int l0 = m.start / bs;
        const int nblk = (m.end - 1) / bs - l0 + 1;
        const int32_t *src = p.block_table + static_cast<int64_t>(m.b) * p.bt_stride + l0;
        const uint32_t dst = smem_u32(s_ids + (wk * 2 + buf) * p.max_ids);
        for (int k = k0; k < nblk; k += kstep) cp_async_4(dst + 4 * k, src + k);
        cp_async_commit();
        nstart = m.start;
        nend = m.end;
        ng = p.nc == 1 ? m.g : m.g / p.nc;  // the slice's KV head
        have_next = true;
        break;
      }
      nbuf = buf;
    };
    // Makes the prefetched piece current; the one after it is prefetched
    // once this piece's first copies are issued.
    auto promote = [&]() {
      act = have_next;
      if (!act) return;
      cp_async_wait_all();  // this item's ids (issued at least one item ago)
      cur = nstart;
      endt = nend;
      gq = ng;
      sel = nbuf;
      lblk = 0;
      off = nstart % bs;
      want_next = true;  // prefetched after this piece's first copies are issued
    };
    // The first piece: the whole warp copies its ids into buffer 0.
    prefetch(0, lane / kWorkers, 32 / kWorkers);
    cp_async_wait_all();
    __syncwarp();
    if (feeder) promote();
    const int *ids = s_ids;
    for (int c = 0;; ++c) {
      const int s = c % NS;
      int rows[MAXBOX];
      int nb = 0;
      bool bad = false;
      if (feeder) {
        if (want_next && c > 0) {  // the piece after the current one: its ids
          want_next = false;
          prefetch(sel ^ 1, 0, 1);
        }
        if (act && cur >= endt) promote();
        ids = s_ids + (lane * 2 + sel) * p.max_ids;
#pragma unroll
        for (int k = 0; k < MAXBOX; ++k) rows[k] = -1;
        if (act) {
          const int ntok = min(ROWS, endt - cur);
#pragma unroll
          for (int k = 0; k < MAXBOX; ++k) {
            if (k >= nbx || k * boxr >= ntok) break;
            const int id = ids[lblk];
            if (id >= 0 && id < p.num_blocks) {
              rows[k] = id * bs + off;
              ++nb;
            } else {
              bad = true;
            }
            off += boxr;
            if (off >= bs) {
              off = 0;
              ++lblk;
            }
          }
          cur += ROWS;
        }
      }
      if (c == 0 && p.after_write) griddep_wait();  // the cache write has landed
      const unsigned live = __ballot_sync(0xffffffffu, feeder && act);
      const unsigned badmask = __ballot_sync(0xffffffffu, bad);
      int nbox = nb;
#pragma unroll
      for (int o = 1; o < kWorkers; o <<= 1)  // lane 0 sums the feeder lanes 0..kWorkers-1
        nbox += __shfl_xor_sync(0xffffffffu, nbox, o);
      bool ok = true;
      if (lane == 0 && c >= NS)
        ok = mbar_wait_bounded(smem_u32(empty + s), ((c / NS) - 1) & 1, p.wait_ns);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok || *s_abort) {
        if (lane == 0) {
          if (!ok) raise_error(p.err, PA_DEVERR_TIMEOUT);
          *s_abort = 1;
          // Do not leave while copies this CTA issued may still land.
          for (int k = c - 1; k >= 0 && k >= c - NS; --k)
            mbar_wait_bounded(smem_u32(full + (k % NS)), (k / NS) & 1);
        }
        cp_async_wait_all();
        return;
      }
      if (live == 0) {
        if (lane == 0) {
          s_hdr[s] = kTerminate;
          mbar_arrive(smem_u32(full + s));
          // Leave only once the copies issued are in: a worker that gave up
          // waiting (a timed-out wait) no longer holds the block open.  Stage
          // c - NS was released by its consumers (the wait above), so its
          // data had landed; its slot now holds the terminate phase.
          for (int k = c - 1; k >= 0 && k > c - NS; --k)
            mbar_wait_bounded(smem_u32(full + (k % NS)), (k / NS) & 1);
        }
        cp_async_wait_all();
        return;
      }
      const uint32_t bar = smem_u32(full + s);
      if (lane == 0) {
        s_hdr[s] = badmask & ((1u << kWorkers) - 1);
        if (badmask) raise_error(p.err, PA_DEVERR_BLOCK_ID);
        // The barrier must expect exactly the bytes that land.
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nbox) * boxr * RP * NR * 2);
      }
      __syncwarp();
      if (feeder) {
        const uint32_t kdst = smem_u32(smem + s * S::kStageBytes);
        const uint32_t vdst = kdst + NR * RB;
#pragma unroll
        for (int k = 0; k < MAXBOX; ++k) {
          if (rows[k] < 0) continue;
          const uint32_t o = (lane * ROWS + k * boxr) * RP;
#pragma unroll
          for (int h = 0; h < NR; ++h) {
            tma_load_3d(kdst + h * RB + o, &tmk, bar, h * 64, gq, rows[k]);
            tma_load_3d(vdst + h * RB + o, &tmv, bar, h * 64, gq, rows[k]);
          }
        }
      }
    }
  }

  // ----------------------------------------------------- consumer = worker --
  float sl = p.scale_log2;  // one-byte pools: times the piece's K scale
  float vsc = 1.f;          // one-byte pools: the piece's V scale
  float slh[QS ? NG : 1][2];  // bf16 queries over one-byte pools: sl times each head's 2^-e
  const int r0 = warp * ROWS;  // this worker's rows in a stage
  const int mj = lane >> 3, mr = lane & 7;
  const int g8 = lane >> 2, t4 = lane & 3;

  uint32_t qf[NG][KSTEPS][2];
  uint32_t qn[NG == 1 ? KSTEPS : 1][2];  // the next piece's query (one column group)
  float o[NG][KSTEPS][4];
  float mst[NG][2], lst[NG][2];
  bool item_bad = false;
  Item cur_item;
  Cursor wc = first_cursor(sc, blockIdx.x * kWorkers + warp);
  int qn_b = -1, qn_g = -1;  // the unit whose query qn holds
  int cur = 0;
  // The one-call step: the piece holds its unit's newest row (position
  // L - 1); the step's input K/V rows of that token are on their way into
  // this worker's shared buffer, with the row's block id and the token's
  // slot_mapping entry (see put_newest).
  bool nw_on = false;
  uint8_t *s_new = smem + S::kNewOffset + warp * S::kNewBytes;
  int64_t *s_nw = reinterpret_cast<int64_t *>(s_new + S::kNewMeta);  // [block id, token b's slot]
  if (sc.balanced) {
    // Empty sequences have no pieces: their (zero) outputs are written here.
    for (int b = blockIdx.x * kWorkers + warp; b < nseq; b += sc.NW) {
      if (s_len[b] != 0) continue;
      uint4 *orow = reinterpret_cast<uint4 *>(static_cast<typename E::T *>(p.out) +
                                              b * p.out_row_stride);
      for (int e = lane; e < p.hq * D / 8; e += 32) orow[e] = make_uint4(0, 0, 0, 0);
    }
  }

  // Writes a finished item: the normalised output when it is its sequence's
  // only partition, else its softmax state for the combine.
  auto finalize = [&](const Item &m, bool bad_item) {
    int nh;
    const int h0 = slice_head0(sc, m.g, nh);
#pragma unroll
    for (int n = 0; n < NG; ++n)
#pragma unroll
      for (int s = 4; s < 32; s <<= 1) {
        lst[n][0] += shfl_xor(lst[n][0], s);
        lst[n][1] += shfl_xor(lst[n][1], s);
      }
#pragma unroll
    for (int n = 0; n < NG; ++n) {
      const int hA = 8 * n + 2 * t4, hB = hA + 1;  // this lane's heads in the slice
      const float lA = lst[n][0], lB = lst[n][1];
      if constexpr (KV8) {
        // O^T rows in the one-byte order: lane (g, t) holds elements
        // (D/8)g .. (D/8)g + D/8 - 1 of heads 2t and 2t + 1, element
        // (D/8)g + i in o[i / 2][i % 2 ? 2 : 0] (head 2t) and
        // o[i / 2][i % 2 ? 3 : 1] (head 2t + 1).
        const int e0 = (D / 8) * g8;
        if (m.direct) {
          typename E::T *out = static_cast<typename E::T *>(p.out) + m.b * p.out_row_stride +
                               h0 * D + e0;
          const float iA = (!bad_item && lA > 0.f) ? vsc / lA : 0.f;
          const float iB = (!bad_item && lB > 0.f) ? vsc / lB : 0.f;
          uint32_t uA[KSTEPS], uB[KSTEPS];
#pragma unroll
          for (int mt = 0; mt < KSTEPS; ++mt) {
            uA[mt] = E::pack2(o[n][mt][0] * iA, o[n][mt][2] * iA);
            uB[mt] = E::pack2(o[n][mt][1] * iB, o[n][mt][3] * iB);
          }
          if constexpr (D == 128) {
            if (hA < nh) {
              uint4 *d = reinterpret_cast<uint4 *>(out + hA * D);
              d[0] = make_uint4(uA[0], uA[1], uA[2], uA[3]);
              d[1] = make_uint4(uA[4], uA[5], uA[6], uA[7]);
            }
            if (hB < nh) {
              uint4 *d = reinterpret_cast<uint4 *>(out + hB * D);
              d[0] = make_uint4(uB[0], uB[1], uB[2], uB[3]);
              d[1] = make_uint4(uB[4], uB[5], uB[6], uB[7]);
            }
          } else {
            if (hA < nh)
              *reinterpret_cast<uint4 *>(out + hA * D) = make_uint4(uA[0], uA[1], uA[2], uA[3]);
            if (hB < nh)
              *reinterpret_cast<uint4 *>(out + hB * D) = make_uint4(uB[0], uB[1], uB[2], uB[3]);
          }
        } else {
          const float f = bad_item ? 0.f : vsc;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int h = hA + hh;
            if (h >= nh) continue;
            float4 *w = reinterpret_cast<float4 *>(p.ws_o + (m.prow + h * m.pstride) * D + e0);
#pragma unroll
            for (int q = 0; q < D / 32; ++q)
              w[q] = make_float4(o[n][2 * q][hh] * f, o[n][2 * q][hh + 2] * f,
                                 o[n][2 * q + 1][hh] * f, o[n][2 * q + 1][hh + 2] * f);
          }
          if (lane < 4) {
            if (hA < nh) {
              p.ws_ml[(m.prow + hA * m.pstride) * 2 + 0] = bad_item ? -INFINITY : mst[n][0];
              p.ws_ml[(m.prow + hA * m.pstride) * 2 + 1] = bad_item ? 0.f : lA;
            }
            if (hB < nh) {
              p.ws_ml[(m.prow + hB * m.pstride) * 2 + 0] = bad_item ? -INFINITY : mst[n][1];
              p.ws_ml[(m.prow + hB * m.pstride) * 2 + 1] = bad_item ? 0.f : lB;
            }
          }
        }
        continue;
      }
      if (m.direct) {
        const float iA = (!bad_item && lA > 0.f) ? 1.f / lA : 0.f;
        const float iB = (!bad_item && lB > 0.f) ? 1.f / lB : 0.f;
        typename E::T *out =
            static_cast<typename E::T *>(p.out) + m.b * p.out_row_stride + h0 * D;
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt) {
          const int d0 = mt * 16 + g8, d1 = d0 + 8;
          if (hA < nh) {
            out[hA * D + d0] = E::from_float(o[n][mt][0] * iA);
            out[hA * D + d1] = E::from_float(o[n][mt][2] * iA);
          }
          if (hB < nh) {
            out[hB * D + d0] = E::from_float(o[n][mt][1] * iB);
            out[hB * D + d1] = E::from_float(o[n][mt][3] * iB);
          }
        }
      } else {
        const int64_t row0 = m.prow;
        const int64_t hstride = m.pstride;
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt) {
          const int d0 = mt * 16 + g8, d1 = d0 + 8;
          if (hA < nh) {
            float *w0 = p.ws_o + (row0 + hA * hstride) * D;
            w0[d0] = bad_item ? 0.f : o[n][mt][0];
            w0[d1] = bad_item ? 0.f : o[n][mt][2];
          }
          if (hB < nh) {
            float *w1 = p.ws_o + (row0 + hB * hstride) * D;
            w1[d0] = bad_item ? 0.f : o[n][mt][1];
            w1[d1] = bad_item ? 0.f : o[n][mt][3];
          }
        }
        if (lane < 4) {
          if (hA < nh) {
            p.ws_ml[(row0 + hA * hstride) * 2 + 0] = bad_item ? -INFINITY : mst[n][0];
            p.ws_ml[(row0 + hA * hstride) * 2 + 1] = bad_item ? 0.f : lA;
          }
          if (hB < nh) {
            p.ws_ml[(row0 + hB * hstride) * 2 + 0] = bad_item ? -INFINITY : mst[n][1];
            p.ws_ml[(row0 + hB * hstride) * 2 + 1] = bad_item ? 0.f : lB;
          }
        }
      }
    }
  };
  // Starts this worker's next piece with tokens; items of empty sequences
  // (fixed schedule) are finished on the spot (zero output).
  auto begin = [&]() -> bool {
    Item m;
    while (next_piece(sc, wc, m)) {
#pragma unroll
      for (int n = 0; n < NG; ++n) {
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt)
          o[n][mt][0] = o[n][mt][1] = o[n][mt][2] = o[n][mt][3] = 0.f;
        mst[n][0] = mst[n][1] = -INFINITY;
        lst[n][0] = lst[n][1] = 0.f;
      }
      item_bad = false;
      int nh;
      const int h0 = slice_head0(sc, m.g, nh);
      if (m.end > m.start) {
        bool have_q = false;
        if constexpr (NG == 1) {
          if (qn_b == m.b && qn_g == m.g) {
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
              qf[0][ks][0] = qn[ks][0];
              qf[0][ks][1] = qn[ks][1];
            }
            have_q = true;
          }
        }
        if (!have_q) load_q<E, D, KV8, NG>(qf, p, m.b, h0, nh, lane);
        cur_item = m;
        cur = m.start;
        const int kvh = p.nc == 1 ? m.g : m.g / p.nc;
        if constexpr (KV8) {
          // The piece's KV head's scales: K's scales the scores, V's the
          // output.  One that is not a positive finite number makes the
          // piece contribute nothing (zeros / an empty softmax state).
          const float ks = __ldg(p.k_scale + kvh), vs = __ldg(p.v_scale + kvh);
          sl = p.scale_log2 * ks;
          vsc = vs;
          if (!(scale_ok(ks) && scale_ok(vs))) {
            item_bad = true;
            if (lane == 0) raise_error(p.err, PA_DEVERR_SCALE);
          }
        }
        if constexpr (QS) {
          float qsc[NG];
          q_bf16_to_f16<D, NG>(qf, qsc);
#pragma unroll
          for (int n = 0; n < NG; ++n) {  // heads 8n + 2t, +1 sit in head columns 2t, 2t + 1
            slh[n][0] = sl * __shfl_sync(0xffffffffu, qsc[n], 8 * t4);
            slh[n][1] = sl * __shfl_sync(0xffffffffu, qsc[n], 8 * t4 + 4);
          }
        }
        // The one-call step: the newest row's block id and, for the usual
        // step (token b is sequence b's new token), token b's slot and its
        // input rows (copied into this worker's buffer: 16 bytes per lane,
        // K then V), all used at the row's stage.
        nw_on = WR && m.end == m.L;
        if (nw_on) {
          // copied asynchronously (no register waits on them here)
          if (lane == 0) {  // the block id lands in the low word
            cp_async_4(smem_u32(s_nw),
                       p.block_table + static_cast<int64_t>(m.b) * p.bt_stride + (m.L - 1) / bs);
            if (m.b < p.nw) cp_async_8(smem_u32(s_nw + 1), p.slot_mapping + m.b);
            else s_nw[1] = -2;
          }
          if (m.b < p.nw) {
            if (lane < D / 4) {
              const typename E::T *src = static_cast<const typename E::T *>(
                                             lane < D / 8 ? p.new_k : p.new_v) +
                                         m.b * p.new_stride + kvh * D + 8 * (lane % (D / 8));
              cp_async_16(smem_u32(s_new + lane * 16), src);
            }
          }
          cp_async_commit();
        }
        if constexpr (NG == 1) {
          // Prefetch the next piece's query one piece ahead.
          Cursor peek = wc;
          Item nm;
          qn_b = qn_g = -1;
          while (next_piece(sc, peek, nm)) {
            if (nm.end <= nm.start) continue;
            int nnh;
            const int nh0 = slice_head0(sc, nm.g, nnh);
            load_q<E, D, KV8, 1>(reinterpret_cast<uint32_t(&)[1][KSTEPS][2]>(qn), p, nm.b, nh0,
                                 nnh, lane);
            qn_b = nm.b;
            qn_g = nm.g;
            break;
          }
        } else {
          // Wider slices keep no second query in registers: pull the next
          // piece's query rows into L2 instead.
          Cursor peek = wc;
          Item nm;
          while (next_piece(sc, peek, nm)) {
            if (nm.end <= nm.start) continue;
            int nnh;
            const int nh0 = slice_head0(sc, nm.g, nnh);
            const char *qb = reinterpret_cast<const char *>(
                static_cast<const typename E::T *>(p.q) + nm.b * p.q_row_stride + nh0 * D);
            const int lines = (nnh * D * 2 + 127) / 128;
            for (int i = lane; i < lines; i += 32)
              asm volatile("prefetch.global.L2 [%0];" ::"l"(qb + i * 128));
            break;
          }
        }
        return true;
      }
      if constexpr (!BAL) finalize(m, false);  // empty sequence: zeros
    }
    return false;
  };
  // Puts the piece's newest row (stage row rr of this worker) in place: the
  // pool row as the TMA loaded it may or may not already hold this step's
  // write, so when a new token is written to that row's slot the row is
  // taken from the token's input instead (one-byte pools take the write's
  // quantiser, so the codes are the ones the write stores).  The token is
  // token b when slot_mapping[b] is the row's slot (the usual step), else the
  // last token sent there; with none, the pool's row stands.  A bad block
  // id leaves the stage as loaded: the piece is flagged by the producer and
  // contributes nothing.
  auto put_newest = [&](uint8_t *kst, int rr) -> bool {
    cp_async_wait_all();
    __syncwarp();
    const int64_t nw_id = *reinterpret_cast<const int32_t *>(s_nw), nw_sm = s_nw[1];
    if (nw_id < 0 || nw_id >= p.num_blocks) return false;
    const int64_t slot = nw_id * bs + (cur_item.L - 1) % bs;
    const int kvh = p.nc == 1 ? cur_item.g : cur_item.g / p.nc;
    if (nw_sm != slot) {
      int t = -1;
      for (int base = 0; base < p.nw; base += 32) {
        const int tt = base + lane;
        const unsigned hit =
            __ballot_sync(0xffffffffu, tt < p.nw && __ldg(p.slot_mapping + tt) == slot);
        if (hit) t = base + 31 - __clz(hit);
      }
      if (t < 0) return false;  // no token of this step is written to the row
      if (lane < D / 4)
        *reinterpret_cast<uint4 *>(s_new + lane * 16) = __ldg(reinterpret_cast<const uint4 *>(
            static_cast<const typename E::T *>(lane < D / 8 ? p.new_k : p.new_v) +
            t * p.new_stride + kvh * D + 8 * (lane % (D / 8))));
      __syncwarp();
    }
    const int row = r0 + rr;
    constexpr int C = D / 8;  // 16-byte chunks of a stage row, per tensor
    if (lane < 2 * C) {
      const int which = lane / C, c = lane % C, h = c >> 3;  // h: 64-element half
      *reinterpret_cast<uint4 *>(kst + which * NH * RB + h * RB + chunk_off<128>(row, c & 7)) =
          *(reinterpret_cast<const uint4 *>(s_new) + lane);
    }
    __syncwarp();
    return true;
  };
  // The next piece starts at the top of the loop, before its first stage is
  // waited for (its query loads overlap the wait).
  bool active = false, need_piece = true;
  for (int c = 0;; ++c) {
    const int s = c % NS;
    if (need_piece) {
      active = begin();
      need_piece = false;
    }
    if (!mbar_wait_bounded(smem_u32(full + s), (c / NS) & 1, p.wait_ns)) {
      raise_error(p.err, PA_DEVERR_TIMEOUT);
      *s_abort = 1;
      break;
    }
    const uint32_t hdr = s_hdr[s];
    if (hdr & kTerminate) break;
    bool released = false;
    if (active) {
      const int end = cur_item.end;
      const int j0 = cur;
      uint8_t *kst = smem + s * S::kStageBytes;
      bool touched = false;  // generic-proxy writes into the stage
      // the piece's newest row (one-call step): this worker's stage row
      // end - 1 - j0
      if (WR && nw_on && end - 1 < j0 + ROWS) touched = put_newest(kst, end - 1 - j0);
      if constexpr (!KV8) {
        if (j0 + ROWS > end) {
          // Rows past the context may hold anything (even NaN); their weight
          // is zero, so make their V rows exact zeros before the P.V product.
          uint8_t *vrows = kst + NH * RB;
          for (int i = lane; i < ROWS * NH * 8; i += 32) {
            const int rr = i / (NH * 8), h = (i / 8) % NH, cc = i % 8;
            if (j0 + rr >= end)
              *reinterpret_cast<uint4 *>(vrows + h * RB + (r0 + rr) * 128 + cc * 16) =
                  make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
          touched = true;
        }
      }
      // One-byte pools with two column groups take the stage's two 16-token
      // tiles one after the other (fewer live registers); otherwise one pass.
      constexpr int PASSES = (KV8 && NG == 2) ? 2 : 1;
      constexpr int NTP = NT / PASSES;       // score tiles per pass
      constexpr int VWW = KV8 ? D / 32 : 1;  // code words per V token row per lane
#pragma unroll
      for (int ps = 0; ps < PASSES; ++ps) {
        float sc2[NG][NTP][4];
#pragma unroll
        for (int n = 0; n < NG; ++n)
#pragma unroll
          for (int u = 0; u < NTP; ++u)
            sc2[n][u][0] = sc2[n][u][1] = sc2[n][u][2] = sc2[n][u][3] = 0.f;
        uint32_t vw[KV8 ? NTP : 1][4][VWW];  // one-byte pools: this lane's V codes
        if constexpr (KV8) {
          // This worker's 32 one-byte K and V rows (two 16-token tiles) go
          // straight to registers.  Codes widen exactly whatever the pool
          // held, so rows past the context need no clearing: their weight is
          // zero.
          //  K, the A operand of S^T = K Q^T (rows: tokens 16u + g, +8):
          //   k-step ks of lane (g, t) is elements (D/4)t + 4ks .. +3 of its
          //   rows (16-byte chunks (D/64)t .. of the row), the query
          //   following suit.
          //  V, the A operand of O^T += V^T P^T (rows: elements of D;
          //   columns: tokens 16u + 2t, +1, +8, +9): the D order of O^T is
          //   free as well, so lane (g, t) owns elements (D/8)g .. (D/8)g +
          //   D/8 - 1 of its token rows, row g of M-tile mt holding element
          //   (D/8)g + 2mt and row g + 8 element (D/8)g + 2mt + 1.
          const uint32_t kr = smem_u32(kst) + r0 * RP;
          const uint32_t vr = smem_u32(kst) + RB + r0 * RP;
          constexpr int KC = D / 64;  // 16-byte K chunks per lane per row
          // K codes: every tile's loads issued before the first widening
          // (one column group), or a chunk at a time (two: fewer registers).
          constexpr int KL = NG == 1 ? KC : 1;  // chunks loaded per batch
#pragma unroll
          for (int cb = 0; cb < KC; cb += KL) {
            uint32_t kw[NTP][2][KL][4];  // [tile][row g | g + 8][chunk][word]
#pragma unroll
            for (int uu = 0; uu < NTP; ++uu)
#pragma unroll
              for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int cc = 0; cc < KL; ++cc)
                  lds128(kr + chunk_off<RP>(16 * (ps * NTP + uu) + g8 + 8 * r,
                                            KC * t4 + cb + cc),
                         kw[uu][r][cc]);

#pragma unroll
            for (int kq = 0; kq < 4 * KL; ++kq) {
              const int ks = 4 * cb + kq;
#pragma unroll
              for (int uu = 0; uu < NTP; ++uu) {
                uint32_t a0, a1, a2, a3;
                widen4<FP8>(kw[uu][0][kq >> 2][kq & 3], a0, a2);
                widen4<FP8>(kw[uu][1][kq >> 2][kq & 3], a1, a3);
#pragma unroll
                for (int n = 0; n < NG; ++n)
                  mma_16816<BF>(sc2[n][uu], a0, a1, a2, a3, qf[n][ks][0], qf[n][ks][1]);
              }
            }
          }
          // V's codes once K's are spent (fewer live registers); their loads
          // overlap the softmax below, and the stage is handed back once the
          // last pass has read them.
          const int v0 = 2 * t4;
#pragma unroll
          for (int uu = 0; uu < NTP; ++uu) {
            const int u = ps * NTP + uu;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int tr = 16 * u + v0 + (i & 1) + 8 * (i >> 1);  // token row
              if constexpr (D == 128) {
                lds128(vr + chunk_off<RP>(tr, g8), reinterpret_cast<uint32_t(&)[4]>(vw[uu][i]));
              } else {
                lds64(vr + chunk_off<RP>(tr, g8 >> 1) + 8 * (g8 & 1), vw[uu][i][0],
                      vw[uu][i][1]);
              }
            }
          }
          if (ps == PASSES - 1) {
            __syncwarp();
            if (touched) fence_proxy_async_smem();  // generic writes before the next TMA
            if (lane == 0) mbar_arrive(smem_u32(empty + s));
            released = true;
          }
          if constexpr (FP8) {
            // An E4M3 byte can be a NaN code: V rows past the context (stale
            // or unwritten) become exact zeros.  K's are masked out of the
            // scores.
            if (j0 + ROWS > end) {
#pragma unroll
              for (int uu = 0; uu < NTP; ++uu)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  if (j0 + 16 * (ps * NTP + uu) + v0 + (i & 1) + 8 * (i >> 1) >= end)
#pragma unroll
                    for (int w = 0; w < VWW; ++w) vw[uu][i][w] = 0u;
            }
          }
        } else {
          // S^T = K Q^T for this worker's 16 tokens.
          const uint32_t kb = smem_u32(kst);
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks) {
            const int row = r0 + (mj & 1) * 8 + mr;
            const int c16 = ks * 2 + (mj >> 1);
            const uint32_t addr =
                kb + (c16 >> 3) * RB + row * 128 + (((c16 & 7) ^ (row & 7)) << 4);
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(addr, a0, a1, a2, a3);
#pragma unroll
            for (int n = 0; n < NG; ++n)
              mma_16816<BF>(sc2[n][0], a0, a1, a2, a3, qf[n][ks][0], qf[n][ks][1]);
          }
        }
        // Scores of tile u = ps * NTP + uu, group n: tokens j0 + 16u + g
        // (sc2[n][uu][0..1], heads 8n + 2t, +1) and j0 + 16u + g + 8
        // (sc2[n][uu][2..3]).
        uint32_t pb[NG][NTP][2];
#pragma unroll
        for (int n = 0; n < NG; ++n) {
          float sv[NTP][4];
          float mx0 = -INFINITY, mx1 = -INFINITY;
          float slA = sl, slB = sl;  // the score factors of this lane's two heads
          if constexpr (QS) {
            slA = slh[n][0];
            slB = slh[n][1];
          }
#pragma unroll
          for (int uu = 0; uu < NTP; ++uu) {
            const int t0 = j0 + 16 * (ps * NTP + uu) + g8, t1 = t0 + 8;
            sv[uu][0] = t0 < end ? sc2[n][uu][0] * slA : -INFINITY;
            sv[uu][1] = t0 < end ? sc2[n][uu][1] * slB : -INFINITY;
            sv[uu][2] = t1 < end ? sc2[n][uu][2] * slA : -INFINITY;
            sv[uu][3] = t1 < end ? sc2[n][uu][3] * slB : -INFINITY;
            mx0 = fmaxf(mx0, fmaxf(sv[uu][0], sv[uu][2]));
            mx1 = fmaxf(mx1, fmaxf(sv[uu][1], sv[uu][3]));
          }
#pragma unroll
          for (int m = 4; m < 32; m <<= 1) {
            mx0 = fmaxf(mx0, shfl_xor(mx0, m));
            mx1 = fmaxf(mx1, shfl_xor(mx1, m));
          }
          const float mn0 = fmaxf(mst[n][0], mx0), mn1 = fmaxf(mst[n][1], mx1);
          const float cr0 = exp2f(mst[n][0] - mn0), cr1 = exp2f(mst[n][1] - mn1);
          mst[n][0] = mn0;
          mst[n][1] = mn1;
          // P is rounded to the operand type for the tensor core; the row
          // sums use the same rounded values, so the output is an exact
          // weighted mean of V under the rounded weights.
          float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
          for (int uu = 0; uu < NTP; ++uu) {
            const uint32_t w0 = M::pack2(exp2f(sv[uu][0] - mn0), exp2f(sv[uu][1] - mn1));  // t0
            const uint32_t w1 = M::pack2(exp2f(sv[uu][2] - mn0), exp2f(sv[uu][3] - mn1));  // t1
            ls0 += M::lo(w0) + M::lo(w1);
            ls1 += M::hi(w0) + M::hi(w1);
            // P^T fragments (tokens x heads) from the S^T accumulator layout.
            pb[n][uu][0] = movmatrix_trans(w0);
            pb[n][uu][1] = movmatrix_trans(w1);
          }
          lst[n][0] = lst[n][0] * cr0 + ls0;
          lst[n][1] = lst[n][1] * cr1 + ls1;
#pragma unroll
          for (int mt = 0; mt < KSTEPS; ++mt) {
            o[n][mt][0] *= cr0;
            o[n][mt][1] *= cr1;
            o[n][mt][2] *= cr0;
            o[n][mt][3] *= cr1;
          }
        }
        // O^T += V^T P^T, one 16-wide slice of D at a time.
        if constexpr (KV8) {
          // Word w of the lane's token-row bytes: M-tiles 2w and 2w + 1.
#pragma unroll
          for (int w = 0; w < VWW; ++w)
#pragma unroll
            for (int uu = 0; uu < NTP; ++uu) {
              uint32_t a0, a1, b0, b1, a2, a3, b2, b3;
              widen_tokens<FP8>(vw[uu][0][w], vw[uu][1][w], a0, a1, b0, b1);  // tokens 2t, +1
              widen_tokens<FP8>(vw[uu][2][w], vw[uu][3][w], a2, a3, b2, b3);  // 2t + 8, + 9
#pragma unroll
              for (int n = 0; n < NG; ++n) {
                mma_16816<BF>(o[n][2 * w], a0, a1, a2, a3, pb[n][uu][0], pb[n][uu][1]);
                mma_16816<BF>(o[n][2 * w + 1], b0, b1, b2, b3, pb[n][uu][0], pb[n][uu][1]);
              }
            }
        } else {
          const uint32_t vb = smem_u32(kst) + NH * RB;
#pragma unroll
          for (int mt = 0; mt < KSTEPS; ++mt) {
            const int row = r0 + (mj >> 1) * 8 + mr;
            const int c16 = mt * 2 + (mj & 1);
            const uint32_t addr =
                vb + (c16 >> 3) * RB + row * 128 + (((c16 & 7) ^ (row & 7)) << 4);
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4_trans(addr, a0, a1, a2, a3);
#pragma unroll
            for (int n = 0; n < NG; ++n)
              mma_16816<BF>(o[n][mt], a0, a1, a2, a3, pb[n][0][0], pb[n][0][1]);
          }
          if (touched) fence_proxy_async_smem();  // generic writes before the next TMA
        }
      }
      if (hdr & (1u << warp)) item_bad = true;
      cur += ROWS;
      if (cur >= end) {
        finalize(cur_item, item_bad);
        need_piece = true;
      }
    }
    if (!released) {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(empty + s));
    }
  }
}

// Merges the pieces of each (sequence, query head) by log-sum-exp:
//   M = max_p m_p,  w_p = 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p l_p.
// One CTA of four warps per (sequence, query head).  Warp w takes pieces
// w, w+4, ... eight at a time -- all their loads issued together, then
// folded into a running (max, sum, D/32 output elements per lane) -- and the
// four warps' states are folded once more through shared memory.  A unit's
// pieces are workspace rows row0 + i * rstride: partitions 0..n-1 (fixed
// schedule) or chunks c0..c1 (balanced schedule, piece (unit u, chunk c) in
// rows (u + c) * hs + h).
constexpr int kCombineWarps = 4;
constexpr int kCombineBatch = 8;
constexpr int kCombineLocalPref = 64;  // most sequences whose prefix sums a CTA forms itself

template <class E, int D>
__global__ void __launch_bounds__(kCombineWarps * 32) decode_combine_kernel(const DecodeParams p) {
  constexpr int V = D / 32;  // output elements per lane
  __shared__ float s_m[kCombineWarps], s_l[kCombineWarps];
  __shared__ float s_o[kCombineWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x / p.hq, h = blockIdx.x - b * p.hq;
  // context_lens is an input of the decode kernel, not its output: read it
  // while the decode kernel is still running.
  const int L = checked_context_len(__ldg(p.context_lens + b), p.capacity, p.max_ctx, p.err, false);
  // Balanced schedule, few sequences: the prefix sums of the token stream
  // from context_lens too (as the decode kernel forms them), so that after
  // the wait only the partial states remain to be read.
  const bool local_pref = p.balanced && p.num_seqs <= kCombineLocalPref;
  int pref_b = 0, total = 0;
  if (local_pref) {
    for (int base = 0; base < p.num_seqs; base += 32) {
      const int sq = base + lane;
      int v = 0;
      if (sq < p.num_seqs)
        v = ceil16(checked_context_len(__ldg(p.context_lens + sq), p.capacity, p.max_ctx, p.err,
                                       false)) *
            p.vh;
      pref_b += __reduce_add_sync(0xffffffffu, sq < b ? v : 0);
      total += __reduce_add_sync(0xffffffffu, v);
    }
  }
  // The unit's pieces: workspace rows row0 + i * rstride, i < n.
  int n = 0;
  int64_t row0 = 0, rstride = 1;
  auto locate = [&]() {
    if (p.balanced) {
      if (L <= 0) return;  // zeros written by the decode kernel
      const int G = p.group, kvh = h / G, hg = h - kvh * G;
      const int slc = hg / p.hs, hh = hg - slc * p.hs;
      const int g = kvh * p.nc + slc;  // the unit within the sequence
      const int C = balanced_chunk(total, p.num_workers, p.chunk_cap);
      const int U = pref_b + g * ceil16(L);  // the unit's first position
      const int c0 = U / C, c1 = (U + L - 1) / C;
      n = c1 - c0 + 1;
      row0 = (static_cast<int64_t>(b) * p.vh + g + c0) * p.hs + hh;
      rstride = p.hs;
    } else {
      n = (L + p.partition_size - 1) / p.partition_size;
      row0 = (static_cast<int64_t>(b) * p.hq + h) * p.num_partitions;
      rstride = 1;
    }
  };
  const bool early = !p.balanced || local_pref;  // known before the decode kernel ends
  if (early) {
    locate();
    if (n <= 1) return;  // written by the decode kernel itself
  }
  griddep_wait();  // the partial states of the decode kernel
  griddep_launch_dependents();
  if (!early) {
    total = p.ws_pref[p.num_seqs];
    pref_b = p.ws_pref[b];
    locate();
  }
  if (n <= 1) return;  // written by the decode kernel itself
  const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml);
  const float *po = p.ws_o + lane * V;

  // This warp's pieces, folded with an online max.
  float M = -INFINITY, Ls = 0.f, acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  for (int i0 = warp; i0 < n; i0 += kCombineWarps * kCombineBatch) {
    float2 st[kCombineBatch];
    float ov[kCombineBatch][V];
#pragma unroll
    for (int k = 0; k < kCombineBatch; ++k) {
      const int i = i0 + k * kCombineWarps;
      const int64_t r = row0 + static_cast<int64_t>(i < n ? i : 0) * rstride;
      st[k] = i < n ? ml[r] : make_float2(-INFINITY, 0.f);
      if constexpr (V == 4) {
        const float4 o4 = i < n ? *reinterpret_cast<const float4 *>(po + r * D)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        ov[k][0] = o4.x;
        ov[k][1] = o4.y;
        ov[k][2] = o4.z;
        ov[k][3] = o4.w;
      } else {
        const float2 o2 =
            i < n ? *reinterpret_cast<const float2 *>(po + r * D) : make_float2(0.f, 0.f);
        ov[k][0] = o2.x;
        ov[k][1] = o2.y;
      }
    }
    float Mn = M;
#pragma unroll
    for (int k = 0; k < kCombineBatch; ++k) Mn = fmaxf(Mn, st[k].x);
    if (Mn == -INFINITY) continue;  // nothing visible yet
    const float cr = exp2f(M - Mn);  // 0 while M is -inf
    Ls *= cr;
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] *= cr;
#pragma unroll
    for (int k = 0; k < kCombineBatch; ++k) {
      const float w = exp2f(st[k].x - Mn);  // 0 for padding and empty pieces
      Ls += w * st[k].y;
#pragma unroll
      for (int v = 0; v < V; ++v) acc[v] += w * ov[k][v];
    }
    M = Mn;
  }
  if (lane == 0) {
    s_m[warp] = M;
    s_l[warp] = Ls;
  }
#pragma unroll
  for (int v = 0; v < V; ++v) s_o[warp][lane * V + v] = acc[v];
  __syncthreads();
  if (warp != 0) return;
  float Mt = -INFINITY;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) Mt = fmaxf(Mt, s_m[w]);
  float lt = 0.f, out_v[V];
#pragma unroll
  for (int v = 0; v < V; ++v) out_v[v] = 0.f;
  if (Mt != -INFINITY) {
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) {
      const float f = exp2f(s_m[w] - Mt);  // 0 for a warp that saw nothing
      lt += f * s_l[w];
#pragma unroll
      for (int v = 0; v < V; ++v) out_v[v] += f * s_o[w][lane * V + v];
    }
  }
  // a sum that is not positive (no visible key, or a non-finite state from a
  // bad block) gives zeros
  const bool good = lt > 0.f;
  const float inv = good ? 1.f / lt : 0.f;
  typename E::T *out =
      static_cast<typename E::T *>(p.out) + b * p.out_row_stride + h * D + lane * V;
  if constexpr (V == 4) {
    *reinterpret_cast<uint2 *>(out) =
        make_uint2(E::pack2(good ? out_v[0] * inv : 0.f, good ? out_v[1] * inv : 0.f),
                   E::pack2(good ? out_v[2] * inv : 0.f, good ? out_v[3] * inv : 0.f));
  } else {
    *reinterpret_cast<uint32_t *>(out) =
        E::pack2(good ? out_v[0] * inv : 0.f, good ? out_v[1] * inv : 0.f);
  }
}

template <class E, int D, bool BAL, int KVF, int NG, bool WR = false>
cudaError_t launch_kernel(const DecodeArgs &a, const DecodeParams &p, cudaStream_t stream) {
  using S = DecodeSmem<D, KVF != 0>;
  const int smem = S::bytes(a.num_seqs, p.max_ids);
  auto kernel = decode_persistent_kernel<E, D, BAL, KVF, NG, WR>;
  cudaError_t e = allow_dynamic_smem<decode_persistent_kernel<E, D, BAL, KVF, NG, WR>>();
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(static_cast<unsigned>(a.grid)), dim3(threads_for(WR)), smem,
                    stream,
                    p, a.tm_k, a.tm_v);
}

// The decode kernel of the schedule, head-group width and head dim in `p`,
// then (when pieces need combining) the merge kernel.  The one-call step
// (p.nw > 0) is built for 16-bit pools and the balanced schedule; the
// launcher sends every other step through a separate write launch.
template <class E, int KVF>
cudaError_t launch_family(const DecodeArgs &a, const DecodeParams &p, cudaStream_t stream) {
  cudaError_t e;
  const bool bal = p.balanced != 0, wide = p.hs > 8;
  if (p.nw > 0) {
    if constexpr (KVF != 0) {
      return cudaErrorInvalidValue;
    } else {
      if (!bal) return cudaErrorInvalidValue;
      e = a.head_dim == 128 ? (wide ? launch_kernel<E, 128, true, KVF, 2, true>(a, p, stream)
                                    : launch_kernel<E, 128, true, KVF, 1, true>(a, p, stream))
                            : (wide ? launch_kernel<E, 64, true, KVF, 2, true>(a, p, stream)
                                    : launch_kernel<E, 64, true, KVF, 1, true>(a, p, stream));
    }
  } else if (a.head_dim == 128) {
    e = bal ? (wide ? launch_kernel<E, 128, true, KVF, 2>(a, p, stream)
                    : launch_kernel<E, 128, true, KVF, 1>(a, p, stream))
            : (wide ? launch_kernel<E, 128, false, KVF, 2>(a, p, stream)
                    : launch_kernel<E, 128, false, KVF, 1>(a, p, stream));
  } else {
    e = bal ? (wide ? launch_kernel<E, 64, true, KVF, 2>(a, p, stream)
                    : launch_kernel<E, 64, true, KVF, 1>(a, p, stream))
            : (wide ? launch_kernel<E, 64, false, KVF, 2>(a, p, stream)
                    : launch_kernel<E, 64, false, KVF, 1>(a, p, stream));
  }
  if (e != cudaSuccess || !a.merge) return e;
  const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.num_q_heads;
  return a.head_dim == 128
             ? launch_pdl(decode_combine_kernel<E, 128>, dim3(static_cast<unsigned>(rows)),
                          dim3(kCombineWarps * 32), 0, stream, p)
             : launch_pdl(decode_combine_kernel<E, 64>, dim3(static_cast<unsigned>(rows)),
                          dim3(kCombineWarps * 32), 0, stream, p);
}

}  // namespace dec

// One translation unit per (element type, pool format).
cudaError_t launch_decode_f16(const DecodeArgs &a, const dec::DecodeParams &p, cudaStream_t s);
cudaError_t launch_decode_bf16(const DecodeArgs &a, const dec::DecodeParams &p, cudaStream_t s);
cudaError_t launch_decode_f16_int8(const DecodeArgs &a, const dec::DecodeParams &p,
                                   cudaStream_t s);
cudaError_t launch_decode_bf16_int8(const DecodeArgs &a, const dec::DecodeParams &p,
                                    cudaStream_t s);
cudaError_t launch_decode_f16_fp8(const DecodeArgs &a, const dec::DecodeParams &p,
                                  cudaStream_t s);
cudaError_t launch_decode_bf16_fp8(const DecodeArgs &a, const dec::DecodeParams &p,
                                   cudaStream_t s);

}  // namespace pa
