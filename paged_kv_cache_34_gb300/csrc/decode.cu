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
//  * Work.  A unit is one (sequence, KV head); every piece of work serves
//    all G query heads of its KV head from the same K/V bytes (GQA sharing).
//    Two schedules cut the units into pieces (split-KV):
//      - fixed partitions (a partition size is given): a unit's context is
//        cut into partitions of P tokens, the pages' scheme; worker w of W
//        takes items w, w+W, ... of the (sequence, KV head, partition) list;
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
//    TMA tile loads (128-byte swizzle) guarded by mbarriers: each stage holds
//    16 tokens of K and V for every worker, read block by block through the
//    block table.  Producer lane w walks worker w's items with incremental
//    (block, offset) counters, and the block ids of the worker's next item
//    are copied into shared memory with cp.async while its current item
//    streams, so no id lookup or division sits on the load-issue path.  Two CTAs per SM keep six
//    stages (192 KB) in flight per SM.
//  * Scores are computed transposed on the tensor cores -- S^T[16 tokens x 8
//    heads] = K[16 x D] Q^T[D x 8] with mma.sync m16n8k16, fp32 accumulate --
//    so the G heads fill the N = 8 side.  The online softmax runs on the
//    fragments (warp-shuffle max over tokens), P^T is formed with movmatrix,
//    and O^T[D x 8] += V^T[D x 16] P^T[16 x 8] reads V through ldmatrix.trans.
//    A worker's next query is prefetched into registers one item ahead.
//  * Exponentials are base 2 with the scale pre-multiplied by log2(e).
#include <math.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kWorkers = kDecodeWarps;
constexpr int kThreads = (kWorkers + 1) * 32;  // + producer warp
constexpr uint32_t kTerminate = 0x100u;        // stage header: no more data

// A stage holds, per K and V, `kRegions` regions of kWorkers x kRows rows of
// 128 bytes (128-byte swizzle): 16-bit pools in 64-element halves, 16 rows
// per worker; INT8 pools (head_dim 128) in one region of whole rows, 32 rows
// per worker -- the same bytes per stage, and twice the tokens per softmax
// step for the widening consumer.
template <int D, bool KV8 = false>
struct DecodeSmem {
  static constexpr int kStages = 3;
  static constexpr int kRows = KV8 ? 2 * kDecodeSub : kDecodeSub;  // per worker
  static constexpr int kRegionBytes = kWorkers * kRows * 128;
  static constexpr int kHalves = D / 64;
  static constexpr int kRegions = KV8 ? 1 : kHalves;
  static constexpr int kStageBytes = 2 * kRegions * kRegionBytes;  // K + V
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kHdrOffset = kBarOffset + 2 * kStages * 8;
  static constexpr int kAbortOffset = kHdrOffset + 32;  // after kStages (<= 8) headers
  static constexpr int kVarOffset = kAbortOffset + 16;  // pref[S+1], len[S], ids
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
  int64_t num_blocks;
  float scale_log2;
  int32_t partition_size, num_partitions, max_ids;
  int32_t balanced, chunk_cap, num_workers;  // balanced schedule (see above)
  float *ws_o, *ws_ml;
  int32_t *ws_pref;  // balanced: the prefix sums, for the merge kernel
  const float *k_scale, *v_scale;  // INT8 pools: per-KV-head dequantisation scales
  int32_t after_write;  // launched directly after this step's cache write
  int32_t *err;
};

// One piece of work: tokens [start, end) of KV head g of sequence b (whose
// context is L tokens).  `direct`: the piece is the unit's whole context and
// writes the output; else its softmax state goes to workspace rows
// prow + h * pstride for the unit's query heads h = 0..G-1.
struct Item {
  int b, g, part, L, start, end;
  bool direct;
  int64_t prow;
  int pstride;
};

__host__ __device__ __forceinline__ int ceil16(int x) { return (x + 15) & ~15; }

// Balanced schedule: chunk size (in 16-rounded token-heads) for T token-heads
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

// Item i of the numbering given by the prefix sums `pref` (items of sequence
// b are pref[b] .. pref[b+1]-1, ordered by KV head then partition).
__device__ __forceinline__ Item decode_item(int i, const int *pref, const int *len, int S,
                                            int hkv, int P) {
  int lo = 0, hi = S;  // pref[lo] <= i < pref[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] <= i) lo = mid;
    else hi = mid;
  }
  Item m;
  m.b = lo;
  m.L = len[lo];
  const int np = m.L > 0 ? (m.L + P - 1) / P : 1;
  const int rem = i - pref[lo];
  m.g = rem / np;  // numbered by KV head, then partition
  m.part = rem - m.g * np;
  m.start = m.part * P;
  m.end = min(m.start + P, m.L);
  if (m.end < m.start) m.end = m.start;
  (void)hkv;
  return m;
}

// What every role of a CTA needs to walk the schedule.
struct Sched {
  const int *pref;  // fixed: items before sequence b; balanced: token-heads before b
  const int *len;   // checked context lengths
  int S, hkv, hq, G, P, NP, NW;
  bool balanced;
  int total;      // fixed: items; balanced: token-heads
  int C, chunks;  // balanced: chunk size and count
};
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
__device__ bool next_piece(const Sched &sc, Cursor &cu, Item &m) {
  if (!sc.balanced) {
    if (cu.i >= sc.total) return false;
    m = decode_item(cu.i, sc.pref, sc.len, sc.S, sc.hkv, sc.P);
    cu.i += sc.NW;
    m.direct = (m.L > 0 ? (m.L + sc.P - 1) / sc.P : 1) == 1;
    m.prow = (static_cast<int64_t>(m.b) * sc.hq + m.g * sc.G) * sc.NP + m.part;
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
    // the unit (sequence b, KV head g) holding position x: pref[b] <= x < pref[b+1]
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
    m.prow = (static_cast<int64_t>(lo) * sc.hkv + g + cu.i) * sc.G;
    m.pstride = 1;
    return true;
  }
  return false;
}

__device__ __forceinline__ float shfl_xor(float v, int m) {
  return __shfl_xor_sync(0xffffffffu, v, m);
}

// A pair of query values as the tensor core's operand type: as stored, or
// (TOF16) rounded from bf16 to the nearest fp16 pair.
template <class E, bool TOF16>
__device__ __forceinline__ uint32_t q_pair(uint32_t w) {
  if constexpr (TOF16 && E::kBF16) return F16::pack2(E::lo(w), E::hi(w));
  return w;
}

// The query as the B operand of S^T = K Q^T: lane (head qh = lane / 4,
// t = lane % 4) feeds k-step ks.  16-bit pools: elements 16ks + 2t, +1 and
// 16ks + 2t + 8, +9 (the ldmatrix order of K).  INT8 pools (D = 128, fp16
// operands): elements 32t + 4ks .. 32t + 4ks + 3, the order in which the
// K fragments are widened -- a dot product over D takes any order both
// operands share.
template <class E, int D, bool KV8 = false>
__device__ __forceinline__ void load_q(uint32_t (&qf)[D / 16][2], const DecodeParams &p,
                                       const Item &m, int lane) {
  static_assert(!KV8 || D == 128, "INT8 pools: head_dim 128");
  const int G = p.group;
  const int qh = lane >> 2;  // head column this lane feeds to Q^T
  const typename E::T *qrow = static_cast<const typename E::T *>(p.q) +
                              m.b * p.q_row_stride + (m.g * G + qh) * D +
                              (KV8 ? 32 : 2) * (lane & 3);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int e0 = KV8 ? 4 * ks : 16 * ks, e1 = KV8 ? 4 * ks + 2 : 16 * ks + 8;
    qf[ks][0] =
        qh < G ? q_pair<E, KV8>(__ldg(reinterpret_cast<const uint32_t *>(qrow + e0))) : 0u;
    qf[ks][1] =
        qh < G ? q_pair<E, KV8>(__ldg(reinterpret_cast<const uint32_t *>(qrow + e1))) : 0u;
  }
}

// Widens four 8-bit codes (one word) to two fp16 pairs exactly: lo gets
// bytes 0-1, hi bytes 2-3 (the lower byte in the lower half).  INT8: with the
// sign bit flipped a code is the byte u = c + 128, the fp16 with bits
// 0x6400 | u is 1024 + u, and subtracting 1152 leaves c.  FP8 (E4M3): every
// E4M3 value is an fp16 value; the hardware converts two per instruction.
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

__device__ __forceinline__ void lds128(uint32_t addr, uint32_t (&w)[4]) {
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "r"(addr));
}

// KVF: the pool format -- 0 fp16/bf16 (as E), 1 INT8 codes, 2 FP8 (E4M3) codes.
template <class E, int D, int BOXR, bool BAL, int KVF>
__global__ void __launch_bounds__(kThreads, kDecodeCtasPerSm)
    decode_persistent_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                             const __grid_constant__ CUtensorMap tmv) {
  constexpr bool KV8 = KVF != 0;  // 8-bit codes, widened to fp16
  constexpr bool FP8 = KVF == 2;
  using S = DecodeSmem<D, KV8>;
  using M = std::conditional_t<KV8, F16, E>;  // the tensor cores' operand type
  constexpr int NH = S::kHalves;
  constexpr int NR = S::kRegions;
  constexpr int KSTEPS = D / 16;
  constexpr int NS = S::kStages;
  constexpr int ROWS = S::kRows;       // tokens per worker per stage
  constexpr int RB = S::kRegionBytes;  // one region of a stage
  constexpr int NT = ROWS / 16;        // score tiles per stage
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
  // Inputs come from earlier kernels.  Launched right after this step's
  // cache write (`after_write`), only the K/V rows can be the write's
  // output: the kernel then reads context_lens, block_table and q at once
  // and waits only before its first K/V load (in the producer below).
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
        items = (BAL ? ceil16(L) : (L > 0 ? (L + P - 1) / P : 1)) * p.hkv;
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
  sc.hkv = p.hkv;
  sc.hq = p.hq;
  sc.G = p.group;
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
        ng = m.g;
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
      int rows[ROWS / BOXR];
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
        for (int k = 0; k < ROWS / BOXR; ++k) rows[k] = -1;
        if (act) {
          const int ntok = min(ROWS, endt - cur);
#pragma unroll
          for (int k = 0; k < ROWS / BOXR; ++k) {
            if (k * BOXR >= ntok) break;
            const int id = ids[lblk];
            if (id >= 0 && id < p.num_blocks) {
              rows[k] = id * bs + off;
              ++nb;
            } else {
              bad = true;
            }
            off += BOXR;
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
        ok = mbar_wait_bounded(smem_u32(empty + s), ((c / NS) - 1) & 1);
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
        }
        cp_async_wait_all();
        return;
      }
      const uint32_t bar = smem_u32(full + s);
      if (lane == 0) {
        s_hdr[s] = badmask & ((1u << kWorkers) - 1);
        if (badmask) raise_error(p.err, PA_DEVERR_BLOCK_ID);
        // The barrier must expect exactly the bytes that land.
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nbox) * BOXR * 128 * NR * 2);
      }
      __syncwarp();
      if (feeder) {
        const uint32_t kdst = smem_u32(smem + s * S::kStageBytes);
        const uint32_t vdst = kdst + NR * RB;
#pragma unroll
        for (int k = 0; k < ROWS / BOXR; ++k) {
          if (rows[k] < 0) continue;
          const uint32_t o = (lane * ROWS + k * BOXR) * 128;
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
  const int G = p.group;
  float sl = p.scale_log2;  // INT8 pools: times the piece's K scale
  float vsc = 1.f;          // INT8 pools: the piece's V scale
  const int r0 = warp * ROWS;  // this worker's rows in a stage
  const int mj = lane >> 3, mr = lane & 7;
  const int h0 = 2 * (lane & 3), h1 = h0 + 1;

  uint32_t qf[KSTEPS][2], qn[KSTEPS][2];
  float o[KSTEPS][4];
  float m0, m1, l0, l1;
  bool item_bad = false;
  Item cur_item;
  Cursor wc = first_cursor(sc, blockIdx.x * kWorkers + warp);
  int qn_b = -1, qn_g = -1;  // the unit whose query qn holds
  int cur = 0;
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
#pragma unroll
    for (int s = 4; s < 32; s <<= 1) {
      l0 += shfl_xor(l0, s);
      l1 += shfl_xor(l1, s);
    }
    if constexpr (KV8) {
      // O^T rows in the INT8 order: lane (g, t) holds elements 16g .. 16g + 15
      // of heads 2t and 2t + 1, element 16g + i in o[i / 2][i % 2 ? 2 : 0]
      // (head 2t) and o[i / 2][i % 2 ? 3 : 1] (head 2t + 1).
      const int e0 = 16 * (lane >> 2);
      if (m.direct) {
        typename E::T *out =
            static_cast<typename E::T *>(p.out) + m.b * p.out_row_stride + m.g * G * D + e0;
        const float i0 = (!bad_item && l0 > 0.f) ? vsc / l0 : 0.f;
        const float i1 = (!bad_item && l1 > 0.f) ? vsc / l1 : 0.f;
        uint32_t u0[8], u1[8];
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt) {
          u0[mt] = E::pack2(o[mt][0] * i0, o[mt][2] * i0);
          u1[mt] = E::pack2(o[mt][1] * i1, o[mt][3] * i1);
        }
        if (h0 < G) {
          uint4 *d0 = reinterpret_cast<uint4 *>(out + h0 * D);
          d0[0] = make_uint4(u0[0], u0[1], u0[2], u0[3]);
          d0[1] = make_uint4(u0[4], u0[5], u0[6], u0[7]);
        }
        if (h1 < G) {
          uint4 *d1 = reinterpret_cast<uint4 *>(out + h1 * D);
          d1[0] = make_uint4(u1[0], u1[1], u1[2], u1[3]);
          d1[1] = make_uint4(u1[4], u1[5], u1[6], u1[7]);
        }
      } else {
        const float f = bad_item ? 0.f : vsc;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int h = h0 + hh;
          if (h >= G) continue;
          float4 *w = reinterpret_cast<float4 *>(p.ws_o + (m.prow + h * m.pstride) * D + e0);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            w[q] = make_float4(o[2 * q][hh] * f, o[2 * q][hh + 2] * f, o[2 * q + 1][hh] * f,
                               o[2 * q + 1][hh + 2] * f);
        }
        if (lane < 4) {
          if (h0 < G) {
            p.ws_ml[(m.prow + h0 * m.pstride) * 2 + 0] = bad_item ? -INFINITY : m0;
            p.ws_ml[(m.prow + h0 * m.pstride) * 2 + 1] = bad_item ? 0.f : l0;
          }
          if (h1 < G) {
            p.ws_ml[(m.prow + h1 * m.pstride) * 2 + 0] = bad_item ? -INFINITY : m1;
            p.ws_ml[(m.prow + h1 * m.pstride) * 2 + 1] = bad_item ? 0.f : l1;
          }
        }
      }
      return;
    }
    if (m.direct) {
      const float i0 = (!bad_item && l0 > 0.f) ? 1.f / l0 : 0.f;
      const float i1 = (!bad_item && l1 > 0.f) ? 1.f / l1 : 0.f;
      typename E::T *out =
          static_cast<typename E::T *>(p.out) + m.b * p.out_row_stride + m.g * G * D;
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt) {
        const int d0 = mt * 16 + (lane >> 2), d1 = d0 + 8;
        if (h0 < G) {
          out[h0 * D + d0] = E::from_float(o[mt][0] * i0);
          out[h0 * D + d1] = E::from_float(o[mt][2] * i0);
        }
        if (h1 < G) {
          out[h1 * D + d0] = E::from_float(o[mt][1] * i1);
          out[h1 * D + d1] = E::from_float(o[mt][3] * i1);
        }
      }
    } else {
      const int64_t row0 = m.prow;
      const int64_t hstride = m.pstride;
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt) {
        const int d0 = mt * 16 + (lane >> 2), d1 = d0 + 8;
        if (h0 < G) {
          float *w0 = p.ws_o + (row0 + h0 * hstride) * D;
          w0[d0] = bad_item ? 0.f : o[mt][0];
          w0[d1] = bad_item ? 0.f : o[mt][2];
        }
        if (h1 < G) {
          float *w1 = p.ws_o + (row0 + h1 * hstride) * D;
          w1[d0] = bad_item ? 0.f : o[mt][1];
          w1[d1] = bad_item ? 0.f : o[mt][3];
        }
      }
      if (lane < 4) {
        if (h0 < G) {
          p.ws_ml[(row0 + h0 * hstride) * 2 + 0] = bad_item ? -INFINITY : m0;
          p.ws_ml[(row0 + h0 * hstride) * 2 + 1] = bad_item ? 0.f : l0;
        }
        if (h1 < G) {
          p.ws_ml[(row0 + h1 * hstride) * 2 + 0] = bad_item ? -INFINITY : m1;
          p.ws_ml[(row0 + h1 * hstride) * 2 + 1] = bad_item ? 0.f : l1;
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
      for (int mt = 0; mt < KSTEPS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
      item_bad = false;
      if (m.end > m.start) {
        if (qn_b == m.b && qn_g == m.g) {
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks) {
            qf[ks][0] = qn[ks][0];
            qf[ks][1] = qn[ks][1];
          }
        } else {
          load_q<E, D, KV8>(qf, p, m, lane);
        }
        cur_item = m;
        cur = m.start;
        if constexpr (KV8) {
          // The piece's KV head's scales: K's scales the scores, V's the
          // output.  One that is not a positive finite number makes the
          // piece contribute nothing (zeros / an empty softmax state).
          const float ks = __ldg(p.k_scale + m.g), vs = __ldg(p.v_scale + m.g);
          const float big = 3.4028234663852886e38f;
          sl = p.scale_log2 * ks;
          vsc = vs;
          if (!(ks > 0.f && ks <= big && vs > 0.f && vs <= big)) {
            item_bad = true;
            if (lane == 0) raise_error(p.err, PA_DEVERR_SCALE);
          }
        }
        // Prefetch the next piece's query one piece ahead.
        Cursor peek = wc;
        Item nm;
        qn_b = qn_g = -1;
        while (next_piece(sc, peek, nm)) {
          if (nm.end <= nm.start) continue;
          load_q<E, D, KV8>(qn, p, nm, lane);
          qn_b = nm.b;
          qn_g = nm.g;
          break;
        }
        return true;
      }
      if constexpr (!BAL) finalize(m, false);  // empty sequence: zeros
    }
    return false;
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
    if (!mbar_wait_bounded(smem_u32(full + s), (c / NS) & 1)) {
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
      float sc[NT][4];
#pragma unroll
      for (int u = 0; u < NT; ++u) sc[u][0] = sc[u][1] = sc[u][2] = sc[u][3] = 0.f;
      bool zeroed = false;
      uint32_t vw[NT][4][4];  // INT8: this lane's V codes (see below)
      if constexpr (KV8) {
        // This worker's 32 int8 K and V rows (two 16-token tiles u) go
        // straight to registers, and the stage is handed back once they are
        // read.  Codes widen to exact fp16 whatever the pool held, so
        // rows past the context need no clearing: their weight is zero.
        //  K, the A operand of S^T = K Q^T (rows: tokens 16u + g, +8): k-step
        //   ks of lane (g, t) is elements 32t + 4ks .. +3 of its rows
        //   (16-byte chunks 2t and 2t + 1), the query following suit.
        //  V, the A operand of O^T += V^T P^T (rows: elements of D;
        //   columns: tokens 16u + 2t, +1, +8, +9): the D order of O^T is
        //   free as well, so lane (g, t) owns elements 16g .. 16g + 15
        //   (chunk g of its token rows), row g of M-tile mt holding element
        //   16g + 2mt and row g + 8 element 16g + 2mt + 1.
        // 128-byte swizzle: chunk c of row r sits at chunk c ^ (r & 7).
        const int g8 = lane >> 2, t4 = lane & 3;
        const uint32_t kr = smem_u32(kst) + r0 * 128;
        const uint32_t vr = kr + RB;
        uint32_t kw[NT][2][2][4];  // [tile][row g | g + 8][chunk 2t | 2t + 1][word]
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
          for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int c = 0; c < 2; ++c)
              lds128(kr + (16 * u + g8 + 8 * r) * 128 + (((2 * t4 + c) ^ g8) << 4), kw[u][r][c]);
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks)
#pragma unroll
          for (int u = 0; u < NT; ++u) {
            uint32_t a0, a1, a2, a3;
            widen4<FP8>(kw[u][0][ks >> 2][ks & 3], a0, a2);
            widen4<FP8>(kw[u][1][ks >> 2][ks & 3], a1, a3);
            mma_16816<false>(sc[u], a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
          }
        // V's codes once K's are spent (fewer live registers); their loads
        // overlap the softmax below.
        const int v0 = 2 * t4;
#pragma unroll
        for (int u = 0; u < NT; ++u) {
          const uint32_t vu = vr + 16 * u * 128;
          lds128(vu + v0 * 128 + ((g8 ^ v0) << 4), vw[u][0]);
          lds128(vu + (v0 + 1) * 128 + ((g8 ^ (v0 + 1)) << 4), vw[u][1]);
          lds128(vu + (v0 + 8) * 128 + ((g8 ^ v0) << 4), vw[u][2]);
          lds128(vu + (v0 + 9) * 128 + ((g8 ^ (v0 + 1)) << 4), vw[u][3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(empty + s));
        released = true;
        if constexpr (FP8) {
          // An E4M3 byte can be a NaN code: V rows past the context (stale or
          // unwritten) become exact zeros.  K's are masked out of the scores.
          if (j0 + ROWS > end) {
#pragma unroll
            for (int u = 0; u < NT; ++u)
#pragma unroll
              for (int i = 0; i < 4; ++i)
                if (j0 + 16 * u + v0 + (i & 1) + 8 * (i >> 1) >= end)
                  vw[u][i][0] = vw[u][i][1] = vw[u][i][2] = vw[u][i][3] = 0u;
          }
        }
      } else {
        const uint32_t kb = smem_u32(kst);
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
          zeroed = true;
        }
        // S^T = K Q^T for this worker's 16 tokens.
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
          const int row = r0 + (mj & 1) * 8 + mr;
          const int c16 = ks * 2 + (mj >> 1);
          const uint32_t addr =
              kb + (c16 >> 3) * RB + row * 128 + (((c16 & 7) ^ (row & 7)) << 4);
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4(addr, a0, a1, a2, a3);
          mma_16816<E::kBF16>(sc[0], a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
        }
      }
      // Scores of tile u: tokens j0 + 16u + g (sc[u][0..1], heads 2t, 2t + 1)
      // and j0 + 16u + g + 8 (sc[u][2..3]).
      float sv[NT][4];
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int u = 0; u < NT; ++u) {
        const int t0 = j0 + 16 * u + (lane >> 2), t1 = t0 + 8;
        sv[u][0] = t0 < end ? sc[u][0] * sl : -INFINITY;
        sv[u][1] = t0 < end ? sc[u][1] * sl : -INFINITY;
        sv[u][2] = t1 < end ? sc[u][2] * sl : -INFINITY;
        sv[u][3] = t1 < end ? sc[u][3] * sl : -INFINITY;
        mx0 = fmaxf(mx0, fmaxf(sv[u][0], sv[u][2]));
        mx1 = fmaxf(mx1, fmaxf(sv[u][1], sv[u][3]));
      }
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
      uint32_t pw[NT][2];
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int u = 0; u < NT; ++u) {
        pw[u][0] = M::pack2(exp2f(sv[u][0] - mn0), exp2f(sv[u][1] - mn1));  // token t0
        pw[u][1] = M::pack2(exp2f(sv[u][2] - mn0), exp2f(sv[u][3] - mn1));  // token t1
        ls0 += M::lo(pw[u][0]) + M::lo(pw[u][1]);
        ls1 += M::hi(pw[u][0]) + M::hi(pw[u][1]);
      }
      l0 = l0 * cr0 + ls0;
      l1 = l1 * cr1 + ls1;
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt) {
        o[mt][0] *= cr0;
        o[mt][1] *= cr1;
        o[mt][2] *= cr0;
        o[mt][3] *= cr1;
      }
      // P^T fragments (tokens x heads) from the S^T accumulator layout.
      uint32_t pb[NT][2];
#pragma unroll
      for (int u = 0; u < NT; ++u) {
        pb[u][0] = movmatrix_trans(pw[u][0]);
        pb[u][1] = movmatrix_trans(pw[u][1]);
      }
      // O^T += V^T P^T, one 16-wide slice of D at a time.
      if constexpr (KV8) {
        // Word w of the token rows: M-tiles 2w and 2w + 1.
#pragma unroll
        for (int w = 0; w < 4; ++w)
#pragma unroll
          for (int u = 0; u < NT; ++u) {
            uint32_t a0, a1, b0, b1, a2, a3, b2, b3;
            widen_tokens<FP8>(vw[u][0][w], vw[u][1][w], a0, a1, b0, b1);  // tokens 2t, 2t + 1
            widen_tokens<FP8>(vw[u][2][w], vw[u][3][w], a2, a3, b2, b3);  // tokens 2t + 8, + 9
            mma_16816<false>(o[2 * w], a0, a1, a2, a3, pb[u][0], pb[u][1]);
            mma_16816<false>(o[2 * w + 1], b0, b1, b2, b3, pb[u][0], pb[u][1]);
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
          mma_16816<E::kBF16>(o[mt], a0, a1, a2, a3, pb[0][0], pb[0][1]);
        }
      }
      if (zeroed) fence_proxy_async_smem();  // generic writes before the next TMA
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
// rows (u + c) * G + h).
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
            p.hkv;
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
      const int G = p.group, g = h / G;
      const int C = balanced_chunk(total, p.num_workers, p.chunk_cap);
      const int U = pref_b + g * ceil16(L);  // the unit's first position
      const int c0 = U / C, c1 = (U + L - 1) / C;
      n = c1 - c0 + 1;
      row0 = (static_cast<int64_t>(b) * p.hkv + g + c0) * G + (h - g * G);
      rstride = G;
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

template <class E, int D, int BOXR, bool BAL, int KVF>
cudaError_t launch_kernel(const DecodeArgs &a, const DecodeParams &p, cudaStream_t stream) {
  using S = DecodeSmem<D, KVF != 0>;
  const int smem = S::bytes(a.num_seqs, p.max_ids);
  auto kernel = decode_persistent_kernel<E, D, BOXR, BAL, KVF>;
  cudaError_t e = allow_dynamic_smem<decode_persistent_kernel<E, D, BOXR, BAL, KVF>>();
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, dim3(static_cast<unsigned>(a.grid)), dim3(kThreads), smem, stream,
                    p, a.tm_k, a.tm_v);
}

template <class E, int D, int BOXR, int KVF>
cudaError_t launch_typed(const DecodeArgs &a, const DecodeParams &p, cudaStream_t stream) {
  const cudaError_t e = p.balanced ? launch_kernel<E, D, BOXR, true, KVF>(a, p, stream)
                                   : launch_kernel<E, D, BOXR, false, KVF>(a, p, stream);
  if (e != cudaSuccess || !a.merge) return e;
  const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.num_q_heads;
  return launch_pdl(decode_combine_kernel<E, D>, dim3(static_cast<unsigned>(rows)),
                    dim3(kCombineWarps * 32), 0, stream, p);
}

template <class E, int D, int KVF = 0>
cudaError_t launch_box(const DecodeArgs &a, const DecodeParams &p, cudaStream_t stream) {
  switch (a.box_rows) {
    case 8: return launch_typed<E, D, 8, KVF>(a, p, stream);
    case 16: return launch_typed<E, D, 16, KVF>(a, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// Largest dynamic shared memory the decode kernel needs for this shape, so
// the host can reject shapes that cannot launch.
size_t decode_smem_bytes(int head_dim, int num_seqs, int partition_size, int block_size,
                         bool kv_int8) {
  const int max_ids = (partition_size > 0 ? partition_size : kDecodeChunkCap) / block_size + 2;
  if (kv_int8) return DecodeSmem<128, true>::bytes(num_seqs, max_ids);
  return head_dim == 128 ? DecodeSmem<128>::bytes(num_seqs, max_ids)
                         : DecodeSmem<64>::bytes(num_seqs, max_ids);
}

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
  p.num_seqs = a.num_seqs;
  p.hq = a.num_q_heads;
  p.hkv = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.scale_log2 = a.scale_log2;
  p.partition_size = a.partition_size;
  p.num_partitions = a.num_partitions;
  p.balanced = a.partition_size == 0;
  p.chunk_cap = kDecodeChunkCap;
  p.num_workers = a.grid * kWorkers;
  p.max_ids = (p.balanced ? kDecodeChunkCap : a.partition_size) / a.block_size + 2;
  p.ws_o = a.ws_o;
  p.ws_ml = a.ws_ml;
  p.ws_pref = a.ws_pref;
  p.after_write = a.after_write ? 1 : 0;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.err = a.d_error;
  const bool bf = a.dtype == PA_BF16;
  if (a.head_dim == 128 && a.kv_int8 && a.kv_fp8)
    return bf ? launch_box<BF16, 128, 2>(a, p, stream) : launch_box<F16, 128, 2>(a, p, stream);
  if (a.head_dim == 128 && a.kv_int8)
    return bf ? launch_box<BF16, 128, 1>(a, p, stream) : launch_box<F16, 128, 1>(a, p, stream);
  if (a.head_dim == 128)
    return bf ? launch_box<BF16, 128>(a, p, stream) : launch_box<F16, 128>(a, p, stream);
  if (a.head_dim == 64)
    return bf ? launch_box<BF16, 64>(a, p, stream) : launch_box<F16, 64>(a, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
