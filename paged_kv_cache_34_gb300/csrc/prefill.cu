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
// here nothing is masked outside the diagonal tiles and nothing is padded):
//  * Work item = (two consecutive 128-row query tiles A and B of one
//    sequence, head unit).  Both tiles share every K/V tile loaded, halving
//    the K/V traffic per flop.  A head unit is one query head, or, when the
//    GQA group is a power of two, all the query heads of one KV head: a tile
//    row is then a (token, head) pair, so the group shares every K/V tile
//    too.  One persistent CTA per SM claims items one
//    at a time from a global counter, in an order that keeps one or two
//    sequences in flight across the GPU (so each sequence's K/V comes from
//    HBM once and is then reused from L2) and runs the heaviest items of a
//    sequence first (so the last items claimed, which set the finish time,
//    are light).
//  * Warp 12 (TMA): loads Q_A and Q_B once, then streams K and V tiles (128
//    tokens each) through separate K (2 buffers) and V (3 buffers) rings,
//    K running one tile ahead of V; a K/V
//    tile is gathered block by block through block_table, one TMA box per
//    block issued by its own lane, with the 128-byte swizzle the MMA
//    descriptors expect.  The next tile's block ids are loaded while the
//    current tile is issued.
//  * Warp 13 (MMA; one elected lane issues): tcgen05.mma kind::f16, M = 128,
//    N = 128, K = 16 x 8: S_t = Q_t K^T into TMEM and O_t += P_t V (V read
//    MN-major straight from its TMA tile, P from TMEM).  The issue order S_A S_B | PV_A S_A' | PV_B
//    S_B' | ... keeps the tensor core busy with one tile while the other
//    tile's softmax runs (ping-pong); the tensor core executes one thread's
//    MMAs in order, so S_t' may overwrite the columns P_t was read from.
//  * Warps 0-3 / 4-7: the softmax of tile A / B, one thread per query row
//    (= TMEM lane): S from TMEM, masks only where a tile crosses the causal
//    edge or the context end, base-2 exponentials on the SFU, P rounded to
//    the input type and written back into TMEM over S.  The running max
//    is only raised -- and O in TMEM rescaled -- when a row's max grows by
//    more than 2^8, which keeps every P <= 256 and the result exact up to
//    rounding.
//  * Epilogue: O / l from TMEM to registers to global memory.
#include <math.h>

#include <atomic>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {

namespace {

// Warpgroups: 0 softmax of tile A, 1 softmax of tile B, 2 epilogue of both
// tiles, 3 producers: warp 12 TMA, 13 MMA, 14-15 idle (setmaxnreg works on
// whole warpgroups).
constexpr int kThreads = 512;
constexpr int kEpiWarp0 = 8, kTmaWarp = 12, kMmaWarp = 13;
// Registers per thread after the split (setmaxnreg, per warpgroup): the
// softmax holds a whole S row per thread, the epilogue a packed O row, the
// producers little.  The split must fit in what the CTA is launched with
// (checked on the host before the first launch).
constexpr int kSoftmaxRegs = 152, kEpilogueRegs = 104, kProducerRegs = 104;
constexpr int kRegPoolNeeded = 128 * (2 * kSoftmaxRegs + kEpilogueRegs + kProducerRegs);
constexpr int kHalf = 128 * 128;    // 128 rows x 64 elements x 2 B
constexpr int kTile = 2 * kHalf;    // 128 x 128 tile, two 64-wide halves
constexpr int kKBufs = 2;  // separate K and V rings (5 buffers)
constexpr int kVBufs = 5 - kKBufs;
constexpr int kKVBufs = kKBufs + kVBufs;
constexpr int kQOff = 0;                           // Q_A, Q_B
constexpr int kKVOff = 2 * kTile;                  // K/V ring
constexpr int kBarOff = kKVOff + kKVBufs * kTile;
enum {
  kQFull = 0,
  kKVFull = 1,
  kKVEmpty = kKVFull + kKVBufs,
  kSFull = kKVEmpty + kKVBufs,
  kPFull = kSFull + 2,
  kQEmpty = kPFull + 2,
  kOFull = kQEmpty + 1,     // per query tile and item: its last PV is done
  kOFree = kOFull + 2,      // per query tile: the epilogue has read O
  kLFull = kOFree + 2,      // per query tile: the softmax has left its row sums
  kVFixed = kLFull + 2,     // the TMA warp has cleared a V tile's tail rows
  kVFixFree = kVFixed + 1,  // ... and the MMA thread has seen it
  kFin = kVFixFree + 1,
  kItemFull = kFin + 1,     // item ring: index published by the TMA warp
  kItemEmpty = kItemFull + 4,  // ... and taken by every other role
  kNumBars = kItemEmpty + 4
};
constexpr int kItemRing = 4;
constexpr int kItemTakers = 13;  // 8 softmax warps, 4 epilogue warps, MMA
constexpr int kLOff = kBarOff + kNumBars * 8;   // float l[2][128]: row sums per tile
constexpr int kMiscOff = kLOff + 2 * 128 * 4;   // ints: [2] TMEM base, [3] abort, [8..11] items
constexpr int kItemWords = 16;                  // one decoded work item (PairItem fields)
constexpr int kItemOff = kMiscOff + 64;         // the decoded items of the ring
constexpr int kSmemBytes = 1024 + kItemOff + kItemRing * kItemWords * 4;
static_assert(kSmemBytes <= 227 * 1024, "prefill shared memory");
constexpr uint32_t kTmemCols = 512;         // S_A | S_B | O_A | O_B (P_t overlays S_t)
constexpr float kRescaleThreshold = 8.0f;   // log2 of the largest P allowed


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
  // Query heads packed into one tile's rows: a tile row is (token, head) =
  // (row >> pg_log2, first head + (row & (pg - 1))), so the pg heads of one
  // KV head share every K/V tile an item loads; hu = hq / pg head units.
  int32_t pg, pg_log2, hu;
  int64_t num_blocks;
  float scale_log2;
  int32_t causal;
  int32_t num_items;
  int32_t sched_slot;
  int32_t *err;
  uint64_t wait_ns;  // bound of a pipeline wait
};

// Work counters for the dynamic item schedule.  A launch uses one slot
// (chosen on the host, round robin): `next` hands out item indices, `done`
// counts CTAs that have finished, and the last CTA to finish puts both back
// to zero, so the slot is ready for the next launch that is ordered after
// this one.  Launches that may run at the same time must use different
// slots; with round-robin choice that fails only when more than kSchedSlots
// prefill launches are in flight at once.
struct __align__(128) SchedSlot {
  unsigned next, done;
};
constexpr int kSchedSlots = 256;
__device__ SchedSlot g_prefill_sched[kSchedSlots];

// Item x of the work list: items are ordered by sequence, then pair of query
// tiles (latest, i.e. heaviest, pair first), then head unit (pg query heads
// of one KV head, packed into the tiles' rows).  The items of one sequence
// are neighbours, so they run at about the same time and share that
// sequence's K/V tiles in L2; head units of one KV group are neighbours too.
// Warp-collective.
__device__ void find_item(const PrefillParams &p, int x, int lane, int *seq_out, int *pair_out,
                          int *head_out) {
  int base = 0;  // items of the sequences before this chunk
  for (int c0 = 0; c0 < p.num_seqs; c0 += 32) {
    const int s = c0 + lane;
    int cnt = 0;
    if (s < p.num_seqs) {
      const int q = __ldg(p.cu + s + 1) - __ldg(p.cu + s);
      if (q > 0 && q <= p.max_seqlen_q) cnt = (((q << p.pg_log2) + 255) / 256) * p.hu;
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, x < base + incl && x >= base + incl - cnt);
    if (hit) {
      const int src = __ffs(hit) - 1;
      const int cs = __shfl_sync(0xffffffffu, cnt, src);
      const int first = base + __shfl_sync(0xffffffffu, incl, src) - cs;
      const int npairs = cs / p.hu;
      const int rem = x - first;
      *seq_out = c0 + src;
      *pair_out = npairs - 1 - rem / p.hu;
      *head_out = rem % p.hu;
      return;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  *seq_out = -1;
  *pair_out = -1;
  *head_out = 0;
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

// Ring slots: K of tile kt in slot kt % 2, V of tile kt in slot 2 + kt % 3;
// the parity is that of the slot's use count.
__device__ __forceinline__ int k_slot(int kt) { return kt % kKBufs; }
__device__ __forceinline__ uint32_t k_par(int kt) { return (kt / kKBufs) & 1; }
__device__ __forceinline__ int v_slot(int kt) { return kKBufs + kt % kVBufs; }
__device__ __forceinline__ uint32_t v_par(int kt) { return (kt / kVBufs) & 1; }

// One work item: a (sequence, pair of query tiles, head unit), with the
// geometry every role derives from it.  Rows are packed (token, head) rows:
// row0[t] is tile t's first, the sequence has q_len << pg_log2 of them.
struct PairItem {
  int seq, h, q_start, q_len, L, lim_base;
  int row0[2], nkv_t[2], nkv;
  bool has_b;
};

// A decoded item in shared memory (the item ring), field by field.
__device__ __forceinline__ void store_item(volatile int *w, const PairItem &it) {
  w[0] = it.seq;
  w[1] = it.h;
  w[2] = it.q_start;
  w[3] = it.q_len;
  w[4] = it.L;
  w[5] = it.lim_base;
  w[6] = it.row0[0];
  w[7] = it.row0[1];
  w[8] = it.nkv_t[0];
  w[9] = it.nkv_t[1];
  w[10] = it.nkv;
  w[11] = it.has_b ? 1 : 0;
}
__device__ __forceinline__ PairItem load_item(const volatile int *w) {
  PairItem it;
  it.seq = w[0];
  it.h = w[1];
  it.q_start = w[2];
  it.q_len = w[3];
  it.L = w[4];
  it.lim_base = w[5];
  it.row0[0] = w[6];
  it.row0[1] = w[7];
  it.nkv_t[0] = w[8];
  it.nkv_t[1] = w[9];
  it.nkv = w[10];
  it.has_b = w[11] != 0;
  return it;
}

// Item x of the work list (see find_item).  Warp-collective.
__device__ PairItem item_at(const PrefillParams &p, int x, int lane, bool report) {
  PairItem it;
  int seq, pair, head;
  find_item(p, x, lane, &seq, &pair, &head);
  it.seq = seq;
  it.h = head;
  it.q_start = it.q_len = it.L = it.lim_base = 0;
  it.row0[0] = it.row0[1] = 0;
  it.nkv_t[0] = it.nkv_t[1] = 0;
  if (seq >= 0) {
    it.q_start = __ldg(p.cu + seq);
    it.q_len = __ldg(p.cu + seq + 1) - it.q_start;
    it.L = checked_context_len(__ldg(p.ctx + seq), p.capacity, p.max_ctx, p.err,
                               report && lane == 0 && it.h == 0 && pair == 0);
    it.lim_base = p.causal ? it.L - it.q_len : 0x3fffffff;  // row i sees keys <= lim_base + i
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      it.row0[t] = pair * 256 + t * 128;
      if (it.row0[t] < (it.q_len << p.pg_log2)) {
        // keys up to those of the tile's last token
        int kv_end = it.L;
        if (p.causal)
          kv_end = min(it.L, it.L - it.q_len + ((it.row0[t] + 127) >> p.pg_log2) + 1);
        if (kv_end < 0) kv_end = 0;
        it.nkv_t[t] = (kv_end + 127) / 128;
      }
    }
  }
  it.nkv = max(it.nkv_t[0], it.nkv_t[1]);
  it.has_b = seq >= 0 && it.row0[1] < (it.q_len << p.pg_log2);
  return it;
}

// D (head_dim) is 64 or 128: a Q, K or V tile row is D / 64 128-byte
// halves; the shared-memory layout is the D = 128 one either way.  SPEC:
// the softmax for launches whose query tiles come one per item (see below).
template <class E, int D, bool SPEC>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmq,
                   const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kBarOff);
  float *l_buf = reinterpret_cast<float *>(smem + kLOff);
  volatile int *misc = reinterpret_cast<volatile int *>(smem + kMiscOff);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  constexpr int kHalves = D / 64;  // 128-byte halves per tile row
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  griddep_wait();  // inputs (e.g. this step's cache write) come from earlier kernels
  griddep_launch_dependents();
  SchedSlot *sched = &g_prefill_sched[p.sched_slot];
  // Item j of this CTA: index published by the TMA warp in ring entry j % 4;
  // every other role takes it from there (lane 0 waits, the warp shares it).
  // Returns false when a wait gave up; *x < 0 ends the list.
  // Item j of the ring: its index (-1: end of the list) and, decoded by
  // the TMA warp that claimed it, its parameters.  Warp-collective.
  volatile int *s_items = reinterpret_cast<volatile int *>(smem + kItemOff);
  auto take_item = [&](int j, int *x, PairItem *it) {
    const int slot = j % kItemRing;
    bool ok = true;
    if (lane == 0)
      ok = mbar_wait_bounded(bar(kItemFull + slot), (j / kItemRing) & 1, p.wait_ns);
    __syncwarp();
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    int v = -1;
    if (ok) {
      v = misc[8 + slot];
      if (v >= 0) *it = load_item(s_items + slot * kItemWords);
    }
    __syncwarp();  // every lane has read the slot
    if (lane == 0) mbar_arrive(bar(kItemEmpty + slot));
    *x = v;
    return ok;
  };
  // Lane 0 waits, the warp learns the outcome.
  auto warp_wait = [&](uint32_t b, uint32_t parity) {
    bool ok = true;
    if (lane == 0) ok = mbar_wait_bounded(b, parity, p.wait_ns);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  };

  if (warp == 0) {
    if (lane == 0) misc[3] = 0;  // abort: some wait gave up
    if (blockIdx.x == 0) check_cu_seqlens(p, lane);
  }
  if (warp == 1 && lane == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t n = 1;
      // one arrival per softmax warp (P) or epilogue warp (O free) of a tile;
      // the row sums are left by every softmax thread
      if (i == kPFull || i == kPFull + 1 || i == kOFree || i == kOFree + 1) n = 4;
      if (i == kLFull || i == kLFull + 1) n = 128;
      if (i >= kItemEmpty && i < kItemEmpty + kItemRing) n = kItemTakers;
      mbar_init(bar(i), n);
    }
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(const_cast<int *>(misc + 2)), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = static_cast<uint32_t>(misc[2]);

  if (warp >= kTmaWarp) {
    reg_dealloc<kProducerRegs>();
    if (warp == kTmaWarp) {
      // ----------------------------------------------------------- TMA --
      if (lane == 0) {
        tma_prefetch_desc(&tmq);
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
      }
      const int bs = p.block_size;
      const int nbox = 128 / bs;  // one box per block, lane k loads block k of a tile
      int kbase = 0;              // K/V tiles of earlier items (ring positions)
      bool ok = true;
      int nk = 0, nv = 0;         // K and V tiles issued in all
      int nq = 0;                 // items whose Q loads were issued
      int nfix = 0;               // V tiles whose tail rows were cleared
      int j = 0;
      int x = blockIdx.x;         // the first item is fixed, the rest are claimed
      for (;; ++j) {
        PairItem it;
        it.seq = -1;
        if (x < p.num_items) it = item_at(p, x, lane, true);
        // Publish the item (or the end of the list) to the other roles.
        if (lane == 0) {
          if (j >= kItemRing)
            ok = mbar_wait_bounded(bar(kItemEmpty + j % kItemRing), ((j / kItemRing) - 1) & 1,
                                   p.wait_ns);
          if (it.seq >= 0 && ok) store_item(s_items + (j % kItemRing) * kItemWords, it);
          misc[8 + j % kItemRing] = it.seq >= 0 && ok ? x : -1;
          mbar_arrive(bar(kItemFull + j % kItemRing));
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok || it.seq < 0) break;
        // Claim the next item now; the answer is first needed next iteration.
        int x_next = 0;
        if (lane == 0) x_next = static_cast<int>(atomicAdd(&sched->next, 1u)) + gridDim.x;
        const int g = (it.h << p.pg_log2) / p.group;
        // Q of item j once the previous item's last QK has read Q.
        if (j > 0) ok = warp_wait(bar(kQEmpty), (j - 1) & 1);
        if (!ok || misc[3]) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t qs = smem_u32(smem + kQOff);
          const int qtiles = it.nkv > 0 ? (it.has_b ? 2 : 1) : 0;
          mbar_arrive_expect_tx(bar(kQFull), qtiles * kHalves * kHalf);
          for (int t = 0; t < qtiles; ++t) {
            // a box of 128 / pg tokens x pg heads: rows in (token, head) order
            const int h0 = it.h << p.pg_log2, tok = it.q_start + (it.row0[t] >> p.pg_log2);
            tma_load_3d(qs + t * kTile, &tmq, bar(kQFull), 0, h0, tok);
            if (kHalves == 2) tma_load_3d(qs + t * kTile + kHalf, &tmq, bar(kQFull), 64, h0, tok);
          }
        }
        ++nq;
        const int32_t *bt = p.block_table + static_cast<int64_t>(it.seq) * p.bt_stride;
        auto load_id = [&](int kt) {
          return (lane < nbox && kt < it.nkv && kt * 128 + lane * bs < it.L)
                     ? __ldg(bt + kt * nbox + lane)
                     : -1;
        };
        // Issue order K0 K1 V0 K2 V1 ...: K runs one tile ahead of V, since S
        // needs K a whole softmax earlier than O needs V.
        int id_k = load_id(0), id_v = -1;
        for (int jj = 0; jj <= it.nkv && ok; ++jj) {
          const int id_nxt = load_id(jj + 1);  // in flight while this step issues
#pragma unroll
          for (int which = 0; which < 2; ++which) {
            const int kt = which == 0 ? jj : jj - 1;  // K of tile jj, then V of tile jj-1
            if (kt < 0 || kt >= it.nkv) continue;
            const int id = which == 0 ? id_k : id_v;
            const bool want = lane < nbox && kt * 128 + lane * bs < it.L;
            const bool valid = want && id >= 0 && id < p.num_blocks;
            if (which == 0 && want && !valid) raise_error(p.err, PA_DEVERR_BLOCK_ID);
            const unsigned vmask = __ballot_sync(0xffffffffu, valid);
            const int n = kbase + kt;  // ring position
            const int slot = which == 0 ? k_slot(n) : v_slot(n);
            const int nuse = which == 0 ? n / kKBufs : n / kVBufs;  // earlier uses of slot
            if (nuse > 0) ok = warp_wait(bar(kKVEmpty + slot), (nuse - 1) & 1);
            if (!ok || misc[3]) {
              ok = false;
              break;
            }
            if (lane == 0)
              mbar_arrive_expect_tx(bar(kKVFull + slot),
                                    static_cast<uint32_t>(__popc(vmask)) * bs * D * 2);
            __syncwarp();
            if (valid) {
              const uint32_t dst = smem_u32(smem + kKVOff + slot * kTile) + lane * bs * 128;
              const CUtensorMap *map = which == 0 ? &tmk : &tmv;
              tma_load_3d(dst, map, bar(kKVFull + slot), 0, g, id * bs);
              if (kHalves == 2) tma_load_3d(dst + kHalf, map, bar(kKVFull + slot), 64, g, id * bs);
            }
            if (which == 0) ++nk;
            else ++nv;
          }
          id_v = id_k;
          id_k = id_nxt;
        }
        // Rows of the item's last V tile past the context end may hold
        // anything (stale or never-written pool rows, even NaN); their
        // weights are 0, but 0 * NaN is NaN: clear them once the tile has
        // landed, before the PV that reads it.  The load was issued just
        // above, so waiting for it here cannot catch an older phase.
        if (ok && it.nkv > 0 && it.L < it.nkv * 128) {
          const int vn = kbase + it.nkv - 1;
          if (nfix > 0) ok = warp_wait(bar(kVFixFree), (nfix - 1) & 1);
          // every lane waits: each then writes into the landed tile
          if (ok) ok = mbar_wait_bounded(bar(kKVFull + v_slot(vn)), v_par(vn), p.wait_ns);
          ok = __all_sync(0xffffffffu, ok);
          if (ok) {
            uint8_t *vt = smem + kKVOff + v_slot(vn) * kTile;
            const int first = it.L - (it.nkv - 1) * 128;  // 1..127
            for (int i = lane; i < (128 - first) * (D / 8); i += 32) {
              const int row = first + i / (D / 8), c16 = i % (D / 8);
              *reinterpret_cast<uint4 *>(vt + (c16 >> 3) * kHalf + row * 128 + (c16 & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();  // generic writes before the tensor core reads
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kVFixed));
            ++nfix;
          }
        }
        kbase += it.nkv;
        x = __shfl_sync(0xffffffffu, x_next, 0);
        if (!ok) break;
      }
      if (!ok && lane == 0) {
        if (!misc[3]) raise_error(p.err, PA_DEVERR_TIMEOUT);
        misc[3] = 1;
      }
      // Do not leave while copies this CTA issued may still land (consumers
      // that gave up waiting no longer hold the block open).
      if (lane == 0) {
        if (nq > 0) mbar_wait_bounded(bar(kQFull), (nq - 1) & 1);
        for (int n = nk - 1; n >= 0 && n >= nk - kKBufs; --n)
          mbar_wait_bounded(bar(kKVFull + k_slot(n)), k_par(n));
        for (int n = nv - 1; n >= 0 && n >= nv - kVBufs; --n)
          mbar_wait_bounded(bar(kKVFull + v_slot(n)), v_par(n));
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // ----------------------------------------------------------- MMA --
      // The whole warp runs this loop; only the MMAs and commits are issued
      // by one elected lane (the same one every time: the warp is converged).
      constexpr bool kBF = E::kBF16;
      const uint32_t id_qk = idesc_f16(kBF, 128, 128, false);
      const uint32_t id_pv = idesc_f16(kBF, 128, D, true);
      const uint64_t q_desc[2] = {sdesc_sw128(smem_u32(smem + kQOff), 16, 1024),
                                  sdesc_sw128(smem_u32(smem + kQOff + kTile), 16, 1024)};
      int kbase = 0;            // ring position of this item's first K/V tile
      int pcnt[2] = {0, 0};     // P tiles consumed per query tile (all items)
      int prev_nkv[2] = {1, 1}; // the previous item's K/V tiles per query tile
      int nfix = 0;             // V tiles whose tail rows the TMA warp cleared
      bool ok = true;
      auto commit = [&](int b) {
        if (elect_one()) umma_commit(bar(b));
        __syncwarp();
      };
      auto qk = [&](int t, int kt) {  // S_t = Q_t K_kt^T
        const uint64_t qd = q_desc[t];
        const uint64_t kd =
            sdesc_sw128(smem_u32(smem + kKVOff + k_slot(kbase + kt) * kTile), 16, 1024);
        if (elect_one()) {
          // K step k: 16 columns = 32 bytes into a 128-byte swizzled row,
          // the second 64 columns in the tile's second half
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = ((k >> 2) * kHalf + (k & 3) * 32) >> 4;
            umma_f16_ss(tbase + t * 128, qd + off, kd + off, id_qk, k > 0 ? 1u : 0u);
          }
          umma_commit(bar(kSFull + t));
        }
        __syncwarp();
      };
      auto pv = [&](int t, int kt) {  // O_t += P_t V_kt, P_t from TMEM
        const uint64_t vd =
            sdesc_sw128(smem_u32(smem + kKVOff + v_slot(kbase + kt) * kTile), kHalf, 1024);
        const uint32_t acc0 = kt > 0 ? 1u : 0u;
        if (elect_one()) {
          // K step k: 16 keys = 16 rows of 128 bytes of the MN-major V tile
#pragma unroll
          for (int k = 0; k < 8; ++k)
            umma_f16_ts(tbase + 256 + t * 128, tbase + t * 128 + 8 * k, vd + ((k * 2048) >> 4),
                        id_pv, k > 0 ? 1u : acc0);
        }
        __syncwarp();
      };
      for (int j = 0;; ++j) {
        int x;
        PairItem it;
        ok = take_item(j, &x, &it);
        if (!ok || x < 0) break;
        // the item's last V tile reaches past the context end: its tail rows
        // are cleared by the TMA warp before any PV reads it
        const bool v_tail = it.nkv > 0 && it.L < it.nkv * 128;
        // S of both tiles is free (their last P was consumed before the
        // previous item's last PV), so this item's first QKs go at once; a
        // tile's first PV waits for the previous item's epilogue to have
        // read that tile's O (o_free).  A tile with no work this item gets
        // an empty S commit, which keeps its softmax warps in step.
        bool owait[2] = {j == 0, j == 0};  // o_free of the previous item seen
        // After an item in which a tile had no work, wait for that item's
        // o_free before committing the tile's next S: the epilogue only
        // frees O after the softmax has handed over its row sums, i.e.
        // after it took the empty commit (never two S phases behind).
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!owait[t] && prev_nkv[t] == 0) {
            if (ok) ok = warp_wait(bar(kOFree + t), (j - 1) & 1);
            owait[t] = true;
          }
        }
        if (ok) ok = warp_wait(bar(kQFull), j & 1);
        if (ok && it.nkv > 0) {
          ok = warp_wait(bar(kKVFull + k_slot(kbase)), k_par(kbase));
          tc_fence_after();
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok) break;
          if (it.nkv_t[t] > 0) {
            qk(t, 0);
          } else {
            if (!owait[t]) ok = warp_wait(bar(kOFree + t), (j - 1) & 1);
            owait[t] = true;
            commit(kSFull + t);
            commit(kOFull + t);  // nothing to add: O is "done" at once
          }
        }
        if (ok && it.nkv > 0) commit(kKVEmpty + k_slot(kbase));
        if (ok && it.nkv <= 1) commit(kQEmpty);  // no further QK reads Q
        for (int kt = 0; ok && kt < it.nkv; ++kt) {
          const bool more = kt + 1 < it.nkv;
          // Each group waits only for its own operands: PV for V_kt and P,
          // the next QK for K_{kt+1}, so a late K never holds back a PV.
          bool have_v = false, have_k = !more;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (kt < it.nkv_t[t]) {
              if (!owait[t]) {
                ok = warp_wait(bar(kOFree + t), (j - 1) & 1);
                owait[t] = true;
                if (!ok) break;
                tc_fence_after();
              }
              if (!have_v) {
                ok = warp_wait(bar(kKVFull + v_slot(kbase + kt)), v_par(kbase + kt));
                if (ok && v_tail && kt + 1 == it.nkv) {  // cleared by the TMA warp
                  ok = warp_wait(bar(kVFixed), nfix & 1);
                  if (lane == 0) mbar_arrive(bar(kVFixFree));
                  ++nfix;
                }
                have_v = true;
              }
              if (ok) ok = warp_wait(bar(kPFull + t), pcnt[t] & 1);
              if (!ok) break;
              tc_fence_after();
              pv(t, kt);
              if (kt + 1 == it.nkv_t[t]) commit(kOFull + t);  // tile t's last PV
              ++pcnt[t];
            }
            if (kt + 1 < it.nkv_t[t]) {
              if (!have_k) {
                ok = warp_wait(bar(kKVFull + k_slot(kbase + kt + 1)), k_par(kbase + kt + 1));
                have_k = true;
                if (!ok) break;
                tc_fence_after();
              }
              qk(t, kt + 1);
            }
          }
          if (!ok) break;
          // One elected block for the step's releases: V_kt, K_{kt+1} and,
          // after the item's last QK, Q.
          if (elect_one()) {
            if (kt + 2 == it.nkv) umma_commit(bar(kQEmpty));
            umma_commit(bar(kKVEmpty + v_slot(kbase + kt)));
            if (more) umma_commit(bar(kKVEmpty + k_slot(kbase + kt + 1)));
          }
          __syncwarp();
        }
        kbase += it.nkv;
        prev_nkv[0] = it.nkv_t[0];
        prev_nkv[1] = it.nkv_t[1];
        if (!ok) break;
      }
      if (!ok && lane == 0) {
        raise_error(p.err, PA_DEVERR_TIMEOUT);
        misc[3] = 1;
      }
      // Every MMA issued above has completed once this barrier fires (the
      // full bound: TMEM is freed after it).
      commit(kFin);
      if (lane == 0) mbar_wait_bounded(bar(kFin), 0);
      __syncwarp();
    }
  } else if (warp >= kEpiWarp0) {
    // ----------------------------------------------------- epilogue --
    // Per item and tile: wait for the tile's last PV and its row sums, read
    // O / l out of TMEM (then O is free for the next item's first PV) and
    // store the rows.  Runs alongside the next item's softmax.
    reg_dealloc<kEpilogueRegs>();
    const int q = warp - kEpiWarp0;  // TMEM lanes 32q .. 32q+31
    const int r = q * 32 + lane;     // query row in the tile
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    bool ok = true;
    for (int j = 0;; ++j) {
      int x;
      PairItem it;
      ok = take_item(j, &x, &it);
      if (!ok || x < 0) break;
#pragma unroll 1
      for (int t = 0; t < 2; ++t) {
        const int nkv_t = it.nkv_t[t];
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar(kOFull + t), j & 1, p.wait_ns));
        tc_fence_after();
        // every thread waits: each reads row sums another warp wrote
        if (ok) ok = mbar_wait_bounded(bar(kLFull + t), j & 1, p.wait_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        const float l = l_buf[t * 128 + r];
        const float inv_l = (nkv_t > 0 && l > 0.f) ? 1.f / l : 0.f;
        const bool rows = it.row0[t] < (it.q_len << p.pg_log2);
        uint32_t w[D / 2];  // the row of O / l, packed to the output type
        if (nkv_t > 0 && rows) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tbase + lane_addr + 256 + t * 128 + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[c * 16 + i] = E::pack2(__uint_as_float(o[2 * i]) * inv_l,
                                       __uint_as_float(o[2 * i + 1]) * inv_l);
          }
        } else {
#pragma unroll
          for (int i = 0; i < D / 2; ++i) w[i] = 0u;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kOFree + t));  // O of this tile is free
        // tile row -> (token, query head)
        const int prow = it.row0[t] + r;
        const int tok = prow >> p.pg_log2;
        const int head = (it.h << p.pg_log2) + (prow & (p.pg - 1));
        const int64_t grow = static_cast<int64_t>(it.q_start) + tok;
        if (rows && tok < it.q_len && grow >= 0 && grow < p.total_q) {
          typename E::T *orow =
              static_cast<typename E::T *>(p.out) + grow * p.out_row_stride + head * D;
#pragma unroll
          for (int c = 0; c < D / 8; ++c)
            *reinterpret_cast<uint4 *>(orow + c * 8) =
                make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        }
      }
      if (!ok) break;
    }
    if (!ok && lane == 0) {
      raise_error(p.err, PA_DEVERR_TIMEOUT);
      misc[3] = 1;
    }
  } else {
    // ------------------------------------------------------- softmax --
    reg_alloc<kSoftmaxRegs>();
    const int t = warp >> 2;   // tile A or B
    const int r = tid & 127;   // query row in the tile == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_tm = tbase + lane_addr + t * 128;
    const uint32_t o_tm = tbase + lane_addr + 256 + t * 128;
    const float sl = p.scale_log2;
    int n = 0;       // S phases of this query tile (QK results and empty commits)
    bool ok = true;
    for (int j = 0;; ++j) {
      int x;
      PairItem it;
      ok = take_item(j, &x, &it);
      if (!ok || x < 0) break;
      const int my_nkv = it.nkv_t[t];
      if (my_nkv == 0) {  // the MMA thread's empty S commit for this tile
        ok = mbar_wait_bounded(bar(kSFull + t), n & 1, p.wait_ns);
        ++n;
        if (!ok) break;
      }
      // last visible key of this row's token
      const int lim = min(it.lim_base + ((it.row0[t] + r) >> p.pg_log2), it.L - 1);
      float m_ref = -INFINITY, l = 0.f;
      for (int kt = 0; kt < my_nkv; ++kt, ++n) {
        ok = mbar_wait_bounded(bar(kSFull + t), n & 1, p.wait_ns);
        if (!ok) break;
        tc_fence_after();
        const int bound = lim - kt * 128;  // columns 0..bound are visible
        const bool edge = bound < 127;     // the tile crosses the causal edge or L
        // The whole S row in one TMEM round trip.
        uint32_t v[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(s_tm + c * 32, *reinterpret_cast<uint32_t(*)[32]>(v + c * 32));
        tmem_wait_ld();
        if (edge) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > bound) v[c] = __float_as_uint(-INFINITY);
        }
        // P = 2^(s * scale*log2(e) - mu) for the row, rounded to the input
        // type for the tensor core and packed two per word into pw; returns
        // the row sum of the same rounded values (exactly widened), so O / l
        // is an exact weighted mean of V under the rounded weights, and the
        // row's largest scaled score in *tmax.
        // With `store`, each 16 words go to TMEM as soon as they are made
        // (the max is already known); otherwise all of them stay in pw.
        // P overlays the first 64 columns of this tile's S in TMEM, two
        // 16-bit values per column (the A operand of O += P V).  S(kt) being
        // complete means PV(kt-1) has read P(kt-1): the tensor core runs one
        // thread's MMAs in order.
        uint32_t pw[64];
        auto p_row = [&](float mu, float *tmax, bool store) -> float {
          const uint64_t sl2 = f2_pack(sl, sl), nmu2 = f2_pack(-mu, -mu);
          float rs[4] = {0.f, 0.f, 0.f, 0.f};
          float mx[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) mx[i] = -INFINITY;
#pragma unroll
          for (int i = 0; i < 64; ++i) {  // column pair
            const float s0 = __uint_as_float(v[2 * i]), s1 = __uint_as_float(v[2 * i + 1]);
            if (!store) mx[i & 3] = fmaxf(mx[i & 3], fmaxf(s0, s1));
            float x0f, x1f;
            f2_unpack(f2_fma(f2_pack(s0, s1), sl2, nmu2), x0f, x1f);
            pw[i] = E::pack2(fast_exp2(x0f), fast_exp2(x1f));  // 2^-inf = 0 when masked
            E::add_halves(pw[i], rs[(i & 1) * 2], rs[(i & 1) * 2 + 1]);
            if (store && (i & 15) == 15)
              tmem_st16(s_tm + (i >> 4) * 16, *reinterpret_cast<uint32_t(*)[16]>(pw + i - 15));
          }
          *tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl;
          return (rs[0] + rs[1]) + (rs[2] + rs[3]);
        };
        // The running max m_ref is only raised -- and O rescaled -- when the
        // tile's max exceeds it by more than kRescaleThreshold (log2 units).
        // SPEC (launches whose queries fit one 128-row tile per sequence:
        // nothing else for the tensor core while this softmax runs): once a
        // row has a finite running max, its exponentials start from it at
        // once, the tile's max being found alongside them; the rare row whose
        // max does jump reloads its scores (still in TMEM: P is stored only
        // after this) and redoes them from the new max.  Otherwise (two query
        // tiles, whose softmaxes alternate with each other's MMAs, or the
        // row's first visible tile) the max comes first.  Measured, the early
        // start only pays where the softmax is the whole critical path, and
        // its code costs the other path when both are built in one kernel.
        auto row_max = [&]() {
          float mx[8];  // raw scores (scale > 0 keeps the order), as a tree
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(v[i]);
#pragma unroll
          for (int c = 8; c < 128; ++c) mx[c & 7] = fmaxf(mx[c & 7], __uint_as_float(v[c]));
          return fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl;
        };
        bool raise_max;
        float m_new, corr, rsum, mt;
        // Both branches hold warp-collective TMEM loads and stores, so each
        // is taken by the whole warp (a row for which the other branch would
        // do gets the same result from this one).
        if (!SPEC || __any_sync(0xffffffffu, m_ref == -INFINITY)) {
          mt = row_max();
          raise_max = mt > m_ref + kRescaleThreshold;  // false only for a fully masked row
          m_new = raise_max ? mt : m_ref;
          corr = raise_max ? fast_exp2(m_ref - m_new) : 1.f;
          rsum = p_row(m_new == -INFINITY ? 0.f : m_new, &mt, true);
        } else {
          rsum = p_row(m_ref, &mt, false);
          raise_max = mt > m_ref + kRescaleThreshold;
          m_new = raise_max ? mt : m_ref;
          corr = raise_max ? fast_exp2(m_ref - m_new) : 1.f;
          if (__any_sync(0xffffffffu, raise_max)) {  // rows that keep m_ref redo the same P
#pragma unroll
            for (int c = 0; c < 4; ++c)
              tmem_ld32(s_tm + c * 32, *reinterpret_cast<uint32_t(*)[32]>(v + c * 32));
            tmem_wait_ld();
            if (edge) {
#pragma unroll
              for (int c = 0; c < 128; ++c)
                if (c > bound) v[c] = __float_as_uint(-INFINITY);
            }
            rsum = p_row(m_new, &mt, true);
          } else {
#pragma unroll
            for (int hf = 0; hf < 4; ++hf)
              tmem_st16(s_tm + hf * 16, *reinterpret_cast<uint32_t(*)[16]>(pw + hf * 16));
          }
        }
        tmem_wait_st();
        if (kt >= 1 && __any_sync(0xffffffffu, raise_max)) {
          // O holds exactly the sum through PV(kt-1): S(kt) being complete
          // means QK(kt) ran, and it was issued after PV(kt-1).  Rescale it.
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(o_tm + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
            tmem_st32(o_tm + c * 32, o);
          }
          tmem_wait_st();
        }
        l = l * corr + rsum;
        m_ref = m_new;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kPFull + t));
      }
      if (!ok) break;
      // Hand the row sums to the epilogue once it has taken the previous
      // item's (its o_free of that item comes after reading them).
      if (j > 0) ok = warp_wait(bar(kOFree + t), (j - 1) & 1);
      if (!ok) break;
      l_buf[t * 128 + r] = l;
      mbar_arrive(bar(kLFull + t));
    }
    if (!ok) {
      raise_error(p.err, PA_DEVERR_TIMEOUT);
      misc[3] = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
  // Every claim of this CTA precedes its `done` count; the last CTA to
  // finish returns the slot to zero for the next launch.
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&sched->done, 1u) == gridDim.x - 1) {
      __threadfence();
      atomicExch(&sched->next, 0u);
      atomicExch(&sched->done, 0u);
    }
  }
}

}  // namespace

// The register split inside the kernel (setmaxnreg) must fit in what the
// CTA is launched with, or its .inc would wait for registers that never
// come: refuse to launch a build where it would not.
template <auto Kernel>
cudaError_t check_register_pool() {
  static const cudaError_t status = [] {
    cudaFuncAttributes attr;
    const cudaError_t e = cudaFuncGetAttributes(&attr, Kernel);
    if (e != cudaSuccess) return e;
    return attr.numRegs * kThreads >= kRegPoolNeeded ? cudaSuccess
                                                     : cudaErrorInvalidConfiguration;
  }();
  return status;
}

template <auto Kernel>
cudaError_t launch_variant(const PrefillParams &p, const PrefillArgs &a, int64_t grid,
                           cudaStream_t stream) {
  cudaError_t e = allow_dynamic_smem<Kernel>();
  if (e == cudaSuccess) e = check_register_pool<Kernel>();
  if (e != cudaSuccess) return e;
  return launch_pdl(Kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), kSmemBytes, stream,
                    p, a.tm_q, a.tm_k, a.tm_v);
}

// Launches so far in this process; picks each launch's schedule slot.
std::atomic<uint32_t> g_prefill_launches{0};

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
  p.pg = a.packed_heads;
  p.pg_log2 = 0;
  while ((1 << p.pg_log2) < p.pg) ++p.pg_log2;
  p.hu = p.hq / p.pg;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.scale_log2 = a.scale_log2;
  p.causal = a.causal;
  p.err = a.d_error;
  p.wait_ns = a.wait_ns;
  // Pairs of query tiles: sum_b ceil(pg q_b / 256) is at most both bounds
  // below; items are (pair, head unit).  One persistent CTA per SM walks them.
  const int64_t max_pairs = ((static_cast<int64_t>(a.max_seqlen_q) << p.pg_log2) + 255) / 256;
  int64_t slots = ((static_cast<int64_t>(a.total_q) << p.pg_log2) + 255LL * a.num_seqs) / 256;
  if (slots > a.num_seqs * max_pairs) slots = a.num_seqs * max_pairs;
  if (slots <= 0) return cudaSuccess;
  const int64_t items = slots * p.hu;
  if (items > 0x7fffffff) return cudaErrorInvalidValue;
  p.num_items = static_cast<int32_t>(items);
  p.sched_slot = static_cast<int32_t>(g_prefill_launches.fetch_add(1) % kSchedSlots);
  const int64_t grid = items < a.num_sms ? items : a.num_sms;
  // No sequence has more than one 128-row query tile (chunked prefill, a few
  // new tokens per sequence): every item is a single tile.
  if ((static_cast<int64_t>(a.max_seqlen_q) << p.pg_log2) <= 128) {
    if (a.dtype == PA_BF16)
      return a.head_dim == 64
                 ? launch_variant<prefill_kernel<BF16, 64, true>>(p, a, grid, stream)
                 : launch_variant<prefill_kernel<BF16, 128, true>>(p, a, grid, stream);
    return a.head_dim == 64 ? launch_variant<prefill_kernel<F16, 64, true>>(p, a, grid, stream)
                            : launch_variant<prefill_kernel<F16, 128, true>>(p, a, grid, stream);
  }
  if (a.dtype == PA_BF16)
    return a.head_dim == 64 ? launch_variant<prefill_kernel<BF16, 64, false>>(p, a, grid, stream)
                            : launch_variant<prefill_kernel<BF16, 128, false>>(p, a, grid, stream);
  return a.head_dim == 64 ? launch_variant<prefill_kernel<F16, 64, false>>(p, a, grid, stream)
                          : launch_variant<prefill_kernel<F16, 128, false>>(p, a, grid, stream);
}

}  // namespace pa
