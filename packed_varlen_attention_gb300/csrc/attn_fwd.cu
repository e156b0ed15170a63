// attn_fwd.cu -- FlashMask attention forward over packed samples on sm_103a.
//
// What is computed (PaddleNLP FlashMask article, section 3): FlashAttention-2
// tiling with an online softmax, where each (Q tile, KV tile) block is first
// classified from the eight per-tile statistics (section 3.2): fully masked
// blocks are skipped, partially masked blocks get the element mask, unmasked
// blocks run no mask arithmetic.  The result equals dense-mask attention
// (section 3.3); the forward pass also returns the softmax log-sum-exp that
// the backward operator consumes (section 3.4).
//
// How it runs on GB300:
//   * Planner (two tiny kernels): one warp per sample-local Q tile counts the
//     blocks that are not fully masked (its cost); a single CTA orders the
//     real Q tiles by cost, largest first (counting sort over cost bins).
//     Only real tiles become work items -- not the fixed grid
//     (seq_count, n_head, ceil(max_seq_len / Br)) of the Varlen-Packing
//     technical document, section 2, whose CTAs past a short sample's end do
//     nothing.
//   * Persistent main kernel, one CTA per SM, pulling items (Q tile x q head)
//     from an atomic counter.  Warp roles:
//       warp 0       producer: classifies the item's KV tiles (warp-parallel,
//                    32 tiles per step), TMA-loads Q once per item and K/V
//                    for every non-skipped tile into a 2-stage ring, and
//                    copies the four mask columns of partially masked tiles;
//       warp 1       MMA issuer (one thread): S = Q K^T into TMEM (two S
//                    buffers), then O += P V into a TMEM accumulator, with
//                    tcgen05.mma kind::f16 (bf16 in, fp32 accumulate);
//       warps 4..7   softmax: one thread per row of the 128-row tile reads
//                    its S row from TMEM, applies the mask (partial blocks
//                    only), keeps the running max / sum, rescales O in TMEM
//                    only when the max grew by more than 2^8, writes P as
//                    bf16 into shared memory (128-byte swizzled, K-major),
//                    and finally normalises O and writes out / lse.
//     The S MMA of tile j+1 runs on the tensor cores while the softmax
//     works on tile j.
//   * Every mbarrier wait is bounded (wall-clock limit) and reports
//     FM_DEVERR_TIMEOUT in the workspace error word instead of hanging.
//
// Layouts: q [T][Hq][D], k/v [T][Hkv][D] bf16, viewed by TMA as 2-D tensors
// (rows = tokens, columns = heads * D) with 64-column (128-byte) boxes and
// 128-byte swizzle; tile rows start at arbitrary token offsets and read into
// the neighbouring sample (masked) or past T (zero fill).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "fm_device.cuh"
#include "fm_internal.h"

namespace fm {
namespace {

constexpr int kThreads = 256;
constexpr int kStages = 2;
constexpr int kTileM = 128;  // MMA M: TMEM lanes = tile rows

enum : int { kClsF = 0, kClsP = 1, kClsU = 2, kClsStop = 3 };
enum : int { kFirst = 1, kLast = 2 };

struct TileMeta {
  int cls;     // kClsP / kClsU / kClsStop
  int flags;   // kFirst | kLast
  int c0, c1;  // key columns [c0, c1)
  int r0, r1;  // query rows of the item [r0, r1)
  int h;       // q head
  int kvh;     // key/value head
};

constexpr int kMetaSlots = 4;

enum Bar : int {
  kKFull = 0,                     // [kStages]  K tile landed (TMA tx)
  kKEmpty = kKFull + kStages,      // [kStages]  S MMA done reading K
  kVFull = kKEmpty + kStages,      // [kStages]  V tile landed
  kVEmpty = kVFull + kStages,      // [kStages]  PV MMA done reading V
  kMFull = kVEmpty + kStages,      // [kMetaSlots] tile metadata written
  kMEmpty = kMFull + kMetaSlots,   // [kMetaSlots] metadata consumed
  kQFull = kMEmpty + kMetaSlots,
  kQEmpty,
  kSFull,  // [2]
  kPFull = kSFull + 2,
  kPEmpty,
  kOEmpty,
  kDrain,
  kNumBars
};

// arrivals on kMEmpty: the V producer lane and the four softmax warps
constexpr int kMEmptyCount = 5;

template <int D, int BN>
struct Layout {
  static constexpr int kQBytes = kTileM * D * 2;
  static constexpr int kKBytes = BN * D * 2;
  static constexpr int kVBytes = BN * D * 2;
  static constexpr int kPBytes = kTileM * BN * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBytes;
  static constexpr int kV = kK + kStages * kKBytes;
  static constexpr int kP = kV + kStages * kVBytes;
  static constexpr int kCols = kP + kPBytes;  // int32 [kMetaSlots][4][BN]
  static constexpr int kMeta = kCols + kMetaSlots * 4 * BN * 4;
  static constexpr int kBars = kMeta + kMetaSlots * static_cast<int>(sizeof(TileMeta));
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kEnd = kAbort + 4;
  static constexpr int kBytes = kEnd + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kTmemS = 0;       // S buffers at columns [0, 2*BN)
  static constexpr int kTmemO = 2 * BN;  // O at columns [2*BN, 2*BN + D)
  static_assert(2 * BN + D <= 512, "TMEM budget");
  static_assert(kBytes <= 232448, "shared memory budget");
};

__device__ __forceinline__ int clamp_tok(int x, int T) { return x < 0 ? 0 : (x > T ? T : x); }

// Block class from the eight statistics of the key tile (FlashMask article,
// section 3.2; rows [r0, r1) half-open, the diagonal counts as lower).
__device__ __forceinline__ int classify_block(int r0, int r1, int c0, int c1, const int* st,
                                              bool has_mask, bool causal) {
  bool lt_full = false, lt_touch = false, ut_full = false, ut_touch = false;
  if (has_mask) {
    lt_full = r0 >= st[1] && r1 <= st[2];
    lt_touch = r0 < st[3] && r1 > st[0];
    ut_full = r0 >= st[5] && r1 <= st[6];
    ut_touch = r0 < st[7] && r1 > st[4];
  }
  if (causal) ut_full = ut_touch = true;
  if (r1 - 1 < c0) return ut_full ? kClsF : (ut_touch ? kClsP : kClsU);
  if (r0 >= c1 - 1) return lt_full ? kClsF : (lt_touch ? kClsP : kClsU);
  if (lt_full && ut_full) return kClsF;
  if (causal || lt_touch || ut_touch) return kClsP;
  return kClsU;
}

__device__ __forceinline__ void load_stats(const AttnParams& p, int mh, int64_t slot, int* st) {
#pragma unroll
  for (int v = 0; v < 8; ++v)
    st[v] = __ldg(p.minmax + (static_cast<int64_t>(mh) * 8 + v) * p.n_kv_slots + slot);
}

// Class of KV tile kt of sample [a, b) for rows [r0, r1), or kClsF past kt_end.
template <int BN>
__device__ __forceinline__ int tile_class(const AttnParams& p, int mh, int s, int a, int b,
                                          int r0, int r1, int kt, int kt_end) {
  if (kt >= kt_end) return kClsF;
  const int c0 = a + kt * BN;
  const int c1 = min(c0 + BN, b);
  int st[8];
  const bool has_mask = p.sri != nullptr;
  if (has_mask) load_stats(p, mh, static_cast<int64_t>(a / BN) + s + kt, st);
  return classify_block(r0, r1, c0, c1, st, has_mask, p.causal != 0);
}

// Number of KV tiles to examine for rows ending at r1 (causal: up to the
// diagonal; every later tile is entirely above it and fully masked).
template <int BN>
__device__ __forceinline__ int kv_tiles_to_scan(const AttnParams& p, int a, int b, int r1) {
  const int n_kv = (b - a + BN - 1) / BN;
  if (p.causal) return min(n_kv, (r1 - 1 - a) / BN + 1);
  return n_kv;
}

// ---------------------------------------------------------------------------
// planner
// ---------------------------------------------------------------------------

template <int BN>
__global__ void __launch_bounds__(256) plan_cost_kernel(const AttnParams p) {
  const int64_t u = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (u >= p.n_qslots) return;
  const int T = static_cast<int>(p.T);
  const int BM = p.block_m;
  int lo = 0, hi = p.n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int64_t base = static_cast<int64_t>(clamp_tok(__ldg(p.cu + mid), T)) / BM + mid;
    if (base <= u) lo = mid; else hi = mid - 1;
  }
  const int s = lo;
  const int a = clamp_tok(__ldg(p.cu + s), T);
  const int b = max(a, clamp_tok(__ldg(p.cu + s + 1), T));
  const int64_t qt = u - (static_cast<int64_t>(a) / BM + s);
  if (qt < 0 || a + qt * BM >= b) {
    if (lane == 0) p.cost[u] = -1;
    return;
  }
  const int r0 = a + static_cast<int>(qt) * BM;
  const int r1 = min(r0 + BM, b);
  const int kt_end = kv_tiles_to_scan<BN>(p, a, b, r1);
  int cost = 0;
  for (int base = 0; base < kt_end; base += 32) {
    const int cls = tile_class<BN>(p, 0, s, a, b, r0, r1, base + lane, kt_end);
    cost += __popc(__ballot_sync(0xffffffffu, cls != kClsF));
  }
  if (lane == 0) {
    p.cost[u] = cost;
    p.slot_info[u] = make_int2(s, static_cast<int>(qt));
    atomicAdd(p.hist + min(cost, kCostBins - 1), 1);
  }
}

__global__ void __launch_bounds__(kCostBins) plan_order_kernel(const AttnParams p) {
  __shared__ int offs[kCostBins];
  __shared__ int warp_tot[kCostBins / 32];
  const int tid = threadIdx.x;
  const int lane = tid & 31, w = tid >> 5;
  // descending cost: position 0 holds the largest bin
  const int bin = kCostBins - 1 - tid;
  const int cnt = p.hist[bin];
  int x = cnt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) warp_tot[w] = x;
  __syncthreads();
  if (w == 0) {
    int t = warp_tot[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, d);
      if (lane >= d) t += y;
    }
    warp_tot[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  const int incl = x + (w > 0 ? warp_tot[w - 1] : 0);
  offs[bin] = incl - cnt;
  if (tid == kCostBins - 1) {
    p.ws->n_qtiles = incl;
    p.ws->n_items = incl * p.hq;
  }
  __syncthreads();
  for (int64_t u = tid; u < p.n_qslots; u += kCostBins) {
    const int c = p.cost[u];
    if (c >= 0) {
      const int pos = atomicAdd(&offs[min(c, kCostBins - 1)], 1);
      p.order[pos] = p.slot_info[u];
    }
  }
  // cu_seqlens sanity: cu[0] = 0, non-decreasing, cu[n] = T
  bool bad = false;
  for (int s = tid; s < p.n_seqs; s += kCostBins) {
    const int a = __ldg(p.cu + s), b = __ldg(p.cu + s + 1);
    if (b < a || a < 0 || b > p.T) bad = true;
  }
  if (tid == 0 && (__ldg(p.cu) != 0 || __ldg(p.cu + p.n_seqs) != p.T)) bad = true;
  if (bad) atomicOr(&p.ws->error_word, static_cast<int>(FM_DEVERR_DATA));
}

// ---------------------------------------------------------------------------
// persistent attention kernel
// ---------------------------------------------------------------------------

template <int D, int BN, typename IdxT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tq,
                    const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv) {
  using L = Layout<D, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  TileMeta* meta = reinterpret_cast<TileMeta*>(smem + L::kMeta);
  int* cols = reinterpret_cast<int*>(smem + L::kCols);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = static_cast<int>(p.T);
  const uint64_t tmo = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars[kKFull + i], 1);
      mbar_init(&bars[kKEmpty + i], 1);
      mbar_init(&bars[kVFull + i], 1);
      mbar_init(&bars[kVEmpty + i], 1);
    }
    for (int i = 0; i < kMetaSlots; ++i) {
      mbar_init(&bars[kMFull + i], 1);
      mbar_init(&bars[kMEmpty + i], kMEmptyCount);
    }
    mbar_init(&bars[kQFull], 1);
    mbar_init(&bars[kQEmpty], 1);
    mbar_init(&bars[kSFull + 0], 1);
    mbar_init(&bars[kSFull + 1], 1);
    mbar_init(&bars[kPFull], 128);
    mbar_init(&bars[kPEmpty], 1);
    mbar_init(&bars[kOEmpty], 128);
    mbar_init(&bars[kDrain], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(&p.ws->error_word, static_cast<int>(FM_DEVERR_TIMEOUT));
  };
  // every lane waits; the warp proceeds only if all lanes saw the phase
  auto warp_wait = [&](int bar, uint32_t parity) -> bool {
    const bool ok = mbar_wait_bounded(&bars[bar], parity, tmo, abort_flag);
    const bool all = __all_sync(0xffffffffu, ok);
    if (!all && lane == 0) fail();
    return all;
  };
  // single-thread wait
  auto lone_wait = [&](int bar, uint32_t parity) -> bool {
    if (mbar_wait_bounded(&bars[bar], parity, tmo, abort_flag)) return true;
    fail();
    return false;
  };

  if (warp == 0) {
    // --------------------------------------------------- K producer + metadata
    const int n_items = p.ws->n_items;
    const int group = p.hq / p.hkv;
    uint32_t kst = 0, kround = 0;    // K ring
    uint32_t mslot = 0, mround = 0;  // metadata ring
    uint32_t q_round = 0;
    uint32_t k_armed[kStages] = {0xffffffffu, 0xffffffffu};
    uint32_t q_armed = 0xffffffffu;
    long long cnt_p = 0, cnt_u = 0, cnt_f = 0;
    bool ok = true;

    auto push_meta = [&](int cls, int flags, int c0, int c1, int r0, int r1, int h, int kvh,
                         bool copy_cols, int mh) -> bool {
      if (!warp_wait(kMEmpty + mslot, (mround & 1) ^ 1)) return false;
      if (copy_cols) {
        const int32_t* src = p.sri + static_cast<int64_t>(mh) * 4 * p.T;
        int* dst = cols + mslot * 4 * BN;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
#pragma unroll
          for (int m = 0; m < BN / 32; ++m) {
            const int jj = m * 32 + lane;
            const int c = c0 + jj;
            dst[v * BN + jj] = (c < T) ? __ldg(src + static_cast<int64_t>(v) * p.T + c) : 0;
          }
        }
      }
      if (lane == 0) {
        TileMeta& m = meta[mslot];
        m.cls = cls;
        m.flags = flags;
        m.c0 = c0;
        m.c1 = c1;
        m.r0 = r0;
        m.r1 = r1;
        m.h = h;
        m.kvh = kvh;
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kMFull + mslot]);
      if (++mslot == kMetaSlots) {
        mslot = 0;
        ++mround;
      }
      return true;
    };

    while (ok) {
      int item = 0;
      if (lane == 0) item = static_cast<int>(atomicAdd(&p.ws->work_counter, 1u));
      item = __shfl_sync(0xffffffffu, item, 0);
      if (item >= n_items) {
        ok = push_meta(kClsStop, 0, 0, 0, 0, 0, 0, 0, false, 0);
        break;
      }
      const int2 qi = p.order[item / p.hq];
      const int h = item % p.hq;
      const int s = qi.x;
      const int kvh = h / group;
      const int mh = p.hm > 1 ? h : 0;
      const int a = clamp_tok(__ldg(p.cu + s), T);
      const int b = max(a, clamp_tok(__ldg(p.cu + s + 1), T));
      const int r0 = min(a + qi.y * p.block_m, b);
      const int r1 = min(r0 + p.block_m, b);
      const int n_kv = (b - a + BN - 1) / BN;
      const int kt_end = (r1 > r0) ? kv_tiles_to_scan<BN>(p, a, b, r1) : 0;

      // pass 1: block classes of the item (counts, number of live tiles)
      int n_live = 0, n_p = 0;
      for (int base = 0; base < kt_end; base += 32) {
        const int cls = tile_class<BN>(p, mh, s, a, b, r0, r1, base + lane, kt_end);
        n_live += __popc(__ballot_sync(0xffffffffu, cls != kClsF));
        n_p += __popc(__ballot_sync(0xffffffffu, cls == kClsP));
      }
      cnt_p += n_p;
      cnt_u += n_live - n_p;
      cnt_f += n_kv - n_live;

      if (n_live == 0) {
        // every key of these rows is masked: o = 0, lse = -inf
        for (int r = r0 + lane; r < r1; r += 32) {
          uint4* dst = reinterpret_cast<uint4*>(
              static_cast<__nv_bfloat16*>(p.out) +
              (static_cast<IdxT>(r) * p.hq + h) * static_cast<IdxT>(D));
#pragma unroll
          for (int u = 0; u < D / 8; ++u) dst[u] = make_uint4(0u, 0u, 0u, 0u);
          p.lse[static_cast<IdxT>(h) * static_cast<IdxT>(p.T) + r] = -CUDART_INF_F;
        }
        continue;
      }

      // pass 2: metadata and K for every tile that is not fully masked
      int pushed = 0;
      for (int base = 0; base < kt_end && ok; base += 32) {
        const int my_cls = tile_class<BN>(p, mh, s, a, b, r0, r1, base + lane, kt_end);
        uint32_t live = __ballot_sync(0xffffffffu, my_cls != kClsF);
        while (live != 0u) {
          const int l = __ffs(live) - 1;
          live &= live - 1u;
          const int cls = __shfl_sync(0xffffffffu, my_cls, l);
          const int c0 = a + (base + l) * BN;
          const int c1 = min(c0 + BN, b);
          const int flags = (pushed == 0 ? kFirst : 0) | (pushed == n_live - 1 ? kLast : 0);
          if (!push_meta(cls, flags, c0, c1, r0, r1, h, kvh, cls == kClsP && p.sri != nullptr,
                         mh)) {
            ok = false;
            break;
          }
          if (pushed == 0) {
            // Q tile of this item, once the previous item's S MMAs are done
            if (!warp_wait(kQEmpty, (q_round & 1) ^ 1)) {
              ok = false;
              break;
            }
            if (lane == 0) {
              mbar_arrive_expect_tx(&bars[kQFull], L::kQBytes);
#pragma unroll
              for (int c = 0; c < D / 64; ++c)
                tma_load_2d(smem + L::kQ + c * (kTileM * 128), &tq, &bars[kQFull],
                            h * D + c * 64, r0);
            }
            q_armed = q_round;
            ++q_round;
          }
          if (!warp_wait(kKEmpty + kst, (kround & 1) ^ 1)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&bars[kKFull + kst], L::kKBytes);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_2d(smem + L::kK + kst * L::kKBytes + c * (BN * 128), &tk,
                          &bars[kKFull + kst], kvh * D + c * 64, c0);
          }
          k_armed[kst] = kround;
          if (++kst == kStages) {
            kst = 0;
            ++kround;
          }
          ++pushed;
        }
      }
    }
    if (!ok) {
      // let every TMA load this warp issued land before the CTA exits
      for (int st = 0; st < kStages; ++st)
        if (k_armed[st] != 0xffffffffu)
          mbar_wait_bounded(&bars[kKFull + st], k_armed[st] & 1, 100000000ull, nullptr);
      if (q_armed != 0xffffffffu)
        mbar_wait_bounded(&bars[kQFull], q_armed & 1, 100000000ull, nullptr);
    }
    if (lane == 0 && p.class_counts != nullptr) {
      atomicAdd(reinterpret_cast<unsigned long long*>(p.class_counts + 0),
                static_cast<unsigned long long>(cnt_f));
      atomicAdd(reinterpret_cast<unsigned long long*>(p.class_counts + 1),
                static_cast<unsigned long long>(cnt_p));
      atomicAdd(reinterpret_cast<unsigned long long*>(p.class_counts + 2),
                static_cast<unsigned long long>(cnt_u));
    }
  } else if (warp == 2) {
    // --------------------------------------------------------------- V producer
    if (lane == 0) {
      uint32_t vst = 0, vround = 0, mslot = 0, mround = 0;
      uint32_t v_armed[kStages] = {0xffffffffu, 0xffffffffu};
      bool ok = true;
      for (;;) {
        if (!lone_wait(kMFull + mslot, mround & 1)) { ok = false; break; }
        const int cls = *reinterpret_cast<volatile int*>(&meta[mslot].cls);
        const int c0 = *reinterpret_cast<volatile int*>(&meta[mslot].c0);
        const int kvh = *reinterpret_cast<volatile int*>(&meta[mslot].kvh);
        mbar_arrive(&bars[kMEmpty + mslot]);
        if (++mslot == kMetaSlots) {
          mslot = 0;
          ++mround;
        }
        if (cls == kClsStop) break;
        if (!lone_wait(kVEmpty + vst, (vround & 1) ^ 1)) { ok = false; break; }
        mbar_arrive_expect_tx(&bars[kVFull + vst], L::kVBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(smem + L::kV + vst * L::kVBytes + c * (BN * 128), &tv,
                      &bars[kVFull + vst], kvh * D + c * 64, c0);
        v_armed[vst] = vround;
        if (++vst == kStages) {
          vst = 0;
          ++vround;
        }
      }
      if (!ok) {
        for (int st = 0; st < kStages; ++st)
          if (v_armed[st] != 0xffffffffu)
            mbar_wait_bounded(&bars[kVFull + st], v_armed[st] & 1, 100000000ull, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kTileM, BN, false);
      constexpr uint32_t kIdescO = idesc_bf16_f32(kTileM, D, true);
      const uint32_t q_addr = smem_u32(smem + L::kQ);
      const uint32_t k_addr = smem_u32(smem + L::kK);
      const uint32_t v_addr = smem_u32(smem + L::kV);
      const uint32_t p_addr = smem_u32(smem + L::kP);
      uint32_t mslot = 0, mround = 0;  // metadata ring
      uint32_t kst = 0, kround = 0, vst = 0, vround = 0;
      uint32_t q_round = 0, p_round = 0, o_round = 0, sbuf = 0;
      int items_done = 0;
      bool ok = true;

      // flags of the next tile (kClsStop -> stop); the softmax warps release
      // the metadata slot
      auto next_meta = [&](int& flags) -> int {
        if (!lone_wait(kMFull + mslot, mround & 1)) return -1;
        const int cls = *reinterpret_cast<volatile int*>(&meta[mslot].cls);
        flags = *reinterpret_cast<volatile int*>(&meta[mslot].flags);
        if (++mslot == kMetaSlots) {
          mslot = 0;
          ++mround;
        }
        return cls;
      };
      auto issue_s = [&](uint32_t buf) -> bool {
        if (!lone_wait(kKFull + kst, kround & 1)) return false;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + L::kTmemS + buf * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk & 3) * 32;
          const uint32_t chunk = kk >> 2;
          const uint64_t ad = sdesc_sw128(q_addr + chunk * (kTileM * 128) + koff, 16, 1024);
          const uint64_t bd =
              sdesc_sw128(k_addr + kst * L::kKBytes + chunk * (BN * 128) + koff, 16, 1024);
          umma_bf16(d_tmem, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars[kSFull + buf]);
        umma_commit(&bars[kKEmpty + kst]);
        if (++kst == kStages) {
          kst = 0;
          ++kround;
        }
        return true;
      };
      auto issue_pv = [&](bool first) -> bool {
        if (!lone_wait(kVFull + vst, vround & 1)) return false;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + L::kTmemO;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint32_t koff = (kk & 3) * 32;
          const uint32_t chunk = kk >> 2;
          const uint64_t ad = sdesc_sw128(p_addr + chunk * (kTileM * 128) + koff, 16, 1024);
          const uint64_t bd =
              sdesc_sw128(v_addr + vst * L::kVBytes + kk * (16 * 128), BN * 128, 1024);
          umma_bf16(d_tmem, ad, bd, kIdescO, (!first || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bars[kVEmpty + vst]);
        umma_commit(&bars[kPEmpty]);
        if (++vst == kStages) {
          vst = 0;
          ++vround;
        }
        return true;
      };
      // S MMA of the first tile of a new item (waits for its Q tile)
      auto start_item = [&](int flags, uint32_t buf) -> bool {
        if (!lone_wait(kQFull, q_round & 1)) return false;
        ++q_round;
        tc_fence_after();
        if (!issue_s(buf)) return false;
        if (flags & kLast) umma_commit(&bars[kQEmpty]);
        return true;
      };

      int cur_flags = 0;
      int cls = next_meta(cur_flags);
      ok = (cls >= 0);
      bool stop = (cls == kClsStop);
      if (ok && !stop) ok = start_item(cur_flags, sbuf);
      while (ok && !stop) {
        int nxt_flags = 0;
        if (!(cur_flags & kLast)) {
          // S of the next tile of the same item overlaps this tile's softmax
          cls = next_meta(nxt_flags);
          if (cls < 0 || cls == kClsStop) { ok = false; break; }
          if (!issue_s(sbuf ^ 1u)) { ok = false; break; }
          if (nxt_flags & kLast) umma_commit(&bars[kQEmpty]);
        }
        if (!lone_wait(kPFull, p_round & 1)) { ok = false; break; }
        ++p_round;
        tc_fence_after();
        if ((cur_flags & kFirst) && items_done > 0) {
          if (!lone_wait(kOEmpty, o_round & 1)) { ok = false; break; }
          ++o_round;
          tc_fence_after();
        }
        if (!issue_pv((cur_flags & kFirst) != 0)) { ok = false; break; }
        if (cur_flags & kLast) {
          ++items_done;
          cls = next_meta(nxt_flags);
          if (cls < 0) { ok = false; break; }
          if (cls == kClsStop) break;
          if (!start_item(nxt_flags, sbuf ^ 1u)) { ok = false; break; }
        }
        cur_flags = nxt_flags;
        sbuf ^= 1u;
      }
      // all issued MMAs complete before TMEM is released
      umma_commit(&bars[kDrain]);
      mbar_wait_bounded(&bars[kDrain], 0, 100000000ull, nullptr);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_tmem = tmem_base + lane_addr + L::kTmemS;
    const uint32_t o_tmem = tmem_base + lane_addr + L::kTmemO;
    const uint32_t p_row = smem_u32(smem + L::kP) + row * 128;
    const float scale_log2 = p.scale_log2;
    const bool has_mask = p.sri != nullptr;
    const bool causal = p.causal != 0;
    uint32_t mslot = 0, mround = 0, sbuf = 0;
    uint32_t s_round[2] = {0u, 0u};
    uint32_t n_tiles = 0;
    float m_run = -CUDART_INF_F, l_run = 0.f;
    int r0 = 0, r1 = 0, h = 0;

    for (;;) {
      if (!warp_wait(kMFull + mslot, mround & 1)) break;
      TileMeta md;
      md.cls = *reinterpret_cast<volatile int*>(&meta[mslot].cls);
      if (md.cls == kClsStop) break;
      md.flags = *reinterpret_cast<volatile int*>(&meta[mslot].flags);
      md.c0 = *reinterpret_cast<volatile int*>(&meta[mslot].c0);
      md.c1 = *reinterpret_cast<volatile int*>(&meta[mslot].c1);
      md.r0 = *reinterpret_cast<volatile int*>(&meta[mslot].r0);
      md.r1 = *reinterpret_cast<volatile int*>(&meta[mslot].r1);
      md.h = *reinterpret_cast<volatile int*>(&meta[mslot].h);
      const uint32_t cur_slot = mslot;
      if (++mslot == kMetaSlots) {
        mslot = 0;
        ++mround;
      }

      const bool first = (md.flags & kFirst) != 0;
      if (first) {
        m_run = -CUDART_INF_F;
        l_run = 0.f;
        r0 = md.r0;
        r1 = md.r1;
        h = md.h;
      }
      if (!warp_wait(kSFull + sbuf, s_round[sbuf] & 1)) break;
      ++s_round[sbuf];
      tc_fence_after();

      float sv[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(s_tmem + sbuf * BN + c * 32, rr);
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[c * 32 + i] = __uint_as_float(rr[i]) * scale_log2;
      }

      const int r = r0 + row;
      if (md.cls == kClsP) {
        const int* cl = cols + cur_slot * 4 * BN;
#pragma unroll
        for (int jj = 0; jj < BN; ++jj) {
          const int c = md.c0 + jj;
          bool masked;
          if (c >= md.c1) {
            masked = true;
          } else if (r >= c) {
            masked = has_mask && (cl[jj] <= r) && (r < cl[BN + jj]);
          } else {
            masked = causal || (has_mask && (cl[2 * BN + jj] <= r) && (r < cl[3 * BN + jj]));
          }
          if (masked) sv[jj] = -CUDART_INF_F;
        }
      } else if (md.c1 - md.c0 < BN) {
        const int valid = md.c1 - md.c0;
#pragma unroll
        for (int jj = 0; jj < BN; ++jj)
          if (jj >= valid) sv[jj] = -CUDART_INF_F;
      }
      // metadata and mask columns of this tile are no longer needed
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kMEmpty + cur_slot]);

      float mt = sv[0];
#pragma unroll
      for (int jj = 1; jj < BN; ++jj) mt = fmaxf(mt, sv[jj]);
      const float m_new = fmaxf(m_run, mt);
      // keep the old reference max unless it grew by more than 2^8
      const bool resc = first || (m_new > m_run + 8.0f);
      float factor = 1.f;
      float m_ref = m_run;
      if (resc) {
        factor = (m_run == -CUDART_INF_F) ? 0.f : ex2_approx(m_run - m_new);
        m_ref = m_new;
      }
      const bool need_o = resc && !first && (m_run != -CUDART_INF_F);
      if (__any_sync(0xffffffffu, need_o)) {
        // O may be rescaled only once the previous PV MMA has finished
        if (!warp_wait(kPEmpty, (n_tiles - 1) & 1)) break;
        tc_fence_after();
        const float f = need_o ? factor : 1.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(o_tmem + c * 32, rr);
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * f);
          tmem_st32(o_tmem + c * 32, rr);
        }
        tmem_st_wait();
      }
      if (resc) l_run = first ? 0.f : l_run * factor;
      m_run = m_ref;

      const float base = (m_ref == -CUDART_INF_F) ? 0.f : m_ref;
      float sum = 0.f;
      uint32_t pk[BN / 2];
#pragma unroll
      for (int jj = 0; jj < BN; jj += 2) {
        const float p0 = ex2_approx(sv[jj] - base);
        const float p1 = ex2_approx(sv[jj + 1] - base);
        sum += p0 + p1;
        pk[jj / 2] = pack_bf16x2(p0, p1);
      }
      l_run += sum;

      // the P buffer is free once the previous PV MMA has finished
      if (n_tiles > 0) {
        if (!warp_wait(kPEmpty, (n_tiles - 1) & 1)) break;
      }
#pragma unroll
      for (int u = 0; u < BN / 8; ++u) {
        const uint32_t kc = u >> 3;
        const uint32_t swz = static_cast<uint32_t>((u & 7) ^ (row & 7));
        st_shared_v4(p_row + kc * (kTileM * 128) + swz * 16, pk[4 * u + 0], pk[4 * u + 1],
                     pk[4 * u + 2], pk[4 * u + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[kPFull]);
      ++n_tiles;
      sbuf ^= 1u;

      if (md.flags & kLast) {
        if (!warp_wait(kPEmpty, (n_tiles - 1) & 1)) break;
        tc_fence_after();
        const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) +
                             (static_cast<IdxT>(r) * p.hq + h) * static_cast<IdxT>(D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(o_tmem + c * 32, rr);
          if (r < r1) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              d4[u] = make_uint4(
                  pack_bf16x2(__uint_as_float(rr[8 * u + 0]) * inv_l,
                              __uint_as_float(rr[8 * u + 1]) * inv_l),
                  pack_bf16x2(__uint_as_float(rr[8 * u + 2]) * inv_l,
                              __uint_as_float(rr[8 * u + 3]) * inv_l),
                  pack_bf16x2(__uint_as_float(rr[8 * u + 4]) * inv_l,
                              __uint_as_float(rr[8 * u + 5]) * inv_l),
                  pack_bf16x2(__uint_as_float(rr[8 * u + 6]) * inv_l,
                              __uint_as_float(rr[8 * u + 7]) * inv_l));
            }
          }
        }
        if (r < r1) {
          p.lse[static_cast<IdxT>(h) * static_cast<IdxT>(p.T) + r] =
              (l_run > 0.f) ? (m_run + __log2f(l_run)) * 0.69314718055994531f : -CUDART_INF_F;
        }
        tc_fence_before();
        mbar_arrive(&bars[kOEmpty]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, L::kTmemCols);
  }
}

__global__ void bounded_wait_probe_kernel(int32_t* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  // nothing ever arrives on `bar`: the wait must give up by itself
  const bool ok = mbar_wait_bounded(&bar, 0, timeout_ns, nullptr);
  __syncthreads();
  if (threadIdx.x == 0) *status = ok ? FM_OK : FM_ERR_TIMEOUT;
}

template <int D, int BN, typename IdxT>
cudaError_t launch_typed(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, int num_sms, cudaStream_t stream) {
  using L = Layout<D, BN>;
  static bool configured = false;  // benign race: the attribute call is idempotent
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, BN, IdxT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t qwarps = p.n_qslots;
  plan_cost_kernel<BN><<<static_cast<unsigned>((qwarps + 7) / 8), 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  plan_order_kernel<<<1, kCostBins, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t max_items = p.n_qslots * p.hq;
  const int grid = static_cast<int>(max_items < num_sms ? max_items : num_sms);
  attn_fwd_kernel<D, BN, IdxT><<<grid, kThreads, L::kBytes, stream>>>(p, tq, tk, tv);
  return cudaGetLastError();
}

}  // namespace

size_t attn_workspace_bytes(int64_t T, int n_seqs, int block_m) {
  const int64_t n_qslots = T / block_m + n_seqs;
  size_t bytes = sizeof(AttnWorkspaceHeader) + kCostBins * sizeof(int);
  bytes += static_cast<size_t>(n_qslots) * (sizeof(int) + 2 * sizeof(int2));
  return (bytes + 255) & ~static_cast<size_t>(255);
}

cudaError_t launch_attn_fwd(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, bool use_int64, int num_sms,
                            cudaStream_t stream) {
  if (p.head_dim == 128) {
    if (p.block_n == 128)
      return use_int64 ? launch_typed<128, 128, int64_t>(p, tq, tk, tv, num_sms, stream)
                       : launch_typed<128, 128, int32_t>(p, tq, tk, tv, num_sms, stream);
    return use_int64 ? launch_typed<128, 64, int64_t>(p, tq, tk, tv, num_sms, stream)
                     : launch_typed<128, 64, int32_t>(p, tq, tk, tv, num_sms, stream);
  }
  if (p.block_n == 128)
    return use_int64 ? launch_typed<64, 128, int64_t>(p, tq, tk, tv, num_sms, stream)
                     : launch_typed<64, 128, int32_t>(p, tq, tk, tv, num_sms, stream);
  return use_int64 ? launch_typed<64, 64, int64_t>(p, tq, tk, tv, num_sms, stream)
                   : launch_typed<64, 64, int32_t>(p, tq, tk, tv, num_sms, stream);
}

cudaError_t launch_bounded_wait_probe(int32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  bounded_wait_probe_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace fm
