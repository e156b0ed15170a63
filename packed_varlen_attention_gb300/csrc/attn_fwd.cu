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
//   * Planner (two tiny kernels, also callable alone so that the layers of
//     one packed batch share one plan): one warp per planner slot (a Q tile,
//     or a sample-local pair of Q tiles) counts the blocks that are not fully
//     masked (its cost); one CTA orders the real slots by cost, largest first
//     (counting sort over cost bins), and writes the header (item count, the
//     sizes and item form planned for).
//     Only real tiles become work -- not the fixed grid
//     (seq_count, n_head, ceil(max_seq_len / Br)) of the Varlen-Packing
//     technical document, section 2, whose CTAs past a short sample's end do
//     nothing.
//   * Persistent main kernel, one CTA per SM, pulling items from an atomic
//     counter; the last CTA to finish claiming resets the counter, so a plan
//     can be used again.  An item is two Q tiles that share every K/V tile
//     the CTA loads: one Q tile for two q heads of one key/value head when
//     the group size is even and every head has the same mask (both tiles
//     then see the same blocks), else two consecutive Q tiles of one q head,
//     paired from the sample's end so that a sample with an odd number of Q
//     tiles leaves its first (under a causal mask cheapest) tile unpaired.
//     Warp roles (384 threads; warps 0..3 at 96 registers, the softmax
//     warpgroups at 200):
//       warp 0      K producer: checks the plan's sizes, classifies the
//                   item's KV tiles for both Q tiles (warp-parallel, 32 tiles
//                   per step), loads Q tile 0 into the Q ring right after,
//                   then publishes per-tile metadata (and the mask columns of
//                   partially masked tiles) in a 4-slot ring and TMA-loads K
//                   per tile into the K/V ring (Q tile 1 after the first K);
//       warp 2      V producer: TMA-loads V per tile into the same ring;
//       warps 1, 3  MMA issuers, one per Q tile, taking strict turns
//                   (tcgen05.mma kind::f16, bf16 in, fp32 accumulate): S_i =
//                   Q_i K^T into TMEM, then O_i += P_i V with P_i read from
//                   TMEM (it overwrites the first half of S_i's columns as
//                   packed bf16);
//       warps 4..7  softmax of Q tile 0, warps 8..11 softmax of Q tile 1: one
//                   thread per tile row (= TMEM lane).  The whole S row is
//                   loaded from TMEM with one wait, masked (partial blocks
//                   only), reduced to its max, turned into
//                   P = 2^(S*scale*log2e - m) with a running sum and stored as
//                   bf16 into TMEM.  O_i is rescaled in TMEM only when the max
//                   grew by more than 2^8; the epilogue normalises O_i and
//                   writes out / lse through shared-memory staging.
//     The MMA order per KV tile is PV_0, S_0(next), PV_1, S_1(next): while one
//     softmax warpgroup works, the tensor cores run the other tile's MMAs.
//   * Every mbarrier wait is bounded (wall-clock limit) and reports
//     FM_DEVERR_TIMEOUT in the workspace error word instead of hanging.
//
// Layouts: q [T][Hq][D], k/v [T][Hkv][D] bf16, viewed by TMA as 2-D tensors
// (rows = tokens, columns = heads * D) with 64-column (128-byte) boxes and
// 128-byte swizzle; tile rows start at arbitrary token offsets and read into
// the neighbouring sample (masked) or past T (zero fill).
#include <cuda_bf16.h>
#include <math_constants.h>

#include <cstring>

#include "attn_common.cuh"
#include "fm_device.cuh"
#include "fm_internal.h"
#include "rope_device.cuh"

namespace fm {
namespace {

// warps 0..3: K producer, MMA issuer(s), V producer; warps 4.. : one softmax
// warpgroup per Q tile of an item (warp w reads TMEM lanes 32*(w%4)..+31).
constexpr int kFirstSoftmaxWarp = 4;
constexpr int kTileM = 128;  // MMA M: TMEM lanes = tile rows
constexpr int kMetaSlots = 4;
// Interval-masked tiles whose columns form at most this many runs of equal
// (LTS, LTE, UTS, UTE) get a run table instead of per-column tests.
constexpr int kMaxRuns = 8;

// Shared-memory rings.  K and V tiles share one ring of kKVSlots slots,
// loaded in the order K(0), V(0), K(1), V(1), ... of the CTA's KV tiles
// (load p into slot p mod kKVSlots): with four slots K(t+2) takes the slot
// K(t) leaves once the S MMAs of tile t are done, and V(t+2) the one V(t)
// leaves after the PV MMAs of tile t.  Q tiles have their own ring of
// kQSlots tile buffers, filled in work order (tile 0, then tile 1 of each
// item); a buffer is reloaded once the tile held there before has had its
// last S MMA, so with two buffers the next item's tile 0 loads as soon as
// the current item's tile 0 has had its last S MMA, while the current item's
// last KV step still runs.
template <int BN>
constexpr int kKVSlots = 4;
template <int BN>
constexpr int kQSlots = (BN == 128) ? 2 : 4;
constexpr int kMaxKVSlots = 4;
constexpr int kMaxQSlots = 4;

// With 64-column key tiles TMEM holds two S buffers per Q tile (S_i of KV
// tile t+2 is computed into the buffer PV_i of tile t has just read, while
// the softmax works on tile t+1).  128-column key tiles fill TMEM with one S
// per Q tile.
//
// QT = Q tiles per work item (one softmax warpgroup each).  QT = 2 shares
// every K/V tile between two Q tiles; TMEM then holds two S buffers per Q
// tile only with 64-column key tiles.  QT = 1 leaves room for two
// 128-column S buffers, so the single softmax warpgroup never waits for its
// own tile's MMAs.
template <int BN, int QT>
constexpr int kSBufs = (QT == 1 || BN == 64) ? 2 : 1;

// MMA issuing warps: each Q tile has its own issuer (warps 1 and 3), so one
// tile's barrier waits never hold up the other tile's MMAs.
template <int QT>
constexpr int kIssuers = QT;

template <int QT>
constexpr int kThreads = 128 + 128 * QT;

// Q tiles per item for 128-column key tiles
constexpr int kQTilesBN128 = 2;

// One S buffer: the two issuers issue their blocks (PV_i of a tile and the
// next S_i) strictly in turn, Q tile 0 first, so the tensor pipe runs one
// tile's block after the other instead of interleaving them.
constexpr bool kIssueTurns = true;

// independent partial maxima per S row
constexpr int kMaxChains = 4;

enum : int { kFirst = 1, kLast = 2, kHasQ1 = 4, kStop = 8 };

struct TileMeta {
  int flags;       // kFirst | kLast | kHasQ1, or kStop
  int cls0, cls1;  // block class for Q tile 0 / Q tile 1
  int c0, c1;      // key columns [c0, c1)
  int r0, r_end;   // query rows of the item [r0, r_end); tile 1 starts at r0 + block_m
  int h, kvh;      // q head, key/value head
  int n_runs;      // partial tiles: runs of equal intervals in the run table, 0 = per column
  int a;           // first row of the sample (RoPE positions count from it)
  int qseq;        // Q ring position of the item's tile 0 (tile 1: qseq + 1)
  int pad[4];
};
static_assert(sizeof(TileMeta) == 64, "TileMeta is 64 bytes");

enum Bar : int {
  kKVFull = 0,                        // [kMaxKVSlots] K or V tile landed (TMA tx)
  kKVEmpty = kKVFull + kMaxKVSlots,   // [kMaxKVSlots] both issuers' MMAs done reading it
  kMFull = kKVEmpty + kMaxKVSlots,    // [kMetaSlots] tile metadata written
  kMEmpty = kMFull + kMetaSlots,      // [kMetaSlots] metadata consumed
  kQFull = kMEmpty + kMetaSlots,      // [kMaxQSlots] Q tile landed
  kQEmpty = kQFull + kMaxQSlots,      // [kMaxQSlots] last S MMA on it done (fused RoPE: and
                                      //   its 128 rows rotated and copied out)
  kSFull = kQEmpty + kMaxQSlots,      // [2 tiles][2 buffers] S_i ready
  kPFull = kSFull + 4,             // [2 tiles][2 buffers] P_i written (128 arrivals)
  kOFull = kPFull + 4,             // [2] last PV_i of the item done (one S buffer)
  kPVDone = kOFull + 2,            // [2 tiles][2 buffers] PV_i done (two S buffers)
  kOEmpty = kPVDone + 4,           // [2] O_i read by the epilogue (128 arrivals)
  kDrain = kOEmpty + 2,            // [2] an issuer's MMAs are all done
  kTurn = kDrain + 2,              // [2] issuer i may issue its next block
  kQRot = kTurn + 2,                  // [kMaxQSlots] Q tile rotated in place (128 arrivals)
  kNumBars = kQRot + kMaxQSlots
};

// arrivals on kMEmpty: the V producer lane, the MMA issuers and the softmax
// warps
template <int QT>
constexpr int kMEmptyCount = 1 + kIssuers<QT> + 4 * QT;

template <int D, int BN, int QT>
struct Layout {
  static constexpr int kQBytes = kTileM * D * 2;  // one Q tile
  static constexpr int kKVBytes = BN * D * 2;     // one K or V tile
  static constexpr int kQ = 0;                    // kQSlots Q tile buffers
  static constexpr int kKV = kQ + kQSlots<BN> * kQBytes;  // kKVSlots K/V slots
  static constexpr int kCols = kKV + kKVSlots<BN> * kKVBytes;  // int32 [kMetaSlots][4][BN]
  static constexpr int kMeta = kCols + kMetaSlots * 4 * BN * 4;
  // int32 [kMetaSlots][kMaxRuns][8]: start column, LTS, LTE, UTS, UTE of each run
  static constexpr int kRuns = kMeta + kMetaSlots * static_cast<int>(sizeof(TileMeta));
  // epilogue staging: per softmax warp, 32 rows x 32 bf16 columns (2 KB)
  static constexpr int kStage = kRuns + kMetaSlots * kMaxRuns * 8 * 4;
  static constexpr int kStageBytesPerWarp = 32 * 64;
  static constexpr int kBars = kStage + 4 * QT * kStageBytesPerWarp;
  static constexpr int kTmemSlot = kBars + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kEnd = kAbort + 4;
  static constexpr int kBytes = kEnd + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns: S_i of buffer b at (i*kSBufs + b)*BN (P_i packed into its
  // first BN/2 columns), O_i at 256 + i*128.
  __host__ __device__ static constexpr uint32_t s_col(int i, uint32_t b) {
    return static_cast<uint32_t>((i * kSBufs<BN, QT> + static_cast<int>(b)) * BN);
  }
  static_assert(QT * kSBufs<BN, QT> * BN <= 256, "S buffers fit below the O columns");
  static_assert(kKVSlots<BN> <= kMaxKVSlots && kQSlots<BN> <= kMaxQSlots, "ring sizes");
  static_assert(kQSlots<BN> >= QT, "an item's Q tiles fit in the ring");
  static_assert(BN <= 128 && D <= 128, "TMEM budget");
  static_assert(kBytes <= 232448, "shared memory budget");
};

// Classes of KV tile kt of sample s ([a, b)) for the two Q tiles of an item:
// rows [r0, r1) and [r1, r2) (the second is empty when r2 == r1).
template <int BN>
__device__ __forceinline__ void tile_classes(const AttnParams& p, int mh, int s, int a, int b,
                                             int r0, int r1, int r2, int kt, int kt_end,
                                             int& cls0, int& cls1) {
  cls0 = cls1 = kClsF;
  if (kt >= kt_end) return;
  const int c0 = a + kt * BN;
  const int c1 = min(c0 + BN, b);
  int st[8];
  const bool has_mask = p.sri != nullptr;
  if (has_mask) {
    const int64_t slot = static_cast<int64_t>(a / BN) + s + kt;
#pragma unroll
    for (int v = 0; v < 8; ++v)
      st[v] = __ldg(p.minmax + (static_cast<int64_t>(mh) * 8 + v) * p.n_kv_slots + slot);
  }
  const bool causal = p.causal != 0;
  cls0 = classify_block(r0, r1, c0, c1, st, has_mask, causal);
  if (r2 > r1) cls1 = classify_block(r1, r2, c0, c1, st, has_mask, causal);
}

// KV tiles to examine for rows ending at r_end (causal: up to the diagonal;
// every later tile is entirely above it and fully masked).
template <int BN>
__device__ __forceinline__ int kv_tiles_to_scan(const AttnParams& p, int a, int b, int r_end) {
  const int n_kv = (b - a + BN - 1) / BN;
  if (p.causal) return min(n_kv, (r_end - 1 - a) / BN + 1);
  return n_kv;
}

// ---------------------------------------------------------------------------
// planner: work unit = (sample, Q tile) for head pairs, else (sample, pair
// of consecutive Q tiles)
// ---------------------------------------------------------------------------

// Rows of item `pair` of the sample [a, b): Q tile 0 [r0, r1), Q tile 1
// [r1, r2) (empty when r2 == r1).  With QT = 2 and an odd number of Q tiles
// the sample's first tile is the one without a partner: items pair tiles
// (1, 2), (3, 4), ... from the back, so under a causal mask the tile that
// runs with one warpgroup only is the cheapest one, not the costliest.
template <int QT>
__device__ __forceinline__ void item_rows(int a, int b, int64_t pair, int bm, int& r0, int& r1,
                                          int& r2) {
  int64_t t0 = pair * QT;  // first Q tile of the item
  bool single = QT == 1;
  if constexpr (QT == 2) {
    const int64_t n_t = (static_cast<int64_t>(b) - a + bm - 1) / bm;
    if (n_t & 1) {
      single = pair == 0;
      t0 = pair == 0 ? 0 : 2 * pair - 1;
    }
  }
  r0 = static_cast<int>(min(static_cast<int64_t>(a) + t0 * bm, static_cast<int64_t>(b)));
  r1 = min(r0 + bm, b);
  r2 = single ? r1 : min(r0 + 2 * bm, b);
}

// Tile sizes and item form of a plan, as stored in the workspace header.
__device__ __forceinline__ int plan_tiles_word(const AttnParams& p) {
  return p.block_m | (p.block_n << 12) | (p.head_pairs << 24);
}

// Rows of the item of slot `tile` in head-pair form: one Q tile [r0, r1) for
// two q heads (r2 = r1: no second row range).
__device__ __forceinline__ void tile_rows(int a, int b, int64_t tile, int bm, int& r0, int& r1,
                                          int& r2) {
  r0 = static_cast<int>(min(static_cast<int64_t>(a) + tile * bm, static_cast<int64_t>(b)));
  r1 = min(r0 + bm, b);
  r2 = r1;
}

// The planner is two programmatic dependent launches (see launch_pdl): each
// waits for the kernel before it, then lets the next one start launching,
// so the attention kernel's set-up overlaps the planner.  Neither needs the
// workspace cleared: the cost kernel writes every slot, the order kernel
// builds its histogram on chip and initialises the whole header.

// One warp per slot: cost = number of blocks that are not fully masked,
// stored as cost * 2 + (the pair has a second Q tile), or -1 for a slot
// without a Q tile.
template <int BN, int QT>
__global__ void __launch_bounds__(256) plan_cost_kernel(const AttnParams p) {
  pdl_trigger();
  pdl_wait();
  const int64_t u = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (u >= p.n_qslots) return;
  const int T = static_cast<int>(p.T);
  const bool hpair = p.head_pairs != 0;
  const int BM2 = (hpair ? 1 : QT) * p.block_m;  // rows of one slot
  int lo = 0, hi = p.n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int64_t base = static_cast<int64_t>(clamp_tok(__ldg(p.cu + mid), T)) / BM2 + mid;
    if (base <= u) lo = mid; else hi = mid - 1;
  }
  const int s = lo;
  const int a = clamp_tok(__ldg(p.cu + s), T);
  const int b = max(a, clamp_tok(__ldg(p.cu + s + 1), T));
  const int64_t pair = u - (static_cast<int64_t>(a) / BM2 + s);
  if (pair < 0 || a + pair * BM2 >= b) {
    if (lane == 0) p.cost[u] = -1;
    return;
  }
  int r0, r1, r2;
  if (hpair)
    tile_rows(a, b, pair, p.block_m, r0, r1, r2);
  else
    item_rows<QT>(a, b, pair, p.block_m, r0, r1, r2);
  const int kt_end = kv_tiles_to_scan<BN>(p, a, b, r2);
  // With one mask per q head the pair's items differ in cost; the order
  // uses the costliest head's count (all heads of a pair run side by side).
  const int n_mh = p.hm > 1 ? p.hm : 1;
  int cost = 0;
  for (int mh = 0; mh < n_mh; ++mh) {
    int c = 0;
    for (int base = 0; base < kt_end; base += 32) {
      int c0, c1;
      tile_classes<BN>(p, mh, s, a, b, r0, r1, r2, base + lane, kt_end, c0, c1);
      c += __popc(__ballot_sync(0xffffffffu, c0 != kClsF));
      c += __popc(__ballot_sync(0xffffffffu, c1 != kClsF));
    }
    cost = max(cost, c);
  }
  if (lane == 0) {
    p.cost[u] = cost * 2 + (r2 > r1 ? 1 : 0);
    p.slot_info[u] = make_int2(s, static_cast<int>(pair));
  }
}

// One CTA: counting sort of the real slots by cost, largest first, and the
// workspace header (item counts, work counter, error word, timeout record).
__global__ void __launch_bounds__(kCostBins) plan_order_kernel(const AttnParams p) {
  __shared__ int hist[kCostBins];
  __shared__ int offs[kCostBins];
  __shared__ int warp_tot[kCostBins / 32];
  __shared__ int n_tiles;
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x;
  const int lane = tid & 31, w = tid >> 5;
  hist[tid] = 0;
  if (tid == 0) n_tiles = 0;
  __syncthreads();
  int my_tiles = 0;
  for (int64_t u = tid; u < p.n_qslots; u += kCostBins) {
    const int c = p.cost[u];
    if (c >= 0) {
      atomicAdd(&hist[min(c >> 1, kCostBins - 1)], 1);
      my_tiles += 1 + (c & 1);
    }
  }
  my_tiles = __reduce_add_sync(0xffffffffu, my_tiles);
  if (lane == 0 && my_tiles != 0) atomicAdd(&n_tiles, my_tiles);
  __syncthreads();
  // descending cost: position 0 holds the largest bin
  const int bin = kCostBins - 1 - tid;
  const int cnt = hist[bin];
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
  __syncthreads();
  for (int64_t u = tid; u < p.n_qslots; u += kCostBins) {
    const int c = p.cost[u];
    if (c >= 0) {
      const int pos = atomicAdd(&offs[min(c >> 1, kCostBins - 1)], 1);
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
  bad = __syncthreads_or(bad) != 0;
  if (tid == kCostBins - 1) {
    AttnWorkspaceHeader* hd = p.ws;
    hd->work_counter = 0u;
    hd->n_qtiles = n_tiles;
    hd->n_items = incl * (p.head_pairs ? p.hq / 2 : p.hq);
    hd->n_tile_items = n_tiles * p.hq;
    hd->error_word = bad ? static_cast<int>(FM_DEVERR_DATA) : 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) hd->diag[i] = 0;
    hd->exit_counter = 0u;
    hd->plan_T = static_cast<int32_t>(p.T);
    hd->plan_n_seqs = p.n_seqs;
    hd->plan_hq = p.hq;
    hd->plan_tiles = plan_tiles_word(p);
  }
}

// Masks columns [J0, J1) of an S row (mode 1: element bits, mode 2: columns
// from `valid` on) and folds them into C independent partial maxima.
template <int J0, int J1, int BN, int C>
__device__ __forceinline__ void mask_and_max(uint32_t (&sr)[BN], const uint32_t (&mbits)[BN / 32],
                                             int mode, int valid, float (&mc)[C]) {
  if (mode == 1) {
#pragma unroll
    for (int j = J0; j < J1; ++j)
      if ((mbits[j >> 5] >> (j & 31)) & 1u) sr[j] = __float_as_uint(-CUDART_INF_F);
  } else if (mode == 2) {
#pragma unroll
    for (int j = J0; j < J1; ++j)
      if (j >= valid) sr[j] = __float_as_uint(-CUDART_INF_F);
  }
#pragma unroll
  for (int j = J0; j < J1; j += 2)
    mc[(j >> 1) % C] = fmax3(mc[(j >> 1) % C], __uint_as_float(sr[j]), __uint_as_float(sr[j + 1]));
}

// Register split between the warpgroups with two Q tiles per item (all four
// warps of a warpgroup run the same instruction).  That kernel is launched
// with kThreads<2> x kLaunchRegs registers; kProducerRegs x 128 +
// kSoftmaxRegs x 256 must not exceed that, which the host checks against the
// compiled register count before launch.  With one Q tile (256 threads)
// every warp keeps the launch budget.
constexpr int kLaunchRegs = 168;
constexpr int kProducerRegs = 96;
constexpr int kSoftmaxRegs = 200;
static_assert(kProducerRegs * 128 + kSoftmaxRegs * 256 <= kThreads<2> * kLaunchRegs,
              "register split exceeds the launch budget");

__device__ __forceinline__ void regs_release() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
}
__device__ __forceinline__ void regs_acquire() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
}

// ---------------------------------------------------------------------------
// persistent attention kernel
// ---------------------------------------------------------------------------

// End of every role: all threads meet, then the warp that allocated TMEM frees it.
template <int D, int BN, int QT>
__device__ __forceinline__ void attn_teardown(uint32_t* tmem_slot, int warp) {
  tc_fence_before();
  asm volatile("bar.sync 1, %0;" ::"n"(kThreads<QT>) : "memory");
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(*reinterpret_cast<volatile uint32_t*>(tmem_slot), Layout<D, BN, QT>::kTmemCols);
  }
}

// Warps 0..3 (reduced register budget): K producer, MMA issuer, V producer
// and one idle warp; warp 0 initialises the barriers, warp 1 owns TMEM.
template <int D, int BN, int QT, typename IdxT, bool ROPE, bool HP>
__device__ __forceinline__ void attn_producer_roles(const AttnParams& p, const CUtensorMap& tq,
                                                    const CUtensorMap& tk,
                                                    const CUtensorMap& tv, const RopeArgs& ra) {
  using L = Layout<D, BN, QT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  TileMeta* meta = reinterpret_cast<TileMeta*>(smem + L::kMeta);
  int* cols = reinterpret_cast<int*>(smem + L::kCols);
  int* runs = reinterpret_cast<int*>(smem + L::kRuns);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = static_cast<int>(p.T);
  const int BM = p.block_m;
  const Sync sy{bars, abort_flag, p.timeout_ns, &p.ws->error_word, lane};
  if (threadIdx.x == 0) {
    for (int i = 0; i < kKVSlots<BN>; ++i) {
      mbar_init(&bars[kKVFull + i], 1);
      mbar_init(&bars[kKVEmpty + i], kIssuers<QT>);
    }
    for (int i = 0; i < kQSlots<BN>; ++i) {
      mbar_init(&bars[kQFull + i], 1);
      // the tile's issuer commits after its last S MMA; with the fused RoPE
      // the 128 threads that rotate (and copy out) the tile arrive as well
      mbar_init(&bars[kQEmpty + i], ROPE ? 1 + 128 : 1);
      mbar_init(&bars[kQRot + i], 128);
    }
    for (int i = 0; i < kMetaSlots; ++i) {
      mbar_init(&bars[kMFull + i], 1);
      mbar_init(&bars[kMEmpty + i], kMEmptyCount<QT>);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kOFull + i], 1);
      mbar_init(&bars[kOEmpty + i], 128);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars[kPVDone + i], 1);
      mbar_init(&bars[kSFull + i], 1);
      mbar_init(&bars[kPFull + i], 128);
    }
    mbar_init(&bars[kDrain], 1);
    mbar_init(&bars[kDrain + 1], 1);
    mbar_init(&bars[kTurn], 1);
    mbar_init(&bars[kTurn + 1], 1);
    *abort_flag = 0;
    mbar_fence_init();
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
  pdl_wait();  // the planner's tables and header (and q, k, v) are ready

  if (warp == 0) {
    // --------------------------------------------------- K producer + metadata
    int n_items = 0;
    {
      // A plan made for other sizes (or overwritten since) is not used; a
      // reused plan is not used either once a call on it has set an error
      // (its counters may not have been reset).  Either way no item runs.
      // two independent 16-byte loads: {work counter, Q tiles, items, error
      // word} and the plan's sizes
      const int4 h0 = *reinterpret_cast<const int4*>(p.ws);
      const int4 hp = *reinterpret_cast<const int4*>(&p.ws->plan_T);
      const bool fits = (hp.x == static_cast<int32_t>(p.T)) & (hp.y == p.n_seqs) &
                        (hp.z == p.hq) & (hp.w == plan_tiles_word(p));
      if (!fits) {
        if (lane == 0) atomicOr(&p.ws->error_word, static_cast<int>(FM_DEVERR_DATA));
      } else if (!(p.reuse_plan && h0.w != 0)) {
        const int64_t cap = p.n_qslots * p.hq;  // entries the order table can hold
        n_items = static_cast<int>(max(static_cast<int64_t>(0),
                                       min(static_cast<int64_t>(h0.z), cap)));
      }
    }
    const int group = p.hq / p.hkv;
    // head-pair items: one Q tile for q heads 2k and 2k + 1 (one key/value
    // head, one mask); otherwise two Q tiles of one q head
    constexpr bool hpair = HP;
    const int per_slot = hpair ? p.hq / 2 : p.hq;  // items per planner slot
    constexpr uint32_t NKV = kKVSlots<BN>, NQ = kQSlots<BN>;
    uint32_t kv_t = 0;               // KV tiles loaded (K(t) is ring load 2t)
    uint32_t mslot = 0, mround = 0;  // metadata ring
    uint32_t q_seq = 0;              // Q tiles loaded (Q ring position)
    uint32_t k_armed[kMaxKVSlots], q_armed[kMaxQSlots];  // ring position last armed, per slot
#pragma unroll
    for (int i = 0; i < kMaxKVSlots; ++i) k_armed[i] = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < kMaxQSlots; ++i) q_armed[i] = 0xffffffffu;
    long long cnt_p = 0, cnt_u = 0, cnt_f = 0;
    bool ok = true;

    auto push_meta = [&](int flags, int cls0, int cls1, int c0, int c1, int r0, int r_end, int h,
                         int kvh, bool copy_cols, int mh, int a, uint32_t qseq) -> bool {
      if (!sy.warp(kMEmpty + mslot, (mround & 1) ^ 1)) return false;
      int n_runs = 0;
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
        __syncwarp();
        // runs of equal interval quadruples among the columns inside the sample
        const int valid = c1 - c0;
        uint32_t run_start[BN / 32];
#pragma unroll
        for (int m = 0; m < BN / 32; ++m) {
          const int jj = m * 32 + lane;
          bool st = false;
          if (jj < valid) {
            st = jj == 0;
#pragma unroll
            for (int v = 0; v < 4; ++v) st |= jj > 0 && dst[v * BN + jj] != dst[v * BN + jj - 1];
          }
          run_start[m] = __ballot_sync(0xffffffffu, st);
          n_runs += __popc(run_start[m]);
        }
        if (n_runs > kMaxRuns) n_runs = 0;  // per-column tests instead
        if (n_runs > 0) {
          int* rt = runs + mslot * kMaxRuns * 8;
          int before = 0;
#pragma unroll
          for (int m = 0; m < BN / 32; ++m) {
            const uint32_t b = run_start[m];
            if ((b >> lane) & 1u) {
              const int k = before + __popc(b & ((1u << lane) - 1u));
              const int jj = m * 32 + lane;
              rt[k * 8 + 0] = jj;
#pragma unroll
              for (int v = 0; v < 4; ++v) rt[k * 8 + 1 + v] = dst[v * BN + jj];
            }
            before += __popc(b);
          }
        }
      }
      if (lane == 0) {
        TileMeta& m = meta[mslot];
        m.n_runs = n_runs;
        m.flags = flags;
        m.cls0 = cls0;
        m.cls1 = cls1;
        m.c0 = c0;
        m.c1 = c1;
        m.r0 = r0;
        m.r_end = r_end;
        m.h = h;
        m.kvh = kvh;
        m.a = a;
        m.qseq = static_cast<int>(qseq);
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

    // Q ring position u -> buffer u % NQ, once the MMAs (and, with the fused
    // RoPE, the rotation) of the tile held there before are done
    auto load_q = [&](uint32_t u, int h, int row0) -> bool {
      const uint32_t b = u % NQ;
      if (!sy.warp(kQEmpty + b, ((u / NQ) & 1u) ^ 1u)) return false;
      if (lane == 0) {
        uint8_t* qdst = smem + L::kQ + b * L::kQBytes;
        mbar_arrive_expect_tx(&bars[kQFull + b], L::kQBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(qdst + c * (kTileM * 128), &tq, &bars[kQFull + b], h * D + c * 64, row0);
      }
      q_armed[b] = u;
      return true;
    };

    while (ok) {
      int item = 0;
      if (lane == 0) item = static_cast<int>(atomicAdd(&p.ws->work_counter, 1u));
      item = __shfl_sync(0xffffffffu, item, 0);
      if (item >= n_items) {
        if (lane == 0) {
          // every CTA claims past the end exactly once; the last one to do
          // so resets the counters, so that the plan can be used again
          __threadfence();
          if (atomicAdd(&p.ws->exit_counter, 1u) == gridDim.x - 1u) {
            p.ws->work_counter = 0u;
            p.ws->exit_counter = 0u;
          }
        }
        ok = push_meta(kStop, kClsF, kClsF, 0, 0, 0, 0, 0, 0, false, 0, 0, 0u);
        break;
      }
      const int2 pi = p.order[item / per_slot];
      const int h = hpair ? 2 * (item % per_slot) : item % per_slot;
      // an entry the planner never writes becomes an empty item (no rows)
      const bool bad_entry = pi.x < 0 || pi.x >= p.n_seqs || pi.y < 0;
      if (bad_entry && lane == 0) atomicOr(&p.ws->error_word, static_cast<int>(FM_DEVERR_DATA));
      const int s = bad_entry ? 0 : pi.x;
      const int kvh = h / group;
      const int mh = p.hm > 1 ? h : 0;
      const int a = clamp_tok(__ldg(p.cu + s), T);
      const int b = max(a, clamp_tok(__ldg(p.cu + s + 1), T));
      int r0, r1, r2;
      if (hpair)
        tile_rows(a, b, bad_entry ? (1 << 30) : pi.y, BM, r0, r1, r2);
      else
        item_rows<QT>(a, b, bad_entry ? (1 << 30) : pi.y, BM, r0, r1, r2);
      // the item's second Q tile: the next q head's (head pairs) or the next
      // rows' (never with one Q tile per item)
      const bool has_q1 = hpair ? r1 > r0 : r2 > r1;
      const int n_kv = (b - a + BN - 1) / BN;
      const int kt_end = (r2 > r0) ? kv_tiles_to_scan<BN>(p, a, b, r2) : 0;

      // pass 1: block classes of both Q tiles (counts, number of live tiles)
      int n_live = 0;
      for (int base = 0; base < kt_end; base += 32) {
        int c0, c1;
        tile_classes<BN>(p, mh, s, a, b, r0, r1, r2, base + lane, kt_end, c0, c1);
        if (hpair) c1 = has_q1 ? c0 : kClsF;  // the same rows and mask
        n_live += __popc(__ballot_sync(0xffffffffu, c0 != kClsF || c1 != kClsF));
        const int p0 = __popc(__ballot_sync(0xffffffffu, c0 == kClsP || c0 == kClsPC));
        const int u0 = __popc(__ballot_sync(0xffffffffu, c0 == kClsU));
        const int p1 = __popc(__ballot_sync(0xffffffffu, c1 == kClsP || c1 == kClsPC));
        const int u1 = __popc(__ballot_sync(0xffffffffu, c1 == kClsU));
        cnt_p += p0 + p1;
        cnt_u += u0 + u1;
        cnt_f -= p0 + u0 + p1 + u1;
      }
      if (r2 > r0) cnt_f += static_cast<long long>(n_kv) * (has_q1 ? 2 : 1);

      if (n_live == 0) {
        // every key of these rows is masked: o = 0, lse = -inf (for both q
        // heads of a head-pair item)
        const int h_end = h + ((hpair && has_q1) ? 2 : 1);
        for (int hh = h; hh < h_end; ++hh) {
          for (int r = r0 + lane; r < r2; r += 32) {
            uint4* dst = reinterpret_cast<uint4*>(
                static_cast<__nv_bfloat16*>(p.out) +
                (static_cast<IdxT>(r) * p.hq + hh) * static_cast<IdxT>(D));
#pragma unroll
            for (int u = 0; u < D / 8; ++u) dst[u] = make_uint4(0u, 0u, 0u, 0u);
            p.lse[static_cast<IdxT>(hh) * static_cast<IdxT>(p.T) + r] = -CUDART_INF_F;
          }
          if constexpr (ROPE) {
            // no Q tile of these rows is loaded: rotate them from q directly
            if (ra.q_rot != nullptr) {
              constexpr int kG = D / 16;  // chunk pairs per row
              for (int idx = lane; idx < (r2 - r0) * kG; idx += 32) {
                const int r = r0 + idx / kG;
                const int g = idx % kG;
                const IdxT off = (static_cast<IdxT>(r) * p.hq + hh) * static_cast<IdxT>(D) + g * 8;
                const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(p.q) + off;
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(ra.q_rot) + off;
                const uint4 x1 = *reinterpret_cast<const uint4*>(src);
                const uint4 x2 = *reinterpret_cast<const uint4*>(src + D / 2);
                const float pos = static_cast<float>(r - a);
                float cs[8], sn[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  rope_cos_sin(pos, ra.freqs.hi[g * 8 + i], ra.freqs.lo[g * 8 + i], 1.0f, cs[i],
                               sn[i]);
                uint4 y1, y2;
                rope_rotate8(x1, x2, cs, sn, y1, y2);
                *reinterpret_cast<uint4*>(dst) = y1;
                *reinterpret_cast<uint4*>(dst + D / 2) = y2;
              }
            }
          }
        }
        continue;
      }

      // The item's Q tile 0 goes first, as soon as its buffer is free (the
      // tile held there before has had its last S MMA): nothing between the
      // classification and this load depends on it.
      if (!load_q(q_seq, h, r0)) {
        ok = false;
        break;
      }

      // pass 2: metadata and K for every tile live for either Q tile.  No
      // K/V tile is prefetched into L2 ahead of its load: with such
      // prefetches (two tiles ahead) the kernel measured up to 7 % slower
      // on the packed workloads.
      int pushed = 0;
      for (int base = 0; base < kt_end && ok; base += 32) {
        int my0, my1;
        tile_classes<BN>(p, mh, s, a, b, r0, r1, r2, base + lane, kt_end, my0, my1);
        if (hpair) my1 = has_q1 ? my0 : kClsF;
        uint32_t live = __ballot_sync(0xffffffffu, my0 != kClsF || my1 != kClsF);
        while (live != 0u) {
          const int l = __ffs(live) - 1;
          live &= live - 1u;
          const int cls0 = __shfl_sync(0xffffffffu, my0, l);
          const int cls1 = __shfl_sync(0xffffffffu, my1, l);
          const int c0 = a + (base + l) * BN;
          const int c1 = min(c0 + BN, b);
          const int flags = (pushed == 0 ? kFirst : 0) | (pushed == n_live - 1 ? kLast : 0) |
                            (has_q1 ? kHasQ1 : 0);
          const bool copy = (cls0 == kClsP || cls1 == kClsP) && p.sri != nullptr;
          if (!push_meta(flags, cls0, cls1, c0, c1, r0, r2, h, kvh, copy, mh, a, q_seq)) {
            ok = false;
            break;
          }
          // K of the tile; after the item's first K, its Q tile 1
          {
            const uint32_t pos = 2u * kv_t;  // K(t): even ring loads
            const uint32_t slot = pos % NKV;
            if (!sy.warp(kKVEmpty + slot, ((pos / NKV) & 1u) ^ 1u)) {
              ok = false;
              break;
            }
            if (lane == 0) {
              mbar_arrive_expect_tx(&bars[kKVFull + slot], L::kKVBytes);
#pragma unroll
              for (int c = 0; c < D / 64; ++c)
                tma_load_2d(smem + L::kKV + slot * L::kKVBytes + c * (BN * 128), &tk,
                            &bars[kKVFull + slot], kvh * D + c * 64, c0);
            }
            k_armed[slot] = pos;
            ++kv_t;
          }
          if (pushed == 0) {
            if (has_q1 && !load_q(q_seq + 1u, hpair ? h + 1 : h, hpair ? r0 : r0 + BM)) {
              ok = false;
              break;
            }
            q_seq += has_q1 ? 2u : 1u;
          }
          ++pushed;
        }
      }
    }
    if (!ok) {
      // let every TMA load this warp issued land before the CTA exits
      for (uint32_t st = 0; st < NKV; ++st)
        if (k_armed[st] != 0xffffffffu)
          mbar_wait_bounded(&bars[kKVFull + st], (k_armed[st] / NKV) & 1u, 100000000ull, nullptr);
      for (uint32_t qb = 0; qb < NQ; ++qb)
        if (q_armed[qb] != 0xffffffffu)
          mbar_wait_bounded(&bars[kQFull + qb], (q_armed[qb] / NQ) & 1u, 100000000ull, nullptr);
    }
    if (lane == 0 && p.class_counts != nullptr) {
      atomicAdd(reinterpret_cast<unsigned long long*>(p.class_counts + 0),
                static_cast<unsigned long long>(cnt_f));
      atomicAdd(reinterpret_cast<unsigned long long*>(p.class_counts + 1),
                static_cast<unsigned long long>(cnt_p));
      atomicAdd(reinterpret_cast<unsigned long long*>(p.class_counts + 2),
                static_cast<unsigned long long>(cnt_u));
    }
    attn_teardown<D, BN, QT>(tmem_slot, warp);
    return;
  } else if (warp == 2) {
    // --------------------------------------------------------------- V producer
    if (lane == 0) {
      constexpr uint32_t NKV = kKVSlots<BN>;
      uint32_t v_t = 0, mslot = 0, mround = 0;  // V(t) is ring load 2t + 1
      uint32_t v_armed[kMaxKVSlots];
#pragma unroll
      for (int i = 0; i < kMaxKVSlots; ++i) v_armed[i] = 0xffffffffu;
      bool ok = true;
      for (;;) {
        if (!sy.lone(kMFull + mslot, mround & 1)) { ok = false; break; }
        const int flags = *reinterpret_cast<volatile int*>(&meta[mslot].flags);
        const int c0 = *reinterpret_cast<volatile int*>(&meta[mslot].c0);
        const int kvh = *reinterpret_cast<volatile int*>(&meta[mslot].kvh);
        mbar_arrive(&bars[kMEmpty + mslot]);
        if (++mslot == kMetaSlots) {
          mslot = 0;
          ++mround;
        }
        if (flags & kStop) break;
        const uint32_t pos = 2u * v_t + 1u;
        const uint32_t slot = pos % NKV;
        if (!sy.lone(kKVEmpty + slot, ((pos / NKV) & 1u) ^ 1u)) { ok = false; break; }
        mbar_arrive_expect_tx(&bars[kKVFull + slot], L::kKVBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(smem + L::kKV + slot * L::kKVBytes + c * (BN * 128), &tv,
                      &bars[kKVFull + slot], kvh * D + c * 64, c0);
        v_armed[slot] = pos;
        ++v_t;
      }
      if (!ok) {
        for (uint32_t st = 0; st < NKV; ++st)
          if (v_armed[st] != 0xffffffffu)
            mbar_wait_bounded(&bars[kKVFull + st], (v_armed[st] / NKV) & 1u, 100000000ull,
                              nullptr);
      }
    }
    attn_teardown<D, BN, QT>(tmem_slot, warp);
    return;
  } else if (warp == 1 || (warp == 3 && QT == 2)) {
    // ----------------------------------------------------------------- MMA issuers
    // The whole warp runs this loop (every branch condition is warp-uniform);
    // MMAs and commits are issued by the lane elect.sync picks.  Both issuers
    // walk the same tile sequence (metadata, K and V rings); issuer `me`
    // issues only for Q tile `me` when there are two.
    {
      const int me = warp == 1 ? 0 : 1;
      constexpr uint32_t kIdescS = idesc_bf16_f32(kTileM, BN, false);
      constexpr uint32_t kIdescO = idesc_bf16_f32(kTileM, D, true);
      constexpr uint32_t NKV = kKVSlots<BN>, NQ = kQSlots<BN>;
      const uint32_t q_addr = smem_u32(smem + L::kQ);
      const uint32_t kv_addr = smem_u32(smem + L::kKV);
      uint32_t mslot = 0, mround = 0;  // metadata ring (released by the other readers)
      uint32_t k_t = 0, v_t = 0;       // KV tiles whose K / V this issuer has consumed
      uint32_t p_round[2] = {0u, 0u}, o_round[2] = {0u, 0u};
      bool o_pending[2] = {false, false};  // an epilogue of tile i has not been waited for
      bool ok = true;
      // K(t) is ring load 2t, V(t) ring load 2t + 1; load p sits in slot
      // p % NKV, and the phase of its full barrier has parity (p / NKV) & 1
      auto k_slot = [&]() -> uint32_t { return (2u * k_t) % NKV; };
      auto k_par = [&]() -> uint32_t { return ((2u * k_t) / NKV) & 1u; };
      auto v_slot = [&]() -> uint32_t { return (2u * v_t + 1u) % NKV; };
      auto v_par = [&]() -> uint32_t { return ((2u * v_t + 1u) / NKV) & 1u; };

      auto next_flags = [&](int& flags, int& qseq) -> bool {
        if (!sy.warp(kMFull + mslot, mround & 1)) return false;
        flags = *reinterpret_cast<volatile int*>(&meta[mslot].flags);
        qseq = *reinterpret_cast<volatile int*>(&meta[mslot].qseq);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kMEmpty + mslot]);
        if (++mslot == kMetaSlots) {
          mslot = 0;
          ++mround;
        }
        return true;
      };
      // Shared-memory descriptors are built once; an MMA step only adds a
      // constant to the start-address field (14 bits of addr >> 4, which no
      // offset inside the tile can overflow).
      const uint64_t q_desc0 = sdesc_sw128(q_addr, 16, 1024);
      const uint64_t k_desc0 = sdesc_sw128(kv_addr, 16, 1024);
      const uint64_t v_desc0 = sdesc_sw128(kv_addr, BN * 128, 1024);
      // S_i = Q_i K^T for the current K tile, Q tile buffer qb, into S buffer sb
      auto issue_s = [&](int i, uint32_t sb, uint32_t qb) {
        const uint32_t d_tmem = tmem_base + L::s_col(i, sb);
        const uint64_t qd = q_desc0 + static_cast<uint64_t>(qb * (L::kQBytes >> 4));
        const uint64_t kd = k_desc0 + static_cast<uint64_t>(k_slot() * (L::kKVBytes >> 4));
        constexpr int QC = (kTileM * 128) >> 4;  // next 64-column chunk of Q
        constexpr int KC = (BN * 128) >> 4;      // next 64-column chunk of K
        if constexpr (D == 128) {
          umma_ss_group8<2, 2, 4, 4, 6, 6, QC, KC, QC + 2, KC + 2, QC + 4, KC + 4, QC + 6, KC + 6>(
              d_tmem, qd, kd, kIdescS, 0u);
        } else {
          umma_ss_group4<2, 2, 4, 4, 6, 6>(d_tmem, qd, kd, kIdescS, 0u);
        }
      };
      // O_i (+)= P_i V for the current V tile, P_i in S buffer sb
      auto issue_pv = [&](int i, bool first, uint32_t sb) {
        const uint32_t d_tmem = tmem_base + 256 + i * 128;
        const uint32_t a_tmem = tmem_base + L::s_col(i, sb);
        const uint64_t vd = v_desc0 + static_cast<uint64_t>(v_slot() * (L::kKVBytes >> 4));
        constexpr int VS = (16 * 128) >> 4;  // 16 rows of V per K=16 step
        if constexpr (BN == 128) {
          umma_ts_group8<VS>(d_tmem, a_tmem, vd, kIdescO, first ? 0u : 1u);
        } else {
          umma_ts_group4<VS>(d_tmem, a_tmem, vd, kIdescO, first ? 0u : 1u);
        }
      };
      auto advance_k = [&]() { ++k_t; };
      auto advance_v = [&]() { ++v_t; };
      auto wait_o_empty = [&](int i, bool first) -> bool {
        if (first && o_pending[i]) {
          if (!sy.warp(kOEmpty + i, o_round[i] & 1)) return false;
          ++o_round[i];
          o_pending[i] = false;
        }
        return true;
      };

      if constexpr (kSBufs<BN, QT> == 2) {
        // The S stream fetches K(t+2) before PV(t) is issued, so K(t+2) must
        // not need V(t)'s slot: four slots (K and V alternate between two
        // pairs of them).
        static_assert(kKVSlots<BN> == 4, "two S buffers need four K/V slots");
        // Two S buffers per Q tile (i = me: this issuer's tile).  The S
        // stream runs two KV tiles ahead of the PV stream: for each tile t,
        // PV_i(t) is followed by S_i(t+2),
        // which overwrites the buffer PV_i(t) has just read (MMAs from one
        // thread run in issue order), so the softmax of tile t+1 never waits
        // for the MMAs of tile t.  Every buffer has its own S-full and P-full
        // barrier: a warpgroup may finish P(t+1) before P(t) is waited for.
        uint32_t qb = 0, qpar = 0;  // this issuer's Q tile of the S stream's item: buffer, parity
        uint32_t s_cnt[2] = {0u, 0u};           // S_i issued (buffer = s_cnt & 1)
        uint32_t pv_cnt[2] = {0u, 0u};          // PV_i issued (buffer = pv_cnt & 1)
        uint32_t fq = 0u;  // 4-bit flags of the (at most four) tiles with S issued, PV not yet
        uint32_t n_s = 0, n_pv = 0;
        bool s_end = false;
        bool rot_wait = false;  // fused RoPE: the fetched tile starts an item, Q not yet awaited
        // next tile of the S stream: its metadata, its item's Q buffer (first
        // tile of an item) and its K tile
        auto s_fetch = [&](int& flags) -> bool {
          int qseq = 0;
          if (!next_flags(flags, qseq)) return false;
          if (flags & kStop) {
            s_end = true;
            return true;
          }
          if (flags & kFirst) {
            const uint32_t u = static_cast<uint32_t>(qseq) + static_cast<uint32_t>(me);
            qb = u % NQ;
            qpar = (u / NQ) & 1u;
            if (me == 0 || (flags & kHasQ1)) {
              if constexpr (ROPE) {
                // the rotated Q is awaited right before the first S MMA: the
                // softmax rotates it only after its last P of the previous item
                rot_wait = true;
              } else {
                if (!sy.warp(kQFull + qb, qpar)) return false;
              }
            }
          }
          if (!sy.warp(kKVFull + k_slot(), k_par())) return false;
          tc_fence_after();
          return true;
        };
        auto s_one = [&](int i) -> bool {
          if constexpr (ROPE) {
            if (rot_wait) {
              if (!sy.warp(kQRot + qb, qpar)) return false;
              rot_wait = false;
              tc_fence_after();
            }
          }
          const uint32_t sb = s_cnt[i] & 1u;
          issue_s(i, sb, qb);
          umma_commit_elect(&bars[kSFull + 2 * i + sb]);
          ++s_cnt[i];
          return true;
        };
        auto s_done = [&](int flags) {
          rot_wait = false;
          umma_commit_elect(&bars[kKVEmpty + k_slot()]);
          if ((flags & kLast) && (me == 0 || (flags & kHasQ1)))
            umma_commit_elect(&bars[kQEmpty + qb]);
          advance_k();
          const uint32_t sh = (n_s & 3u) * 4u;
          fq = (fq & ~(0xFu << sh)) | (static_cast<uint32_t>(flags & 0xF) << sh);
          ++n_s;
        };
        for (int w = 0; w < 2 && ok && !s_end; ++w) {
          int f = 0;
          if (!s_fetch(f)) {
            ok = false;
            break;
          }
          if (s_end) break;
          if ((me == 0 || (f & kHasQ1)) && !s_one(me)) {
            ok = false;
            break;
          }
          s_done(f);
        }
        while (ok && n_pv < n_s) {
          const int cur = static_cast<int>((fq >> ((n_pv & 3u) * 4u)) & 0xFu);
          const bool first = (cur & kFirst) != 0;
          const bool last = (cur & kLast) != 0;
          int nxt = 0;
          bool ahead = false;
          if (!s_end) {
            if (!s_fetch(nxt)) { ok = false; break; }
            ahead = !s_end;
          }
          if (!sy.warp(kKVFull + v_slot(), v_par())) { ok = false; break; }
          {
            const int i = me;
            if (i == 0 || (cur & kHasQ1)) {
              const uint32_t sb = pv_cnt[i] & 1u;
              if (!wait_o_empty(i, first)) { ok = false; break; }
              if (!sy.warp(kPFull + 2 * i + sb, (pv_cnt[i] >> 1) & 1u)) { ok = false; break; }
              tc_fence_after();
              issue_pv(i, first, sb);
              umma_commit_elect(&bars[kPVDone + 2 * i + sb]);
              ++pv_cnt[i];
              if (last) o_pending[i] = true;
            }
            if (ahead && (i == 0 || (nxt & kHasQ1)) && !s_one(i)) { ok = false; break; }
          }
          umma_commit_elect(&bars[kKVEmpty + v_slot()]);
          advance_v();
          if (ahead) s_done(nxt);
          ++n_pv;
        }
      } else {
        // One S buffer per Q tile, one issuer per Q tile (i = me).  Per KV
        // tile: once P_i is in TMEM, PV_i and then S_i(next), which
        // overwrites the columns P_i occupies (MMAs from one thread run in
        // issue order).  K, V and Q stages are released when both issuers
        // have committed (their empty barriers count two arrivals).
        uint32_t turn_round = 0;
        // strict alternation of the issuers' blocks (issuer 0 goes first: its
        // first wait is on the phase before the barrier's first)
        auto take_turn = [&]() -> bool {
          if constexpr (kIssueTurns) {
            const uint32_t par = (me == 0) ? ((turn_round & 1u) ^ 1u) : (turn_round & 1u);
            if (!sy.warp(kTurn + me, par)) return false;
            ++turn_round;
          }
          return true;
        };
        auto pass_turn = [&]() {
          if constexpr (kIssueTurns) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kTurn + (me ^ 1)]);
          }
        };
        uint32_t my_qb = 0;  // Q tile buffer of this issuer's tile in the current item
        // S MMAs (all BN key columns) of the first tile of an item
        auto start_item = [&](int flags, int qseq) -> bool {
          const uint32_t u = static_cast<uint32_t>(qseq) + static_cast<uint32_t>(me);
          my_qb = u % NQ;
          const uint32_t qpar = (u / NQ) & 1u;
          const bool mine = me == 0 || (flags & kHasQ1);
          if (mine) {
            if constexpr (ROPE) {
              if (!sy.warp(kQRot + my_qb, qpar)) return false;
            } else {
              if (!sy.warp(kQFull + my_qb, qpar)) return false;
            }
          }
          if (!sy.warp(kKVFull + k_slot(), k_par())) return false;
          tc_fence_after();
          if (!take_turn()) return false;
          if (mine) {
            issue_s(me, 0u, my_qb);
            umma_commit_elect(&bars[kSFull + 2 * me]);
          }
          pass_turn();
          umma_commit_elect(&bars[kKVEmpty + k_slot()]);
          if ((flags & kLast) && mine) umma_commit_elect(&bars[kQEmpty + my_qb]);
          advance_k();
          return true;
        };
        int cur = 0, cur_qseq = 0;
        ok = next_flags(cur, cur_qseq);
        if (ok && !(cur & kStop)) ok = start_item(cur, cur_qseq);
        while (ok && !(cur & kStop)) {
          const bool first = (cur & kFirst) != 0;
          const bool last = (cur & kLast) != 0;
          const bool q1 = (cur & kHasQ1) != 0;
          int nxt = 0;
          if (!sy.warp(kKVFull + v_slot(), v_par())) { ok = false; break; }
          if (!last) {
            if (!sy.warp(kKVFull + k_slot(), k_par())) { ok = false; break; }
            tc_fence_after();
            // the metadata of this K tile was written before its load was armed
            nxt = *reinterpret_cast<volatile int*>(&meta[mslot].flags);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kMEmpty + mslot]);
            if (++mslot == kMetaSlots) {
              mslot = 0;
              ++mround;
            }
          }
          if (!(me == 0 || q1)) {
            // no block for this tile: keep the alternation
            if (!take_turn()) { ok = false; break; }
            pass_turn();
          }
          if (me == 0 || q1) {
            const int i = me;
            if (!wait_o_empty(i, first)) { ok = false; break; }
            if (!sy.warp(kPFull + 2 * i, p_round[i] & 1)) { ok = false; break; }
            ++p_round[i];
            tc_fence_after();
            if (!take_turn()) { ok = false; break; }
            issue_pv(i, first, 0u);
            if (last) {
              umma_commit_elect(&bars[kOFull + i]);
              o_pending[i] = true;
            } else {
              issue_s(i, 0u, my_qb);
              umma_commit_elect(&bars[kSFull + 2 * i]);
            }
            pass_turn();
          }
          umma_commit_elect(&bars[kKVEmpty + v_slot()]);
          advance_v();
          if (!last) {
            umma_commit_elect(&bars[kKVEmpty + k_slot()]);
            if ((nxt & kLast) && (me == 0 || q1)) umma_commit_elect(&bars[kQEmpty + my_qb]);
            advance_k();
          } else {
            int nq = 0;
            if (!next_flags(nxt, nq)) { ok = false; break; }
            if (nxt & kStop) break;
            if (!start_item(nxt, nq)) { ok = false; break; }
          }
          cur = nxt;
        }
      }
      // all issued MMAs complete before TMEM is released
      umma_commit_elect(&bars[kDrain + me]);
      mbar_wait_bounded(&bars[kDrain + me], 0, 100000000ull, nullptr);
    }
    attn_teardown<D, BN, QT>(tmem_slot, warp);
    return;
  } else {
    attn_teardown<D, BN, QT>(tmem_slot, warp);  // idle warp
  }
}

// Warps 4..11 (raised register budget): softmax of Q tile 0 (warps 4..7) and
// of Q tile 1 (warps 8..11).
// Fused RoPE: rotates row `row` of a Q tile in shared memory (128-byte
// swizzle: 16-byte chunk j of row r sits at chunk j ^ (r & 7) of the row's
// 128 bytes; channels [0, 64) in the first 64-column box, [64, 128) in the
// second).  The row holds a token at position `pos` of its sample.
template <int D>
__device__ __forceinline__ void rope_q_tile_row(const RopeArgs& ra, uint32_t tile, int row,
                                                float pos) {
  constexpr int kG = D / 16;  // chunk pairs per row
  const uint32_t row_addr = tile + static_cast<uint32_t>(row) * 128u;
  const uint32_t sw = static_cast<uint32_t>(row & 7);
#pragma unroll 2
  for (int g = 0; g < kG; ++g) {
    const int g2 = g + kG;
    const uint32_t a1 = row_addr + (g >> 3) * (kTileM * 128) + (((g & 7) ^ sw) << 4);
    const uint32_t a2 = row_addr + (g2 >> 3) * (kTileM * 128) + (((g2 & 7) ^ sw) << 4);
    const uint4 x1 = ld_shared_v4(a1);
    const uint4 x2 = ld_shared_v4(a2);
    float cs[8], sn[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      rope_cos_sin(pos, ra.freqs.hi[g * 8 + i], ra.freqs.lo[g * 8 + i], 1.0f, cs[i], sn[i]);
    uint4 y1, y2;
    rope_rotate8(x1, x2, cs, sn, y1, y2);
    st_shared_v4(a1, y1.x, y1.y, y1.z, y1.w);
    st_shared_v4(a2, y2.x, y2.y, y2.z, y2.w);
  }
}

// Copies rows [0, n_rows) of a rotated Q tile from shared memory to
// q_rot[t0 + row][h] with the 128 threads of a warpgroup (thread `tid`):
// consecutive threads take consecutive 16-byte chunks of a row, so every
// warp store covers whole rows.
template <int D, typename IdxT>
__device__ __forceinline__ void store_q_tile(const AttnParams& p, const RopeArgs& ra,
                                             uint32_t tile, int tid, int n_rows, int t0, int h) {
  constexpr int kC = D / 8;  // 16-byte chunks per row
  __nv_bfloat16* base = static_cast<__nv_bfloat16*>(ra.q_rot);
  for (int e = tid; e < n_rows * kC; e += 128) {
    const int row = e / kC;
    const int c = e % kC;
    const uint32_t src =
        tile + (c >> 3) * (kTileM * 128) + row * 128 + (((c & 7) ^ (row & 7)) << 4);
    const uint4 x = ld_shared_v4(src);
    *reinterpret_cast<uint4*>(base + (static_cast<IdxT>(t0 + row) * p.hq + h) *
                                         static_cast<IdxT>(D) + c * 8) = x;
  }
}

template <int D, int BN, int QT, typename IdxT, bool ROPE, bool HP>
__device__ __forceinline__ void attn_softmax_role(const AttnParams& p, const RopeArgs& ra) {
  using L = Layout<D, BN, QT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  TileMeta* meta = reinterpret_cast<TileMeta*>(smem + L::kMeta);
  int* cols = reinterpret_cast<int*>(smem + L::kCols);
  const int* runs = reinterpret_cast<const int*>(smem + L::kRuns);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int BM = p.block_m;
  const Sync sy{bars, abort_flag, p.timeout_ns, &p.ws->error_word, lane};
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  {
    // ------------------------------------------------------------------ softmax
    const int wg = (warp - kFirstSoftmaxWarp) >> 2;  // which Q tile of the item
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t o_tmem = tmem_base + lane_addr + 256 + wg * 128;
    const float scale_log2 = p.scale_log2;
    const bool causal = p.causal != 0;
    uint32_t mslot = 0, mround = 0;
    uint32_t n_tiles = 0, o_round = 0;  // KV tiles of this warpgroup so far; epilogues
    float m_run = -CUDART_INF_F, l_run = 0.f;
    int rt0 = 0, rt1 = 0, h = 0;
    constexpr uint32_t NQ = kQSlots<BN>;
    uint32_t item_qb = 0, item_qpar = 0;  // fused RoPE: Q tile buffer of this item, its parity

    // Epilogue of an item: once its last PV is done, O / l -> bf16 out rows
    // (guarded: rows from e_rt1 on belong to the next sample) and lse.
    // `wait_bar` / `wait_par`: the barrier phase of that last PV.
    // Each warp stages its 32 rows 32 columns at a time in shared memory
    // (16-byte chunk u of row r at chunk u ^ ((r >> 1) & 3) of the row's 64
    // bytes: conflict-free both ways) and stores them 8 rows per instruction,
    // 64 contiguous bytes per row, instead of one 16-byte piece of 32
    // different rows per instruction.
    auto epilogue = [&](int e_r, int e_rt1, int e_h, float e_m, float e_l, int wait_bar,
                        uint32_t wait_par) -> bool {
      if (!sy.warp(wait_bar, wait_par)) return false;
      tc_fence_after();
      const uint32_t stage =
          smem_u32(smem + L::kStage) +
          static_cast<uint32_t>(((threadIdx.x >> 5) - kFirstSoftmaxWarp) * L::kStageBytesPerWarp);
      const float inv_l = (e_l > 0.f) ? 1.f / e_l : 0.f;
      const uint64_t inv_l2 = pack_f32x2(inv_l, inv_l);
      {
        const int tok0 = e_r - lane;  // token of this warp's first row
        // rows of this warp: one 64-bit base, 32-bit offsets (32 * Hq * D fits)
        __nv_bfloat16* const dst0 = static_cast<__nv_bfloat16*>(p.out) +
                                    (static_cast<IdxT>(tok0) * p.hq + e_h) * static_cast<IdxT>(D);
        const int row_elems = p.hq * D;
        const uint32_t my_row = stage + static_cast<uint32_t>(lane) * 64u;
        const uint32_t my_sw = static_cast<uint32_t>((lane >> 1) & 3);
        // the whole O row with one TMEM load and one wait (the S row is dead)
        uint32_t orow[D];
        tmem_ld_row<D>(o_tmem, orow);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          const uint32_t* rr = orow + c * 32;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            st_shared_v4(my_row + ((static_cast<uint32_t>(u) ^ my_sw) << 4),
                         scale_pack_bf16x2(rr[8 * u + 0], rr[8 * u + 1], inv_l2),
                         scale_pack_bf16x2(rr[8 * u + 2], rr[8 * u + 3], inv_l2),
                         scale_pack_bf16x2(rr[8 * u + 4], rr[8 * u + 5], inv_l2),
                         scale_pack_bf16x2(rr[8 * u + 6], rr[8 * u + 7], inv_l2));
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int rl = 8 * i + (lane >> 2);  // row within the warp's 32
            const uint32_t u = static_cast<uint32_t>(lane & 3);
            const uint4 v = ld_shared_v4(stage + static_cast<uint32_t>(rl) * 64u +
                                         ((u ^ static_cast<uint32_t>((rl >> 1) & 3)) << 4));
            if (tok0 + rl < e_rt1)
              *reinterpret_cast<uint4*>(dst0 + (rl * row_elems + c * 32 + static_cast<int>(u) * 8)) = v;
          }
          __syncwarp();
        }
      }
      if (e_r < e_rt1) {
        p.lse[static_cast<IdxT>(e_h) * static_cast<IdxT>(p.T) + e_r] =
            (e_l > 0.f) ? (e_m + __log2f(e_l)) * 0.69314718055994531f : -CUDART_INF_F;
      }
      tc_fence_before();
      mbar_arrive(&bars[kOEmpty + wg]);
      return true;
    };
    // Fused RoPE defers an item's epilogue until the next item's Q tile is
    // rotated.  With two S buffers this is required: the MMA issuer waits for
    // that Q before it issues the item's last PV, which the epilogue waits
    // for.  With one it lets the rotation overlap the last PV and the next
    // S MMAs overlap the epilogue.  Until then h, rt0, rt1, m_run and l_run
    // still hold the item's values; its last tile is tile n_tiles - 1 of this
    // warpgroup.
    constexpr bool kDefer = ROPE;
    bool epi_pending = false;
    auto flush_epilogue = [&]() -> bool {
      if (!epi_pending) return true;
      epi_pending = false;
      const uint32_t lt = n_tiles - 1u;
      if constexpr (kSBufs<BN, QT> == 2)
        return epilogue(rt0 + row, rt1, h, m_run, l_run, kPVDone + 2 * wg + (lt & 1u),
                        (lt >> 1) & 1u);
      else
        return epilogue(rt0 + row, rt1, h, m_run, l_run, kOFull + wg, (o_round - 1u) & 1u);
    };

    for (;;) {
      if (!sy.warp(kMFull + mslot, mround & 1)) break;
      // the slot's first 32 bytes, {flags, cls0, cls1, c0} and {c1, r0,
      // r_end, h}, in two loads (ordered after the acquiring wait above)
      const int4 ma = *reinterpret_cast<const int4*>(meta + mslot);
      const int4 mb = *(reinterpret_cast<const int4*>(meta + mslot) + 1);
      const int flags = ma.x;
      if (flags & kStop) {
        if constexpr (kDefer) flush_epilogue();
        break;
      }
      const int cls = wg == 0 ? ma.y : ma.z;
      const int c0 = ma.w;
      const int c1 = mb.x;
      const bool first = (flags & kFirst) != 0;
      // the item's q head and rows (taken over once a deferred epilogue of
      // the previous item is done)
      int n_h = h, n_rt0 = rt0, n_rt1 = rt1;
      if (first) {
        // head pairs: the same rows, head h + wg; otherwise rows r0 + wg * BM
        n_h = mb.w + (HP ? wg : 0);
        n_rt0 = mb.y + (HP ? 0 : wg * BM);
        n_rt1 = min(n_rt0 + BM, mb.z);
        if constexpr (ROPE) {
          // the Q ring position of this warpgroup's tile (read before the
          // slot is released below)
          const uint32_t u = static_cast<uint32_t>(meta[mslot].qseq) + static_cast<uint32_t>(wg);
          item_qb = u % NQ;
          item_qpar = (u / NQ) & 1u;
        }
        if constexpr (!ROPE) {
          h = n_h;
          rt0 = n_rt0;
          rt1 = n_rt1;
        }
      }
      const uint32_t cur_slot = mslot;
      if (++mslot == kMetaSlots) {
        mslot = 0;
        ++mround;
      }
      if (wg == 1 && !(flags & kHasQ1)) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kMEmpty + cur_slot]);
        if constexpr (kDefer) {
          if (!flush_epilogue()) break;
        }
        continue;
      }
      if constexpr (ROPE) {
        if (first) {
          // this warpgroup's Q tile of the item: rotate it in place once it
          // has landed, then hand it to the tensor cores
          const int a_start = meta[cur_slot].a;
          const uint32_t qtile = smem_u32(smem + L::kQ + item_qb * L::kQBytes);
          if (!sy.warp(kQFull + item_qb, item_qpar)) break;
          rope_q_tile_row<D>(ra, qtile, row, static_cast<float>(max(n_rt0 + row - a_start, 0)));
          fence_proxy_async_smem();
          const int rb = kQRot + static_cast<int>(item_qb);
          mbar_arrive(&bars[rb]);
          if (ra.q_rot != nullptr) {
            // every row of the tile is rotated once the phase completes; the
            // buffer is refilled only after the arrival below
            if (!sy.warp(rb, item_qpar)) break;
            store_q_tile<D, IdxT>(p, ra, qtile, row, n_rt1 - n_rt0, n_rt0, n_h);
          }
          // this thread is done with the buffer (the issuer's commit after the
          // item's last S MMA completes its empty phase)
          mbar_arrive(&bars[kQEmpty + item_qb]);
          if constexpr (kDefer) {
            if (!flush_epilogue()) break;
          }
          h = n_h;
          rt0 = n_rt0;
          rt1 = n_rt1;
        }
      }
      if (first) {
        m_run = -CUDART_INF_F;
        l_run = 0.f;
      }
      const int r = rt0 + row;
      const int valid = c1 - c0;  // columns inside the sample
      uint32_t mbits[BN / 32];    // element mask of a partially masked block
      if (cls == kClsPC) {
        // causal diagonal: column c0 + jj is masked iff it lies above row r
        // or outside the sample; 32 columns at a time with shifts
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          const int d = r - (c0 + c * 32);  // columns jj - 32c > d are above the row
          const uint32_t above = d >= 31 ? 0u : (d < 0 ? 0xffffffffu : (0xffffffffu << (d + 1)));
          const int v = valid - c * 32;     // columns from v on are outside the sample
          const uint32_t out = v >= 32 ? 0u : (v <= 0 ? 0xffffffffu : (0xffffffffu << v));
          mbits[c] = above | out;
        }
      } else if (cls == kClsP && meta[cur_slot].n_runs > 0) {
        // the same rule over runs of columns with equal intervals: each run
        // [s, e) splits at the diagonal into a lower part (masked iff
        // LTS <= r < LTE) and an upper part (masked iff causal or
        // UTS <= r < UTE); columns from `valid` on are outside the sample
        const int n_runs = meta[cur_slot].n_runs;
        const int* rt = runs + cur_slot * kMaxRuns * 8;
        const int rr = r - c0 + 1;  // columns below rr are on or below the diagonal
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) mbits[c] = range_bits(valid, BN, c);
        for (int k = 0; k < n_runs; ++k) {
          const int4 ra = *reinterpret_cast<const int4*>(rt + k * 8);  // start, LTS, LTE, UTS
          const int ute = rt[k * 8 + 4];
          const int e = (k + 1 < n_runs) ? rt[(k + 1) * 8] : valid;
          const bool lm = (ra.y <= r) & (r < ra.z);
          const bool um = causal | ((ra.w <= r) & (r < ute));
          const int mid = min(max(rr, ra.x), e);  // [s, mid) lower, [mid, e) upper
#pragma unroll
          for (int c = 0; c < BN / 32; ++c)
            mbits[c] |= (lm ? range_bits(ra.x, mid, c) : 0u) | (um ? range_bits(mid, e, c) : 0u);
        }
      } else if (cls == kClsP) {
        // column intervals: row r is masked in column j iff it lies in
        // [LTS_j, LTE_j) on or below the diagonal, or above the diagonal and
        // (causal or in [UTS_j, UTE_j)); branch-free, four columns per load
        const int* cl = cols + cur_slot * 4 * BN;
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t bits = 0;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const int jj = c * 32 + i;
            const int4 lts = *reinterpret_cast<const int4*>(cl + jj);
            const int4 lte = *reinterpret_cast<const int4*>(cl + BN + jj);
            const int4 uts = *reinterpret_cast<const int4*>(cl + 2 * BN + jj);
            const int4 ute = *reinterpret_cast<const int4*>(cl + 3 * BN + jj);
            const int a[4] = {lts.x, lts.y, lts.z, lts.w};
            const int e[4] = {lte.x, lte.y, lte.z, lte.w};
            const int ua[4] = {uts.x, uts.y, uts.z, uts.w};
            const int ue[4] = {ute.x, ute.y, ute.z, ute.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const bool lower = r >= c0 + jj + t;
              const bool in_lt = (a[t] <= r) & (r < e[t]);
              const bool in_ut = causal | ((ua[t] <= r) & (r < ue[t]));
              const bool m = (jj + t >= valid) | (lower ? in_lt : in_ut);
              bits |= static_cast<uint32_t>(m) << (i + t);
            }
          }
          mbits[c] = bits;
        }
      }
      // metadata and mask columns of this tile are no longer needed
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kMEmpty + cur_slot]);

      // S buffer of this tile and the parity of its S-full / P-full phase
      const uint32_t sb = n_tiles % kSBufs<BN, QT>;
      const uint32_t spar = (n_tiles / kSBufs<BN, QT>) & 1u;
      const uint32_t s_cur = tmem_base + lane_addr + L::s_col(wg, sb);
      if (!sy.warp(kSFull + 2 * wg + sb, spar)) break;
      tc_fence_after();

      bool o_ok = true;
      if (cls == kClsF) {
        // live only for the other Q tile: contributes nothing, P = 0
        uint32_t z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_st16(s_cur + c * 16, z);
        tmem_st_wait();
      } else {
        // the whole S row in registers: one TMEM load, one wait
        uint32_t sr[BN];
        const int mmode = (cls == kClsP || cls == kClsPC) ? 1 : (valid < BN ? 2 : 0);
        float mc[kMaxChains];
#pragma unroll
        for (int i = 0; i < kMaxChains; ++i) mc[i] = -CUDART_INF_F;
        tmem_ld_row<BN>(s_cur, sr);
        // masked elements to -inf, row max (two new elements per three-input max)
        mask_and_max<0, BN>(sr, mbits, mmode, valid, mc);
        float mt = mc[0];
#pragma unroll
        for (int i = 1; i < kMaxChains; ++i) mt = fmaxf(mt, mc[i]);
        // scores in the log2 domain: x = s * scale * log2(e)
        const float mt2 = mt * scale_log2;
        const float m_new = fmaxf(m_run, mt2);
        // keep the old reference max unless it grew by more than 2^8
        const bool resc = first || (m_new > m_run + 8.0f);
        float factor = 1.f;
        float m_ref = m_run;
        if (resc) {
          factor = (m_run == -CUDART_INF_F) ? 0.f : ex2_approx(m_run - m_new);
          m_ref = m_new;
        }
        const bool need_o = resc && !first && (m_run != -CUDART_INF_F);
        if (resc) l_run = first ? 0.f : l_run * factor;
        m_run = m_ref;

        if (__any_sync(0xffffffffu, need_o)) {
          // rescale O before this tile's P reaches a PV MMA.  One S buffer:
          // the previous PV completed before S, which was issued after it.
          // Two S buffers: S was issued before the previous PV, so wait for
          // that PV here.  Its done barrier belongs to its S buffer; the
          // barrier's previous phase (the PV two tiles back) completed before
          // this tile's S, so the parity is exact.
          if constexpr (kSBufs<BN, QT> == 2) {
            const uint32_t pt = n_tiles - 1u;
            o_ok = sy.warp(kPVDone + 2 * wg + (pt & 1u), (pt >> 1) & 1u);
            tc_fence_after();
          }
          if (o_ok) {
            const float f = need_o ? factor : 1.f;
            // 16 columns at a time: the S row is still live in registers
#pragma unroll 1
            for (int c = 0; c < D / 16; ++c) {
              uint32_t rr[16];
              tmem_ld16(o_tmem + c * 16, rr);
#pragma unroll
              for (int i = 0; i < 16; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * f);
              tmem_st16(o_tmem + c * 16, rr);
            }
            tmem_st_wait();
          }
        }
        const float neg_base = (m_ref == -CUDART_INF_F) ? 0.f : -m_ref;
        const uint64_t scale2 = pack_f32x2(scale_log2, scale_log2);
        const uint64_t base2 = pack_f32x2(neg_base, neg_base);
        uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};  // eight partial row sums
        // P = 2^(x - m) as bf16 into the first half of the S columns
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const int j = c * 32 + i;
            pk[i >> 1] = exp2_pair_bf16(sr[j], sr[j + 1], scale2, base2, sum2[(i >> 1) & 3]);
          }
          tmem_st16(s_cur + c * 16, pk);
        }
        tmem_st_wait();
        l_run += (sum_f32x2(sum2[0]) + sum_f32x2(sum2[1])) + (sum_f32x2(sum2[2]) + sum_f32x2(sum2[3]));
      }
      if (!o_ok) break;
      tc_fence_before();
      mbar_arrive(&bars[kPFull + 2 * wg + sb]);

      if (flags & kLast) {
        // O_i is final once the PV of this tile is done (MMAs complete in
        // issue order, so every earlier PV is done too)
        int wbar;
        uint32_t wpar;
        if constexpr (kSBufs<BN, QT> == 2) {
          wbar = kPVDone + 2 * wg + sb;
          wpar = spar;
        } else {
          wbar = kOFull + wg;
          wpar = o_round & 1;
        }
        ++o_round;
        if constexpr (kDefer) {
          epi_pending = true;
        } else {
          if (!epilogue(r, rt1, h, m_run, l_run, wbar, wpar)) break;
        }
      }
      ++n_tiles;
    }
    attn_teardown<D, BN, QT>(tmem_slot, warp);
  }
}

template <int D, int BN, int QT, typename IdxT, bool ROPE, bool HP>
__global__ void __launch_bounds__(kThreads<QT>, 1)
    attn_fwd_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tq,
                    const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv,
                    const __grid_constant__ RopeArgs ra) {
  // The register split comes first so that no value crosses from one budget
  // into the other.
  if ((threadIdx.x >> 5) < 4) {
    if constexpr (QT == 2) regs_release();
    attn_producer_roles<D, BN, QT, IdxT, ROPE, HP>(p, tq, tk, tv, ra);
  } else {
    if constexpr (QT == 2) regs_acquire();
    attn_softmax_role<D, BN, QT, IdxT, ROPE, HP>(p, ra);
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

template <int BN, int QT>
cudaError_t launch_plan(const AttnParams& p, cudaStream_t stream) {
  cudaError_t e = launch_pdl(plan_cost_kernel<BN, QT>,
                             dim3(static_cast<unsigned>((p.n_qslots + 7) / 8)), dim3(256), 0,
                             stream, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(plan_order_kernel, dim3(1), dim3(kCostBins), 0, stream, p);
}

template <int D, int BN, int QT, typename IdxT, bool ROPE, bool HP>
cudaError_t launch_typed(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const RopeArgs& ra, int num_sms,
                         cudaStream_t stream) {
  using L = Layout<D, BN, QT>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static unsigned long long configured = 0ull;  // one bit per device; setting twice is harmless
  if (dev >= 64 || !((configured >> dev) & 1ull)) {
    // The warpgroups' register split must fit in what the launch allocates,
    // or setmaxnreg.inc would wait forever: refuse to launch otherwise.
    cudaFuncAttributes attr;
    e = cudaFuncGetAttributes(&attr, attn_fwd_kernel<D, BN, QT, IdxT, ROPE, HP>);
    if (e != cudaSuccess) return e;
    if (QT == 2 && attr.numRegs * kThreads<QT> < kProducerRegs * 128 + kSoftmaxRegs * 256)
      return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(attn_fwd_kernel<D, BN, QT, IdxT, ROPE, HP>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured |= 1ull << dev;
  }
  const int64_t n_slots = p.n_qslots;
  if (!p.reuse_plan) {
    e = launch_plan<BN, QT>(p, stream);
    if (e != cudaSuccess) return e;
  }
  const int64_t max_items = n_slots * p.hq;
  const int grid = static_cast<int>(max_items < num_sms ? max_items : num_sms);
  return launch_pdl(attn_fwd_kernel<D, BN, QT, IdxT, ROPE, HP>, dim3(grid), dim3(kThreads<QT>),
                    L::kBytes, stream, p, tq, tk, tv, ra);
}

}  // namespace

size_t attn_workspace_bytes(int64_t T, int n_seqs, int block_m) {
  const int64_t n_qslots = T / block_m + n_seqs;
  size_t bytes = sizeof(AttnWorkspaceHeader);
  bytes += static_cast<size_t>(n_qslots) * (sizeof(int) + 2 * sizeof(int2));
  return (bytes + 255) & ~static_cast<size_t>(255);
}

namespace {

// HP: work items of one Q tile for two q heads (head pairs), else two Q
// tiles of one q head.
template <bool ROPE, bool HP>
cudaError_t launch_attn_dispatch_hp(const AttnParams& p, const CUtensorMap& tq,
                                    const CUtensorMap& tk, const CUtensorMap& tv,
                                    const RopeArgs& ra, bool use_int64, int num_sms,
                                    cudaStream_t stream) {
  constexpr int Q2 = kQTilesBN128;
  if (p.head_dim == 128) {
    if (p.block_n == 128)
      return use_int64 ? launch_typed<128, 128, Q2, int64_t, ROPE, HP>(p, tq, tk, tv, ra, num_sms, stream)
                       : launch_typed<128, 128, Q2, int32_t, ROPE, HP>(p, tq, tk, tv, ra, num_sms, stream);
    return use_int64 ? launch_typed<128, 64, 2, int64_t, ROPE, HP>(p, tq, tk, tv, ra, num_sms, stream)
                     : launch_typed<128, 64, 2, int32_t, ROPE, HP>(p, tq, tk, tv, ra, num_sms, stream);
  }
  if (p.block_n == 128)
    return use_int64 ? launch_typed<64, 128, Q2, int64_t, ROPE, HP>(p, tq, tk, tv, ra, num_sms, stream)
                     : launch_typed<64, 128, Q2, int32_t, ROPE, HP>(p, tq, tk, tv, ra, num_sms, stream);
  return use_int64 ? launch_typed<64, 64, 2, int64_t, ROPE, HP>(p, tq, tk, tv, ra, num_sms, stream)
                   : launch_typed<64, 64, 2, int32_t, ROPE, HP>(p, tq, tk, tv, ra, num_sms, stream);
}

template <bool ROPE>
cudaError_t launch_attn_dispatch(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const RopeArgs& ra, bool use_int64,
                                 int num_sms, cudaStream_t stream) {
  return p.head_pairs
             ? launch_attn_dispatch_hp<ROPE, true>(p, tq, tk, tv, ra, use_int64, num_sms, stream)
             : launch_attn_dispatch_hp<ROPE, false>(p, tq, tk, tv, ra, use_int64, num_sms, stream);
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, bool use_int64, int num_sms,
                            cudaStream_t stream, const RopeArgs* rope) {
  if (rope != nullptr)
    return launch_attn_dispatch<true>(p, tq, tk, tv, *rope, use_int64, num_sms, stream);
  RopeArgs none;
  memset(&none, 0, sizeof(none));
  return launch_attn_dispatch<false>(p, tq, tk, tv, none, use_int64, num_sms, stream);
}

cudaError_t launch_attn_plan(const AttnParams& p, cudaStream_t stream) {
  return p.block_n == 128 ? launch_plan<128, kQTilesBN128>(p, stream)
                          : launch_plan<64, 2>(p, stream);
}

cudaError_t launch_bounded_wait_probe(int32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  bounded_wait_probe_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace fm
