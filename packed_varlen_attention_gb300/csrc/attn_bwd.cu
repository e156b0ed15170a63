// attn_bwd.cu -- FlashMask attention backward over packed samples on sm_103a.
//
// What is computed (PaddleNLP FlashMask article, section 3.4: the backward
// operator takes q, k, v, the column intervals, out, softmax_lse and the
// output gradient; section 3.3: the block-skipping kernel equals dense-mask
// attention, so its gradient is the gradient of dense-mask attention).  For
// every sample, q head h (key/value head g = h / (Hq / Hkv)) and unmasked
// pair (i, j):
//     p_ij  = exp(scale * q_i . k_j - lse_i)      (lse from the forward pass)
//     dp_ij = do_i . v_j,   delta_i = do_i . o_i
//     ds_ij = p_ij * (dp_ij - delta_i)
//     dq_i  = scale * sum_j ds_ij k_j
//     dk_j  = scale * sum_{h in group, i} ds_ij q_i
//     dv_j  = sum_{h in group, i} p_ij do_i
// The same block classes as the forward pass (section 3.2) skip fully masked
// blocks and restrict the element mask to partially masked ones.
//
// How it runs on GB300 -- five launches (prep, then a one-CTA planner and
// the persistent kernel for each pass), every sum owned by one CTA (no
// atomics, so the gradients are bitwise reproducible):
//   * prep: one pass over out and dout: -delta_i and -lse_i * log2(e) per
//     (head, row) into the workspace (fp32).
//   * dK/dV kernel: a work item is one 128-key tile of one key/value head;
//     it walks every q head of the group and every 64-row Q tile that is not
//     fully masked, keeping dK and dV in TMEM for the whole item.
//   * dQ kernel: a work item is one 128-row Q tile of one q head; it walks
//     the 64-key tiles that are not fully masked, keeping dQ in TMEM.
// Both are one persistent kernel template (one CTA per SM pulling items from
// an atomic counter) with the same warp roles (384 threads):
//   warp 0   producer: block classes of the item's steps, per-step metadata
//            in an 8-slot ring, TMA loads of the two resident tiles (R1, R2:
//            K, V or Q, dO; 128 rows) once per item and of the first
//            streamed tile (C1: Q or K; 64 rows) per step;
//   warp 2   TMA loads of the second streamed tile (C2: dO or V) per step;
//   warp 1   MMA issuer of X = R1 C1^T and Y = R2 C2^T (tcgen05.mma
//            kind::f16, M = 128, N = 64, fp32 in TMEM, two buffers);
//   warp 3   MMA issuer of the accumulating products, operand A read from
//            TMEM: dV += P^T dO and dK += dS^T Q, or dQ += dS K;
//   warps 4..11  elementwise, two warpgroups, one thread per TMEM lane,
//            each warpgroup 32 of the 64 streamed columns: masks X, forms
//            P = 2^(X * scale * log2 e - lse * log2 e) and
//            dS = P * (Y - delta), stores them as bf16 into TMEM over X and
//            Y, and writes the gradients of the item at its end.
// X / Y of step t+1 run on the tensor cores while the elementwise warps work
// on step t.
// Every mbarrier wait is bounded and reports FM_DEVERR_TIMEOUT instead of
// hanging.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "attn_common.cuh"
#include "fm_device.cuh"
#include "fm_internal.h"

namespace fm {
namespace {

enum : int { kModeDQ = 0, kModeDKV = 1 };

constexpr int kBwdThreads = 384;
constexpr int kRes = 128;       // resident tile rows = TMEM lanes
constexpr int kSub = 64;        // streamed tile rows
constexpr int kStatTile = 128;  // key tile of the block statistics
constexpr int kBwdMeta = 8;     // metadata ring slots
constexpr int kSlotBytes = 1024;
constexpr int kMaxStages = 8;

template <int D>
constexpr int kBwdStages = D == 128 ? 4 : 6;

enum : int { kFirst = 1, kLast = 2, kStop = 8 };

struct BwdMeta {
  int flags;  // kFirst | kLast, or kStop
  int cls;    // block class of this step
  int c0;     // first row (token) of the streamed tile
  int r0;     // first row (token) of the resident tile
  int b;      // end of the sample
  int h;      // q head of this step
  int kvh;    // key/value head
  int mh;     // mask head
  int pad[8];
};
static_assert(sizeof(BwdMeta) == 64, "BwdMeta is 64 bytes");

constexpr int kMaxBufs = 3;  // X / Y buffers: 3 for dQ, 2 for dK/dV (TMEM budget)

enum BwdBar : int {
  bCFull = 0,                      // [stages] both streamed tiles landed (two producers)
  bCEmpty = bCFull + kMaxStages,   // [stages] accumulating MMAs of the step done
  bMFull = bCEmpty + kMaxStages,
  bRFull = bMFull + kBwdMeta,   // both resident tiles of an item landed
  bREmpty,                      // last X/Y MMAs of an item done
  bSFull,                       // [buffers] X and Y ready
  bPFull = bSFull + kMaxBufs,   // [buffers] P / dS written (one arrival per warp)
  bAccFull = bPFull + kMaxBufs, // last accumulating MMA of an item done
  bAccEmpty,                    // accumulators read by the epilogue (one per warp)
  bTSDone,                      // [buffers] accumulating MMAs of the buffer's step done
  bDrain = bTSDone + kMaxBufs,  // [2 issuers]
  bNumBars = bDrain + 2
};

// A metadata slot needs no release barrier: the producer writes slot u mod 8
// only after stage (u - 1) mod NS was freed, i.e. after the accumulating MMAs
// of step u - 1 - NS, which follow every read of steps <= u - 1 - NS (the
// elementwise warps read a step's slot before its P-full, the C2 producer
// before its load).  The slot's previous step u - 8 is among them when
// NS <= 7.
static_assert(kBwdStages<64> <= kBwdMeta - 1 && kBwdStages<128> <= kBwdMeta - 1,
              "metadata ring reuse is ordered by the stage ring");
// arrivals on bPFull and bAccEmpty: one per elementwise warp
constexpr int kBwdEwWarps = 8;

template <int D, int Mode>
struct BwdLayout {
  static constexpr int NS = kBwdStages<D>;
  // X / Y buffers: the loop X/Y ready -> P/dS -> accumulating MMAs -> buffer
  // free spans NB steps.  dK/dV keeps two fp32 accumulators (2 D columns) in
  // TMEM and fits two buffers; dQ keeps one and fits three.
  static constexpr int NB = Mode == kModeDQ ? 3 : 2;
  static constexpr int kRBytes = kRes * D * 2;
  static constexpr int kCBytes = kSub * D * 2;
  static constexpr int kR = 0;  // R1, then R2
  static constexpr int kC1 = 2 * kRBytes;
  static constexpr int kC2 = kC1 + NS * kCBytes;
  static constexpr int kSlots = kC2 + NS * kCBytes;  // per-step data, kSlotBytes each
  static constexpr int kMeta = kSlots + kBwdMeta * kSlotBytes;
  // flags of the step held by each stage (published by the stage's full
  // barrier) and of the step in each X / Y buffer (published by P-full)
  static constexpr int kStageFlags = kMeta + kBwdMeta * static_cast<int>(sizeof(BwdMeta));
  static constexpr int kBufFlags = kStageFlags + kMaxStages * 4;
  static constexpr int kBars = kBufFlags + 16;
  static constexpr int kTmemSlot = kBars + bNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kEnd = kAbort + 4;
  static constexpr int kBytes = kEnd + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns: X of buffer b at 64 b (P packed over its columns 0..15
  // and 32..47), Y at 64 (NB + b) (dS likewise), accumulators from 128 NB:
  // dQ, or dV then dK.
  __host__ __device__ static constexpr uint32_t x_col(uint32_t b) { return 64u * b; }
  __host__ __device__ static constexpr uint32_t y_col(uint32_t b) { return 64u * (NB + b); }
  static constexpr uint32_t kAcc0 = 128 * NB;
  static constexpr uint32_t kAcc1 = 128 * NB + D;
  static_assert(kAcc0 + (Mode == kModeDQ ? D : 2 * D) <= kTmemCols, "TMEM budget");
  static_assert(NB <= kMaxBufs, "buffer barriers");
  static_assert(NS <= kMaxStages, "stage barriers");
  static_assert(kBytes <= 232448, "shared memory budget");
  static_assert(kSub * 4 * 4 <= kSlotBytes, "slot holds four interval vectors");
};

// sample of packed tile slot u (slots: floor(cu[s] / tile) + s + t)
__device__ __forceinline__ int slot_sample(const AttnBwdParams& p, int64_t u, int tile) {
  const int T = static_cast<int>(p.T);
  int lo = 0, hi = p.n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int64_t base = static_cast<int64_t>(clamp_tok(__ldg(p.cu + mid), T)) / tile + mid;
    if (base <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void load_stats(const AttnBwdParams& p, int mh, int64_t slot,
                                           int (&st)[8]) {
#pragma unroll
  for (int v = 0; v < 8; ++v)
    st[v] = __ldg(p.minmax + (static_cast<int64_t>(mh) * 8 + v) * p.n_kv_slots + slot);
}

// The 128-row tile of packed slot u (slots: floor(cu[s] / 128) + s + t).
struct ResTile {
  int s, a, b;  // sample and its token range [a, b)
  int r0, r1;   // rows of the tile
  int64_t t;    // tile index in the sample
  bool real;    // false for slots that hold no tile
};

__device__ __forceinline__ ResTile res_tile(const AttnBwdParams& p, int64_t u) {
  const int T = static_cast<int>(p.T);
  ResTile rt;
  rt.s = slot_sample(p, u, kRes);
  rt.a = clamp_tok(__ldg(p.cu + rt.s), T);
  rt.b = max(rt.a, clamp_tok(__ldg(p.cu + rt.s + 1), T));
  rt.t = u - (static_cast<int64_t>(rt.a) / kRes + rt.s);
  rt.real = rt.t >= 0 && rt.a + rt.t * kRes < rt.b;
  rt.r0 = rt.real ? rt.a + static_cast<int>(rt.t) * kRes : rt.a;
  rt.r1 = min(rt.r0 + kRes, rt.b);
  return rt;
}

// dQ steps of a Q tile: key tiles of 64 columns up to the diagonal (causal)
// or the sample end; key tile k covers [a + 64k, min(a + 64k + 64, b)) and
// takes the statistics of the 128-column tile holding it.
__device__ __forceinline__ int dq_n_steps(const AttnBwdParams& p, const ResTile& rt) {
  return p.causal ? (rt.r1 - 1 - rt.a) / kSub + 1 : (rt.b - rt.a + kSub - 1) / kSub;
}
__device__ __forceinline__ int dq_class(const AttnBwdParams& p, const ResTile& rt, int mh, int k,
                                        int n_sub) {
  if (k >= n_sub) return kClsF;
  const int c0 = rt.a + k * kSub;
  const int c1 = min(c0 + kSub, rt.b);
  int st[8];
  if (p.sri != nullptr)
    load_stats(p, mh, static_cast<int64_t>(rt.a / kStatTile) + rt.s + k / 2, st);
  return classify_block(rt.r0, rt.r1, c0, c1, st, p.sri != nullptr, p.causal != 0);
}

// dK/dV steps of a key tile, per q head: Q tiles of 64 rows from the one
// holding the diagonal (causal) or the sample start; step k covers rows
// [a + 64 (q_first + k), ...).
__device__ __forceinline__ int dkv_q_first(const AttnBwdParams& p, const ResTile& rt) {
  return p.causal ? (rt.r0 - rt.a) / kSub : 0;
}
__device__ __forceinline__ int dkv_class(const AttnBwdParams& p, const ResTile& rt, int mh, int k,
                                         int q_first, int n_q) {
  if (k >= n_q) return kClsF;
  const int q0 = rt.a + (q_first + k) * kSub;
  const int q1 = min(q0 + kSub, rt.b);
  int st[8];
  if (p.sri != nullptr) load_stats(p, mh, static_cast<int64_t>(rt.a / kStatTile) + rt.s + rt.t, st);
  return classify_block(q0, q1, rt.r0, rt.r1, st, p.sri != nullptr, p.causal != 0);
}

// Steps of the dK/dV item of tile rt under mask head mh: its 64-row Q tiles
// that are not fully masked.
__device__ __forceinline__ int dkv_tile_steps(const AttnBwdParams& p, const ResTile& rt, int mh) {
  const int q_first = dkv_q_first(p, rt);
  const int n_q = (rt.b - rt.a + kSub - 1) / kSub - q_first;
  int st[8];
  if (p.sri != nullptr) load_stats(p, mh, static_cast<int64_t>(rt.a / kStatTile) + rt.s + rt.t, st);
  int n = 0;
  for (int k = 0; k < n_q; ++k) {
    const int q0 = rt.a + (q_first + k) * kSub;
    const int q1 = min(q0 + kSub, rt.b);
    n += classify_block(q0, q1, rt.r0, rt.r1, st, p.sri != nullptr, p.causal != 0) != kClsF;
  }
  return n;
}

// P and dS for two elements: p = 2^(x * c + nl), ds = p * (y + nd); returns
// both as bf16x2 (first element in the low half).
__device__ __forceinline__ void bwd_pair(uint32_t x0, uint32_t x1, uint32_t y0, uint32_t y1,
                                         uint64_t c2, uint64_t nl2, uint64_t nd2, uint32_t& pk,
                                         uint32_t& dsk) {
  asm("{\n\t.reg .b64 x, e, p, y, t;\n\t.reg .f32 e0, e1, p0, p1, t0, t1;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "fma.rn.f32x2 e, x, %6, %7;\n\t"
      "mov.b64 {e0, e1}, e;\n\t"
      "ex2.approx.ftz.f32 p0, e0;\n\t"
      "ex2.approx.ftz.f32 p1, e1;\n\t"
      "mov.b64 p, {p0, p1};\n\t"
      "mov.b64 y, {%4, %5};\n\t"
      "add.f32x2 t, y, %8;\n\t"
      "mul.f32x2 t, t, p;\n\t"
      "mov.b64 {t0, t1}, t;\n\t"
      "cvt.rn.bf16x2.f32 %0, p1, p0;\n\t"
      "cvt.rn.bf16x2.f32 %1, t1, t0;\n\t}"
      : "=r"(pk), "=r"(dsk)
      : "r"(x0), "r"(x1), "r"(y0), "r"(y1), "l"(c2), "l"(nl2), "l"(nd2));
}

// 32 consecutive columns at each of two TMEM addresses, one wait for both.
__device__ __forceinline__ void tmem_ld32_pair(uint32_t ta, uint32_t tb, uint32_t (&a)[32],
                                               uint32_t (&b)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]), "=r"(b[16]), "=r"(b[17]), "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]), "=r"(b[24]), "=r"(b[25]), "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31])
      : "r"(ta), "r"(tb)
      : "memory");
}

// Four accumulating MMAs (K = 16 each) whose A operand comes from TMEM at
// column offsets 0, 8, 32, 40 (the packed halves the two elementwise
// warpgroups write) and whose B operand advances by OB per step.
template <int OB>
__device__ __forceinline__ void umma_ts_group4_split(uint32_t d_tmem, uint32_t a_tmem,
                                                     uint64_t b_desc, uint32_t idesc,
                                                     uint32_t acc0) {
  asm volatile("{\n\t.reg .pred p, q, e;\n\t.reg .b32 el;\n\t"
               ".reg .b64 b;\n\t.reg .b32 a;\n\t"
               "elect.sync el|e, 0xffffffff;\n\t"
               "setp.ne.b32 p, %4, 0;\n\t"
               "setp.eq.u32 q, 0, 0;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
               "add.u32 a, %1, 8;\n\tadd.s64 b, %2, %5;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
               "add.u32 a, %1, 32;\n\tadd.s64 b, %2, %6;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
               "add.u32 a, %1, 40;\n\tadd.s64 b, %2, %7;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
               "}"
               :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc0),
                  "n"(1 * OB), "n"(2 * OB), "n"(3 * OB)
               : "memory");
}

// ---------------------------------------------------------------------------
// prep: -delta and -lse * log2(e)
// ---------------------------------------------------------------------------

// One group of D/8 threads per (token, head) row, 8 elements per thread.
template <int D, typename IdxT>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const AttnBwdParams p) {
  constexpr int G = D / 8;
  pdl_trigger();
  pdl_wait();
  const int64_t n_rows = p.T * p.hq;
  const int64_t r = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) / G;
  const int part = threadIdx.x % G;
  float acc = 0.f;
  if (r < n_rows) {
    const uint4 o4 = __ldg(reinterpret_cast<const uint4*>(
                               static_cast<const __nv_bfloat16*>(p.out) + static_cast<IdxT>(r) * D) +
                           part);
    const uint4 d4 = __ldg(reinterpret_cast<const uint4*>(
                               static_cast<const __nv_bfloat16*>(p.dout) + static_cast<IdxT>(r) * D) +
                           part);
    const uint32_t ow[4] = {o4.x, o4.y, o4.z, o4.w};
    const uint32_t dw[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[u]));
      const float2 df = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dw[u]));
      acc = fmaf(of.x, df.x, acc);
      acc = fmaf(of.y, df.y, acc);
    }
  }
#pragma unroll
  for (int d = G / 2; d > 0; d >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, d);
  if (r < n_rows && part == 0) {
    const int64_t t = r / p.hq;
    const int h = static_cast<int>(r % p.hq);
    const IdxT o = static_cast<IdxT>(h) * static_cast<IdxT>(p.T) + static_cast<IdxT>(t);
    const float l = __ldg(p.lse + o);
    p.ndelta[o] = -acc;
    p.nlse2[o] = (l == -CUDART_INF_F) ? -CUDART_INF_F : -l * 1.4426950408889634f;
  }
}

// ---------------------------------------------------------------------------
// planner: the 128-row tiles of every sample, longest samples first
// ---------------------------------------------------------------------------

// One CTA.  Samples are ordered by their number of 128-row tiles, longest
// first (counting sort, lengths capped at kCostBins - 1 tiles); the tiles of
// a sample stay together, dK/dV in tile order and dQ in reverse tile order,
// so that under a causal mask the tiles with the most steps come first and
// the concurrently running items of one sample share their streamed tiles in
// L2.  dK/dV items can be long (a key tile near the start of a long causal
// sample walks every later Q tile of every q head of its group): when the
// largest one exceeds half of the work per CTA, the sample order leaves a
// tail of one CTA still on a large item, so the key tiles are ordered by
// their own step counts instead, largest first (the costliest mask head's
// count).  Only real tiles are listed.
template <int Mode>
__global__ void __launch_bounds__(kCostBins) bwd_plan_order_kernel(const AttnBwdParams p) {
  __shared__ int tiles_in_bin[kCostBins];
  __shared__ int step_bin[kCostBins];  // dK/dV: key tiles per step count
  __shared__ int warp_tot[kCostBins / 32];
  __shared__ unsigned long long steps_total;
  __shared__ int steps_max;
  __shared__ int by_steps;
  const int T = static_cast<int>(p.T);
  int* order = Mode == kModeDQ ? p.order_q : p.order_kv;
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x;
  const int lane = tid & 31, w = tid >> 5;
  tiles_in_bin[tid] = 0;
  step_bin[tid] = 0;
  if (tid == 0) {
    steps_total = 0ull;
    steps_max = 0;
  }
  __syncthreads();
  auto n_tiles_of = [&](int s) -> int {
    const int a = clamp_tok(__ldg(p.cu + s), T);
    const int b = max(a, clamp_tok(__ldg(p.cu + s + 1), T));
    return (b - a + kRes - 1) / kRes;
  };
  for (int s = tid; s < p.n_seqs; s += kCostBins) {
    const int n = n_tiles_of(s);
    if (n > 0) atomicAdd(&tiles_in_bin[min(n, kCostBins - 1)], n);
  }
  const int n_mh = p.hm > 1 ? p.hm : 1;
  auto kv_steps = [&](const ResTile& rt) -> int {
    int c = 0;
    for (int mh = 0; mh < n_mh; ++mh) c = max(c, dkv_tile_steps(p, rt, mh));
    return c;
  };
  if (Mode == kModeDKV) {
    unsigned long long my_total = 0ull;
    int my_max = 0;
    for (int64_t u = tid; u < p.n_res_slots; u += kCostBins) {
      const ResTile rt = res_tile(p, u);
      if (!rt.real) continue;
      const int c = kv_steps(rt);
      my_total += static_cast<unsigned long long>(c);
      my_max = max(my_max, c);
      atomicAdd(&step_bin[min(c, kCostBins - 1)], 1);
    }
    if (my_total != 0ull) atomicAdd(&steps_total, my_total);
    if (my_max != 0) atomicMax(&steps_max, my_max);
  }
  __syncthreads();
  if (Mode == kModeDKV) {
    // an item walks its key tile for every q head of the group: the largest
    // item is group * max steps, the work per CTA Hq * total / CTAs
    if (tid == 0) {
      const unsigned long long group = static_cast<unsigned long long>(p.hq / p.hkv);
      by_steps = 2ull * group * static_cast<unsigned long long>(steps_max) *
                     static_cast<unsigned long long>(max(p.num_sms, 1)) >
                 static_cast<unsigned long long>(p.hq) * steps_total;
    }
    __syncthreads();
    if (by_steps) tiles_in_bin[tid] = step_bin[tid];
    __syncthreads();
  }
  // exclusive prefix over bins in descending order (position 0: largest bin)
  const int bin = kCostBins - 1 - tid;
  const int cnt = tiles_in_bin[bin];
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
    warp_tot[lane] = t;
  }
  __syncthreads();
  const int incl = x + (w > 0 ? warp_tot[w - 1] : 0);
  tiles_in_bin[bin] = incl - cnt;  // now the bin's next free position
  if (tid == kCostBins - 1) {
    // the header needs no clearing by the caller: this planner initialises
    // its pass's counter (and, before the first pass, the error record)
    if (Mode == kModeDQ) {
      p.ws->bwd_q_tiles = incl;
      p.ws->work_counter = 0u;
    } else {
      p.ws->bwd_kv_tiles = incl;
      p.ws->work_counter_kv = 0u;
      p.ws->error_word = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) p.ws->diag[i] = 0;
    }
    // the tables after the header now hold the backward's order: a forward
    // plan in this workspace is gone
    p.ws->plan_n_seqs = 0;
  }
  __syncthreads();
  if (Mode == kModeDKV && by_steps) {
    for (int64_t u = tid; u < p.n_res_slots; u += kCostBins) {
      const ResTile rt = res_tile(p, u);
      if (rt.real)
        order[atomicAdd(&tiles_in_bin[min(kv_steps(rt), kCostBins - 1)], 1)] = static_cast<int>(u);
    }
    return;
  }
  for (int s = tid; s < p.n_seqs; s += kCostBins) {
    const int n = n_tiles_of(s);
    if (n == 0) continue;
    const int pos = atomicAdd(&tiles_in_bin[min(n, kCostBins - 1)], n);
    const int a = clamp_tok(__ldg(p.cu + s), T);
    const int base = a / kRes + s;  // slot of the sample's first tile
    for (int t = 0; t < n; ++t) order[pos + t] = base + (Mode == kModeDQ ? n - 1 - t : t);
  }
}

// ---------------------------------------------------------------------------
// dK/dV and dQ kernels
// ---------------------------------------------------------------------------

template <int D, int Mode>
__device__ __forceinline__ void bwd_teardown(uint32_t* tmem_slot, int warp) {
  tc_fence_before();
  asm volatile("bar.sync 1, %0;" ::"n"(kBwdThreads) : "memory");
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(*reinterpret_cast<volatile uint32_t*>(tmem_slot), BwdLayout<D, Mode>::kTmemCols);
  }
}

// Zero gradients of resident rows [r0, r1) (an item none of whose blocks is
// live): dq of head h, or dk and dv of head h.
template <int D, int Mode, typename IdxT>
__device__ __forceinline__ void zero_rows(const AttnBwdParams& p, int r0, int r1, int h,
                                          int lane) {
  const int heads = Mode == kModeDQ ? p.hq : p.hkv;
  for (int r = r0 + lane; r < r1; r += 32) {
    const IdxT off = (static_cast<IdxT>(r) * heads + h) * static_cast<IdxT>(D);
    uint4* d0 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(Mode == kModeDQ ? p.dq : p.dv) + off);
#pragma unroll
    for (int u = 0; u < D / 8; ++u) d0[u] = make_uint4(0u, 0u, 0u, 0u);
    if (Mode == kModeDKV) {
      uint4* d1 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dk) + off);
#pragma unroll
      for (int u = 0; u < D / 8; ++u) d1[u] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

template <int D, int Mode, typename IdxT>
__device__ __forceinline__ void bwd_producer_roles(const AttnBwdParams& p, const CUtensorMap& tr1,
                                                   const CUtensorMap& tr2, const CUtensorMap& tc1,
                                                   const CUtensorMap& tc2) {
  using L = BwdLayout<D, Mode>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  BwdMeta* meta = reinterpret_cast<BwdMeta*>(smem + L::kMeta);
  uint8_t* slots = smem + L::kSlots;
  volatile int* stage_flags = reinterpret_cast<volatile int*>(smem + L::kStageFlags);
  volatile int* buf_flags = reinterpret_cast<volatile int*>(smem + L::kBufFlags);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = static_cast<int>(p.T);
  const Sync sy{bars, abort_flag, p.timeout_ns, &p.ws->error_word, lane};
  if (threadIdx.x == 0) {
    for (int i = 0; i < L::NS; ++i) {
      mbar_init(&bars[bCFull + i], 2);
      mbar_init(&bars[bCEmpty + i], 1);
    }
    for (int i = 0; i < kBwdMeta; ++i) {
      mbar_init(&bars[bMFull + i], 1);
    }
    mbar_init(&bars[bRFull], 1);
    mbar_init(&bars[bREmpty], 1);
    for (int i = 0; i < kMaxBufs; ++i) {
      mbar_init(&bars[bSFull + i], 1);
      mbar_init(&bars[bPFull + i], kBwdEwWarps);
      mbar_init(&bars[bTSDone + i], 1);
    }
    mbar_init(&bars[bAccFull], 1);
    mbar_init(&bars[bAccEmpty], kBwdEwWarps);
    for (int i = 0; i < 2; ++i) mbar_init(&bars[bDrain + i], 1);
    *abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tr1);
    tma_prefetch_desc(&tr2);
    tma_prefetch_desc(&tc1);
    tma_prefetch_desc(&tc2);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // previous kernels' outputs (planner tables, -lse, -delta) are ready

  if (warp == 0) {
    // ------------------------------------------------- producer + metadata
    const int group = p.hq / p.hkv;
    const int n_heads_item = Mode == kModeDQ ? p.hq : p.hkv;
    const int64_t n_items =
        static_cast<int64_t>(Mode == kModeDQ ? p.ws->bwd_q_tiles : p.ws->bwd_kv_tiles) *
        n_heads_item;
    uint32_t* counter = Mode == kModeDQ ? &p.ws->work_counter : &p.ws->work_counter_kv;
    uint32_t mslot = 0, mround = 0;
    uint32_t cst = 0, cround = 0;
    uint32_t r_round = 0;
    uint32_t c_armed[kMaxStages];
#pragma unroll
    for (int i = 0; i < kMaxStages; ++i) c_armed[i] = 0xffffffffu;
    uint32_t r_armed = 0xffffffffu;
    bool ok = true;

    auto push_meta = [&](int flags, int cls, int c0, int r0, int b, int h, int kvh,
                         int mh) -> bool {
      if (!(flags & kStop)) {
        uint8_t* sd = slots + mslot * kSlotBytes;
        if (Mode == kModeDQ) {
          if (cls == kClsP) {
            // the four interval vectors of the 64 key columns
            int* cl = reinterpret_cast<int*>(sd);
            const int32_t* src = p.sri + static_cast<int64_t>(mh) * 4 * p.T;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
#pragma unroll
              for (int m = 0; m < kSub / 32; ++m) {
                const int jj = m * 32 + lane;
                const int c = c0 + jj;
                cl[v * kSub + jj] =
                    (c < b && c < T) ? __ldg(src + static_cast<int64_t>(v) * p.T + c) : 0;
              }
            }
          }
        } else {
          // -lse*log2(e) and -delta of the 64 query rows; rows outside the
          // sample get -inf (p = 0 without a mask test) and 0
          float* nl = reinterpret_cast<float*>(sd);
          float* nd = nl + kSub;
#pragma unroll
          for (int m = 0; m < kSub / 32; ++m) {
            const int jj = m * 32 + lane;
            const int i = c0 + jj;
            float a = -CUDART_INF_F, d = 0.f;
            if (i < b && i < T) {
              const IdxT o = static_cast<IdxT>(h) * static_cast<IdxT>(p.T) + static_cast<IdxT>(i);
              a = __ldg(p.nlse2 + o);
              d = __ldg(p.ndelta + o);
            }
            nl[jj] = a;
            nd[jj] = d;
          }
        }
      }
      if (lane == 0) {
        BwdMeta& m = meta[mslot];
        m.flags = flags;
        m.cls = cls;
        m.c0 = c0;
        m.r0 = r0;
        m.b = b;
        m.h = h;
        m.kvh = kvh;
        m.mh = mh;
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[bMFull + mslot]);
      if (++mslot == kBwdMeta) {
        mslot = 0;
        ++mround;
      }
      return true;
    };

    // one step: metadata, the resident tiles (first step), the C1 tile
    auto push_step = [&](int flags, int cls, int c0, int r0, int b, int h, int kvh,
                         int mh) -> bool {
      if (!push_meta(flags, cls, c0, r0, b, h, kvh, mh)) return false;
      if (flags & kFirst) {
        if (!sy.warp(bREmpty, (r_round & 1) ^ 1)) return false;
        if (lane == 0) {
          const int rx = (Mode == kModeDQ ? h : kvh) * D;
          mbar_arrive_expect_tx(&bars[bRFull], 2 * L::kRBytes);
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            tma_load_2d(smem + L::kR + c * (kRes * 128), &tr1, &bars[bRFull], rx + c * 64, r0);
            tma_load_2d(smem + L::kR + L::kRBytes + c * (kRes * 128), &tr2, &bars[bRFull],
                        rx + c * 64, r0);
          }
        }
        r_armed = r_round;
        ++r_round;
      }
      if (!sy.warp(bCEmpty + cst, (cround & 1) ^ 1)) return false;
      if (lane == 0) {
        const int cx = (Mode == kModeDQ ? kvh : h) * D;
        stage_flags[cst] = flags;
        mbar_arrive_expect_tx(&bars[bCFull + cst], L::kCBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(smem + L::kC1 + cst * L::kCBytes + c * (kSub * 128), &tc1,
                      &bars[bCFull + cst], cx + c * 64, c0);
      }
      c_armed[cst] = cround;
      if (++cst == L::NS) {
        cst = 0;
        ++cround;
      }
      return true;
    };

    while (ok) {
      int64_t item = 0;
      if (lane == 0) item = static_cast<int64_t>(atomicAdd(counter, 1u));
      item = __shfl_sync(0xffffffffu, item, 0);
      if (item >= n_items) {
        // the stop token: through the metadata ring (C2 producer,
        // elementwise warps) and through the next stage (issuers)
        ok = push_meta(kStop, kClsF, 0, 0, 0, 0, 0, 0) &&
             sy.warp(bCEmpty + cst, (cround & 1) ^ 1);
        if (ok && lane == 0) {
          stage_flags[cst] = kStop;
          mbar_arrive(&bars[bCFull + cst]);
        }
        break;
      }
      // tiles in the planner's order (longest samples first), heads fastest
      const int64_t u = __ldg((Mode == kModeDQ ? p.order_q : p.order_kv) + item / n_heads_item);
      const int hi = static_cast<int>(item % n_heads_item);
      const ResTile rt = res_tile(p, u);
      if (!rt.real) continue;  // (the planner lists real tiles only)
      const int a = rt.a, b = rt.b, r0 = rt.r0, r1 = rt.r1;

      if (Mode == kModeDQ) {
        const int h = hi;
        const int kvh = h / group;
        const int mh = p.hm > 1 ? h : 0;
        const int n_sub = dq_n_steps(p, rt);
        auto cls_of = [&](int k) -> int { return dq_class(p, rt, mh, k, n_sub); };
        int n_live = 0;
        for (int base = 0; base < n_sub; base += 32)
          n_live += __popc(__ballot_sync(0xffffffffu, cls_of(base + lane) != kClsF));
        if (n_live == 0) {
          zero_rows<D, Mode, IdxT>(p, r0, r1, h, lane);
          continue;
        }
        int pushed = 0;
        for (int base = 0; base < n_sub && ok; base += 32) {
          const int my = cls_of(base + lane);
          uint32_t live = __ballot_sync(0xffffffffu, my != kClsF);
          while (live != 0u) {
            const int l = __ffs(live) - 1;
            live &= live - 1u;
            const int cls = __shfl_sync(0xffffffffu, my, l);
            const int flags = (pushed == 0 ? kFirst : 0) | (pushed == n_live - 1 ? kLast : 0);
            if (!push_step(flags, cls, a + (base + l) * kSub, r0, b, h, kvh, mh)) {
              ok = false;
              break;
            }
            ++pushed;
          }
        }
      } else {
        const int kvh = hi;
        const int q_first = dkv_q_first(p, rt);
        const int n_q = (b - a + kSub - 1) / kSub - q_first;
        auto cls_of = [&](int h, int k) -> int {
          return dkv_class(p, rt, p.hm > 1 ? h : 0, k, q_first, n_q);
        };
        int n_live = 0;
        for (int h = kvh * group; h < (kvh + 1) * group; ++h)
          for (int base = 0; base < n_q; base += 32)
            n_live += __popc(__ballot_sync(0xffffffffu, cls_of(h, base + lane) != kClsF));
        if (n_live == 0) {
          zero_rows<D, Mode, IdxT>(p, r0, r1, kvh, lane);
          continue;
        }
        int pushed = 0;
        for (int h = kvh * group; h < (kvh + 1) * group && ok; ++h) {
          const int mh = p.hm > 1 ? h : 0;
          for (int base = 0; base < n_q && ok; base += 32) {
            const int my = cls_of(h, base + lane);
            uint32_t live = __ballot_sync(0xffffffffu, my != kClsF);
            while (live != 0u) {
              const int l = __ffs(live) - 1;
              live &= live - 1u;
              const int cls = __shfl_sync(0xffffffffu, my, l);
              const int flags = (pushed == 0 ? kFirst : 0) | (pushed == n_live - 1 ? kLast : 0);
              if (!push_step(flags, cls, a + (q_first + base + l) * kSub, r0, b, h, kvh, mh)) {
                ok = false;
                break;
              }
              ++pushed;
            }
          }
        }
      }
    }
    if (!ok) {
      // let every TMA load this warp issued land before the CTA exits
      for (int st = 0; st < L::NS; ++st)
        if (c_armed[st] != 0xffffffffu)
          mbar_wait_bounded(&bars[bCFull + st], c_armed[st] & 1, 100000000ull, nullptr);
      if (r_armed != 0xffffffffu)
        mbar_wait_bounded(&bars[bRFull], r_armed & 1, 100000000ull, nullptr);
    }
    bwd_teardown<D, Mode>(tmem_slot, warp);
    return;
  } else if (warp == 2) {
    // ------------------------------------------------------------ C2 producer
    if (lane == 0) {
      uint32_t cst = 0, cround = 0, mslot = 0, mround = 0;
      uint32_t c_armed[kMaxStages];
      for (int i = 0; i < kMaxStages; ++i) c_armed[i] = 0xffffffffu;
      bool ok = true;
      for (;;) {
        if (!sy.lone(bMFull + mslot, mround & 1)) { ok = false; break; }
        const int flags = *reinterpret_cast<volatile int*>(&meta[mslot].flags);
        const int c0 = *reinterpret_cast<volatile int*>(&meta[mslot].c0);
        const int h = *reinterpret_cast<volatile int*>(&meta[mslot].h);
        const int kvh = *reinterpret_cast<volatile int*>(&meta[mslot].kvh);
        if (++mslot == kBwdMeta) {
          mslot = 0;
          ++mround;
        }
        if (!sy.lone(bCEmpty + cst, (cround & 1) ^ 1)) { ok = false; break; }
        if (flags & kStop) {
          mbar_arrive(&bars[bCFull + cst]);  // second arrival of the stop stage
          break;
        }
        const int cx = (Mode == kModeDQ ? kvh : h) * D;
        mbar_arrive_expect_tx(&bars[bCFull + cst], L::kCBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(smem + L::kC2 + cst * L::kCBytes + c * (kSub * 128), &tc2,
                      &bars[bCFull + cst], cx + c * 64, c0);
        c_armed[cst] = cround;
        if (++cst == L::NS) {
          cst = 0;
          ++cround;
        }
      }
      if (!ok) {
        for (int st = 0; st < L::NS; ++st)
          if (c_armed[st] != 0xffffffffu)
            mbar_wait_bounded(&bars[bCFull + st], c_armed[st] & 1, 100000000ull, nullptr);
      }
    }
    bwd_teardown<D, Mode>(tmem_slot, warp);
    return;
  } else if (warp == 1 || warp == 3) {
    // ----------------------------------------------------------- MMA issuers
    // Warp 1 issues X / Y of every step, warp 3 the accumulating MMAs; the
    // whole warp runs each loop, elect.sync picks the issuing lane.  While one
    // issuer waits on a barrier or commits, the other's MMAs keep the tensor
    // pipe busy.  Cross-issuer order: X / Y of step t overwrite the buffer the
    // accumulating MMAs of step t-NB read, so warp 1 waits for their
    // completion (TSDone); the accumulating MMAs of step t read P / dS of
    // step t, whose elementwise pass started after X / Y of step t were
    // complete.  All accumulation comes from one thread, in step order.
    constexpr uint32_t kIdescXY = idesc_bf16_f32(kRes, kSub, false);
    constexpr uint32_t kIdescAcc = idesc_bf16_f32(kRes, D, true);
    const uint32_t r_addr = smem_u32(smem + L::kR);
    const uint32_t c1_addr = smem_u32(smem + L::kC1);
    const uint32_t c2_addr = smem_u32(smem + L::kC2);
    const int me = warp == 1 ? 0 : 1;
    uint32_t st = 0, round = 0, n = 0;  // stage ring position, steps done
    bool ok = true;
    if (me == 0) {
      // K-major operands of X = R1 C1^T and Y = R2 C2^T
      const uint64_t r1_desc = sdesc_sw128(r_addr, 16, 1024);
      const uint64_t r2_desc = sdesc_sw128(r_addr + L::kRBytes, 16, 1024);
      const uint64_t c1_desc = sdesc_sw128(c1_addr, 16, 1024);
      const uint64_t c2_desc = sdesc_sw128(c2_addr, 16, 1024);
      constexpr int RC = (kRes * 128) >> 4;  // next 64-column chunk of a resident tile
      constexpr int CC = (kSub * 128) >> 4;  // next 64-column chunk of a streamed tile
      uint32_t r_round = 0;
      for (;;) {
        // the stage's full barrier also publishes the step's flags
        if (!sy.warp(bCFull + st, round & 1)) { ok = false; break; }
        const int flags = stage_flags[st];
        if (flags & kStop) break;
        if (flags & kFirst) {
          if (!sy.warp(bRFull, r_round & 1)) { ok = false; break; }
          ++r_round;
        }
        const uint32_t xb = n % L::NB;
        if (!sy.warp(bTSDone + xb, ((n / L::NB) & 1u) ^ 1u)) { ok = false; break; }
        tc_fence_after();
        const uint64_t cd1 = c1_desc + static_cast<uint64_t>(st * (L::kCBytes >> 4));
        const uint64_t cd2 = c2_desc + static_cast<uint64_t>(st * (L::kCBytes >> 4));
        if constexpr (D == 128) {
          umma_ss_group8<2, 2, 4, 4, 6, 6, RC, CC, RC + 2, CC + 2, RC + 4, CC + 4, RC + 6, CC + 6>(
              tmem_base + L::x_col(xb), r1_desc, cd1, kIdescXY, 0u);
          umma_ss_group8<2, 2, 4, 4, 6, 6, RC, CC, RC + 2, CC + 2, RC + 4, CC + 4, RC + 6, CC + 6>(
              tmem_base + L::y_col(xb), r2_desc, cd2, kIdescXY, 0u);
        } else {
          umma_ss_group4<2, 2, 4, 4, 6, 6>(tmem_base + L::x_col(xb), r1_desc, cd1, kIdescXY, 0u);
          umma_ss_group4<2, 2, 4, 4, 6, 6>(tmem_base + L::y_col(xb), r2_desc, cd2, kIdescXY, 0u);
        }
        umma_commit_elect(&bars[bSFull + xb]);
        if (flags & kLast) umma_commit_elect(&bars[bREmpty]);
        ++n;
        if (++st == L::NS) {
          st = 0;
          ++round;
        }
      }
    } else {
      // MN-major streamed operands of the accumulating MMAs (N = D across
      // the 64-column chunks, K = streamed rows)
      const uint64_t c1_mn = sdesc_sw128(c1_addr, kSub * 128, 1024);
      const uint64_t c2_mn = sdesc_sw128(c2_addr, kSub * 128, 1024);
      constexpr int KS = (16 * 128) >> 4;  // 16 streamed rows (one K step)
      uint32_t acc_round = 0;
      bool acc_pending = false;
      for (;;) {
        // P-full also publishes the step's flags (and the stop token)
        const uint32_t xb = n % L::NB;
        if (!sy.warp(bPFull + xb, (n / L::NB) & 1u)) { ok = false; break; }
        const int flags = buf_flags[xb];
        if (flags & kStop) break;
        const bool first = (flags & kFirst) != 0;
        if (first && acc_pending) {
          if (!sy.warp(bAccEmpty, acc_round & 1)) { ok = false; break; }
          ++acc_round;
          acc_pending = false;
        }
        tc_fence_after();
        const uint64_t m1 = c1_mn + static_cast<uint64_t>(st * (L::kCBytes >> 4));
        const uint64_t m2 = c2_mn + static_cast<uint64_t>(st * (L::kCBytes >> 4));
        const uint32_t acc = first ? 0u : 1u;
        if (Mode == kModeDQ) {
          // dQ += dS K
          umma_ts_group4_split<KS>(tmem_base + L::kAcc0, tmem_base + L::y_col(xb), m1, kIdescAcc,
                                   acc);
        } else {
          // dV += P^T dO, dK += dS^T Q
          umma_ts_group4_split<KS>(tmem_base + L::kAcc0, tmem_base + L::x_col(xb), m2, kIdescAcc,
                                   acc);
          umma_ts_group4_split<KS>(tmem_base + L::kAcc1, tmem_base + L::y_col(xb), m1, kIdescAcc,
                                   acc);
        }
        umma_commit_elect(&bars[bTSDone + xb]);
        umma_commit_elect(&bars[bCEmpty + st]);
        if (flags & kLast) {
          umma_commit_elect(&bars[bAccFull]);
          acc_pending = true;
        }
        ++n;
        if (++st == L::NS) {
          st = 0;
          ++round;
        }
      }
    }
    (void)ok;
    // all MMAs this issuer issued complete before TMEM is released
    umma_commit_elect(&bars[bDrain + me]);
    mbar_wait_bounded(&bars[bDrain + me], 0, 100000000ull, nullptr);
    bwd_teardown<D, Mode>(tmem_slot, warp);
    return;
  } else {
    bwd_teardown<D, Mode>(tmem_slot, warp);  // idle warp
  }
}

// Warps 4..11: P, dS and the epilogue, two warpgroups.  Both take every
// step; warpgroup w handles streamed columns [32 w, 32 w + 32) of it, which
// halves the time from X / Y ready to P / dS written (the part of a step the
// tensor cores wait for).  Thread = TMEM lane = resident row.  At the end of
// an item warpgroup 0 writes dQ columns [0, D/2) or dV, warpgroup 1 dQ
// columns [D/2, D) or dK.
template <int D, int Mode, typename IdxT>
__device__ __forceinline__ void bwd_elementwise_role(const AttnBwdParams& p) {
  using L = BwdLayout<D, Mode>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  const BwdMeta* meta = reinterpret_cast<const BwdMeta*>(smem + L::kMeta);
  const uint8_t* slots = smem + L::kSlots;
  volatile int* buf_flags = reinterpret_cast<volatile int*>(smem + L::kBufFlags);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = static_cast<int>(p.T);
  const Sync sy{bars, abort_flag, p.timeout_ns, &p.ws->error_word, lane};
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  const int wg = (warp - 4) >> 2;  // which 32 streamed columns
  const int row = (warp & 3) * 32 + lane;
  const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const bool causal = p.causal != 0;
  const uint64_t c2 = pack_f32x2(p.scale_log2, p.scale_log2);
  uint32_t mslot = 0, mround = 0, n_steps = 0, acc_cnt = 0;
  // dQ: -lse*log2(e) and -delta of this row; dK/dV: intervals of this key
  float nl_row = -CUDART_INF_F, nd_row = 0.f;
  int lts = 0, lte = 0, uts = 0, ute = 0, cur_mh = -1;

  for (;;) {
    if (!sy.warp(bMFull + mslot, mround & 1)) break;
    const int4 ma = *reinterpret_cast<const int4*>(meta + mslot);      // flags, cls, c0, r0
    const int4 mb = *(reinterpret_cast<const int4*>(meta + mslot) + 1);  // b, h, kvh, mh
    const int flags = ma.x;
    const uint32_t xb = n_steps % L::NB;
    if (flags & kStop) {
      // pass the stop token to the accumulating issuer through the next
      // buffer, once the issuer has taken the flags of that buffer's previous
      // step (its MMAs for that step are done)
      if (!sy.warp(bTSDone + xb, ((n_steps / L::NB) & 1u) ^ 1u)) break;
      if (warp == 4 && lane == 0) buf_flags[xb] = kStop;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[bPFull + xb]);
      break;
    }
    const int cls = ma.y, c0 = ma.z, r0 = ma.w;
    const int b = mb.x, h = mb.y, kvh = mb.z, mh = mb.w;
    const int r = r0 + row;  // resident row of this thread
    const uint32_t cur_slot = mslot;
    if (++mslot == kBwdMeta) {
      mslot = 0;
      ++mround;
    }
    // element mask of this warpgroup's 32 streamed columns (bit set = masked)
    uint32_t mbits = 0u;
    const int cw = c0 + 32 * wg;  // first column of the warpgroup
    if (Mode == kModeDQ) {
      if (flags & kFirst) {
        nl_row = -CUDART_INF_F;
        nd_row = 0.f;
        if (r < T) {
          const IdxT o = static_cast<IdxT>(h) * static_cast<IdxT>(p.T) + static_cast<IdxT>(r);
          nl_row = __ldg(p.nlse2 + o);
          nd_row = __ldg(p.ndelta + o);
        }
      }
      // columns = keys cw + j; from `valid` on they are outside the sample
      const int valid = b - cw;
      if (cls == kClsPC) {
        mbits = range_bits(r - cw + 1, 32, 0) | range_bits(valid, 32, 0);
      } else if (cls == kClsP) {
        const int* cl = reinterpret_cast<const int*>(slots + cur_slot * kSlotBytes) + 32 * wg;
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const int4 a4 = *reinterpret_cast<const int4*>(cl + i);
          const int4 e4 = *reinterpret_cast<const int4*>(cl + kSub + i);
          const int4 ua4 = *reinterpret_cast<const int4*>(cl + 2 * kSub + i);
          const int4 ue4 = *reinterpret_cast<const int4*>(cl + 3 * kSub + i);
          const int av[4] = {a4.x, a4.y, a4.z, a4.w};
          const int ev[4] = {e4.x, e4.y, e4.z, e4.w};
          const int uav[4] = {ua4.x, ua4.y, ua4.z, ua4.w};
          const int uev[4] = {ue4.x, ue4.y, ue4.z, ue4.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const bool lower = r >= cw + i + q;
            const bool in_lt = (av[q] <= r) & (r < ev[q]);
            const bool in_ut = causal | ((uav[q] <= r) & (r < uev[q]));
            const bool m = (i + q >= valid) | (lower ? in_lt : in_ut);
            mbits |= static_cast<uint32_t>(m) << (i + q);
          }
        }
      } else {
        mbits = range_bits(valid, 32, 0);
      }
    } else {
      // columns = queries cw + j; rows outside the sample already carry
      // -lse*log2(e) = -inf
      if (flags & kFirst) cur_mh = -1;  // new key rows
      if (cls == kClsP && mh != cur_mh) {
        cur_mh = mh;
        lts = lte = uts = ute = 0;
        if (r < T) {
          const int32_t* src = p.sri + static_cast<int64_t>(mh) * 4 * p.T + r;
          lts = __ldg(src);
          lte = __ldg(src + p.T);
          uts = __ldg(src + 2 * p.T);
          ute = __ldg(src + 3 * p.T);
        }
      }
      if (cls == kClsPC) {
        // query rows above the key (i < j) are masked
        mbits = range_bits(0, r - cw, 0);
      } else if (cls == kClsP) {
        // i >= j: masked iff LTS <= i < LTE; i < j: iff causal or UTS <= i < UTE
        const int lo0 = max(lts, r) - cw, lo1 = lte - cw;
        const int up0 = causal ? 0 : uts - cw;
        const int up1 = (causal ? r : min(ute, r)) - cw;
        mbits = range_bits(lo0, lo1, 0) | range_bits(up0, up1, 0);
      }
    }

    if (!sy.warp(bSFull + xb, (n_steps / L::NB) & 1u)) break;
    tc_fence_after();
    const uint32_t x_t = tmem_base + lane_addr + L::x_col(xb);
    const uint32_t y_t = tmem_base + lane_addr + L::y_col(xb);
    {
      uint32_t xr[32], yr[32];
      tmem_ld32_pair(x_t + 32 * wg, y_t + 32 * wg, xr, yr);
      if (mbits != 0u) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if ((mbits >> j) & 1u) xr[j] = __float_as_uint(-CUDART_INF_F);
      }
      const float* nl_col = reinterpret_cast<const float*>(slots + cur_slot * kSlotBytes) + 32 * wg;
      const float* nd_col = nl_col + kSub;
      uint32_t pk[16], dk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        uint64_t nl2a, nl2b, nd2a, nd2b;
        if (Mode == kModeDQ) {
          nl2a = nl2b = pack_f32x2(nl_row, nl_row);
          nd2a = nd2b = pack_f32x2(nd_row, nd_row);
        } else {
          const float4 a4 = *reinterpret_cast<const float4*>(nl_col + j);
          const float4 d4 = *reinterpret_cast<const float4*>(nd_col + j);
          nl2a = pack_f32x2(a4.x, a4.y);
          nl2b = pack_f32x2(a4.z, a4.w);
          nd2a = pack_f32x2(d4.x, d4.y);
          nd2b = pack_f32x2(d4.z, d4.w);
        }
        bwd_pair(xr[j], xr[j + 1], yr[j], yr[j + 1], c2, nl2a, nd2a, pk[j >> 1], dk[j >> 1]);
        bwd_pair(xr[j + 2], xr[j + 3], yr[j + 2], yr[j + 3], c2, nl2b, nd2b, pk[(j >> 1) + 1],
                 dk[(j >> 1) + 1]);
      }
      // bf16 pairs of columns [32 w, 32 w + 32) go to packed columns
      // [32 w, 32 w + 16): each warpgroup overwrites only columns it has
      // read itself.  The accumulating MMAs read the packed operand at
      // column offsets 0, 8 (streamed rows 0..31) and 32, 40 (rows 32..63).
      if (Mode == kModeDKV) tmem_st16(x_t + 32 * wg, pk);
      tmem_st16(y_t + 32 * wg, dk);
    }
    tmem_st_wait();
    tc_fence_before();
    if (warp == 4 && lane == 0) buf_flags[xb] = flags;
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[bPFull + xb]);

    if (flags & kLast) {
      if (!sy.warp(bAccFull, acc_cnt & 1u)) break;
      ++acc_cnt;
      tc_fence_after();
      const bool store = r < b;
      const int heads = Mode == kModeDQ ? p.hq : p.hkv;
      const int hh = Mode == kModeDQ ? h : kvh;
      const IdxT off = (static_cast<IdxT>(store ? r : 0) * heads + hh) * static_cast<IdxT>(D);
      // dQ columns [wg D/2, wg D/2 + D/2) (scaled); dV (unscaled) or dK (scaled)
      constexpr int kCols = Mode == kModeDQ ? D / 2 : D;
      const float f = (Mode == kModeDKV && wg == 0) ? 1.f : p.scale;
      __nv_bfloat16* dst =
          static_cast<__nv_bfloat16*>(Mode == kModeDQ ? p.dq : (wg == 0 ? p.dv : p.dk)) + off +
          (Mode == kModeDQ ? wg * (D / 2) : 0);
      const uint32_t acc_t = tmem_base + lane_addr +
                             (Mode == kModeDQ ? L::kAcc0 + wg * (D / 2)
                                              : (wg == 0 ? L::kAcc0 : L::kAcc1));
      const uint64_t f2 = pack_f32x2(f, f);
#pragma unroll
      for (int c = 0; c < kCols / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(acc_t + c * 32, rr);
        if (store) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            d4[u] = make_uint4(scale_pack_bf16x2(rr[8 * u + 0], rr[8 * u + 1], f2),
                               scale_pack_bf16x2(rr[8 * u + 2], rr[8 * u + 3], f2),
                               scale_pack_bf16x2(rr[8 * u + 4], rr[8 * u + 5], f2),
                               scale_pack_bf16x2(rr[8 * u + 6], rr[8 * u + 7], f2));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[bAccEmpty]);
    }
    ++n_steps;
  }
  bwd_teardown<D, Mode>(tmem_slot, warp);
}

template <int D, int Mode, typename IdxT>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_kernel(const AttnBwdParams p, const __grid_constant__ CUtensorMap tr1,
                    const __grid_constant__ CUtensorMap tr2,
                    const __grid_constant__ CUtensorMap tc1,
                    const __grid_constant__ CUtensorMap tc2) {
  if ((threadIdx.x >> 5) < 4)
    bwd_producer_roles<D, Mode, IdxT>(p, tr1, tr2, tc1, tc2);
  else
    bwd_elementwise_role<D, Mode, IdxT>(p);
}

template <int D, int Mode, typename IdxT>
cudaError_t launch_mode(const AttnBwdParams& p, const CUtensorMap& tr1, const CUtensorMap& tr2,
                        const CUtensorMap& tc1, const CUtensorMap& tc2, int num_sms,
                        cudaStream_t stream) {
  using L = BwdLayout<D, Mode>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static unsigned long long configured = 0ull;  // one bit per device
  if (dev >= 64 || !((configured >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(attn_bwd_kernel<D, Mode, IdxT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured |= 1ull << dev;
  }
  e = launch_pdl(bwd_plan_order_kernel<Mode>, dim3(1), dim3(kCostBins), 0, stream, p);
  if (e != cudaSuccess) return e;
  const int64_t items = p.n_res_slots * (Mode == kModeDQ ? p.hq : p.hkv);
  const int grid = static_cast<int>(items < num_sms ? items : num_sms);
  return launch_pdl(attn_bwd_kernel<D, Mode, IdxT>, dim3(grid), dim3(kBwdThreads), L::kBytes,
                    stream, p, tr1, tr2, tc1, tc2);
}

template <int D, typename IdxT>
cudaError_t launch_all(const AttnBwdParams& p, const BwdMaps& m, int num_sms,
                       cudaStream_t stream) {
  const int64_t rows = p.T * p.hq;
  const int64_t blocks = (rows * (D / 8) + 255) / 256;
  cudaError_t e = launch_pdl(bwd_prep_kernel<D, IdxT>, dim3(static_cast<unsigned>(blocks)),
                             dim3(256), 0, stream, p);
  if (e != cudaSuccess) return e;
  AttnBwdParams pp = p;
  pp.num_sms = num_sms;
  e = launch_mode<D, kModeDKV, IdxT>(pp, m.k128, m.v128, m.q64, m.do64, num_sms, stream);
  if (e != cudaSuccess) return e;
  return launch_mode<D, kModeDQ, IdxT>(pp, m.q128, m.do128, m.k64, m.v64, num_sms, stream);
}

}  // namespace

// Workspace: header (initialised by the planners) | order_q | order_kv (n_slots ints
// each) | -lse*log2(e) | -delta ([Hq][T] floats each).
size_t attn_bwd_clear_bytes() { return sizeof(AttnWorkspaceHeader); }

size_t attn_bwd_workspace_bytes(int64_t T, int n_seqs, int n_heads_q) {
  const int64_t n_slots = T / kRes + n_seqs;
  size_t bytes = attn_bwd_clear_bytes() + 2 * static_cast<size_t>(n_slots) * sizeof(int);
  bytes = (bytes + 15) & ~static_cast<size_t>(15);
  bytes += 2 * static_cast<size_t>(T) * n_heads_q * sizeof(float);
  return (bytes + 255) & ~static_cast<size_t>(255);
}

void attn_bwd_bind_workspace(AttnBwdParams& p, void* workspace, int64_t T, int n_seqs,
                             int n_heads_q) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int64_t n_slots = T / kRes + n_seqs;
  p.ws = reinterpret_cast<AttnWorkspaceHeader*>(ws);
  int* ints = reinterpret_cast<int*>(ws + sizeof(AttnWorkspaceHeader));
  p.order_q = ints;
  p.order_kv = ints + n_slots;
  size_t off = attn_bwd_clear_bytes() + 2 * static_cast<size_t>(n_slots) * sizeof(int);
  off = (off + 15) & ~static_cast<size_t>(15);
  p.nlse2 = reinterpret_cast<float*>(ws + off);
  p.ndelta = p.nlse2 + T * n_heads_q;
}

cudaError_t launch_attn_bwd(const AttnBwdParams& p, const BwdMaps& maps, bool use_int64,
                            int num_sms, cudaStream_t stream) {
  if (p.head_dim == 128)
    return use_int64 ? launch_all<128, int64_t>(p, maps, num_sms, stream)
                     : launch_all<128, int32_t>(p, maps, num_sms, stream);
  return use_int64 ? launch_all<64, int64_t>(p, maps, num_sms, stream)
                   : launch_all<64, int32_t>(p, maps, num_sms, stream);
}

}  // namespace fm
