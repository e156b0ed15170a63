// mask_minmax.cu -- FlashMask preprocessing: per key tile, the minimum and
// maximum of each column-interval vector (PaddleNLP FlashMask article,
// section 3.1: eight vectors LTStart/LTEnd/UTStart/UTEnd min/max).
//
// One warp per (mask head, tile slot).  Tiles are sample-local and live in
// slot floor(cu[s] / Bc) + s + j (tile j of sample s), so a slot finds its
// sample with one binary search over cu_seqlens and no prefix sum is needed.
// The warp reads the tile's columns of the four vectors with coalesced loads
// and reduces them with warp-wide min/max; lane 0 writes the eight numbers.
#include "fm_device.cuh"
#include "fm_internal.h"

namespace fm {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int BN>
__global__ void __launch_bounds__(kThreads) mask_block_minmax_kernel(
    const int32_t* __restrict__ sri, int hm, int64_t T, const int32_t* __restrict__ cu,
    int n_seqs, int32_t* __restrict__ out, int64_t n_slots) {
  pdl_trigger();
  pdl_wait();
  const int64_t warp_global = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (warp_global >= n_slots * hm) return;
  const int h = static_cast<int>(warp_global / n_slots);
  const int64_t slot = warp_global % n_slots;

  // sample owning this slot: largest s with floor(cu[s] / BN) + s <= slot
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int64_t base = static_cast<int64_t>(__ldg(cu + mid)) / BN + mid;
    if (base <= slot) lo = mid; else hi = mid - 1;
  }
  const int64_t a = min(max(static_cast<int64_t>(__ldg(cu + lo)), int64_t(0)), T);
  const int64_t b = min(max(static_cast<int64_t>(__ldg(cu + lo + 1)), a), T);
  const int64_t j = slot - (a / BN + lo);
  const int64_t c0 = a + j * BN;
  const int64_t c1 = min(c0 + BN, b);
  const bool valid = (j >= 0) && (c0 < b);

  int mn[4], mx[4];
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    mn[v] = INT32_MAX;
    mx[v] = INT32_MIN;
  }
  if (valid) {
    const int32_t* base = sri + static_cast<int64_t>(h) * 4 * T;
#pragma unroll
    for (int m = 0; m < BN / 32; ++m) {
      const int64_t c = c0 + m * 32 + lane;
      if (c < c1) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int x = __ldg(base + v * T + c);
          mn[v] = min(mn[v], x);
          mx[v] = max(mx[v], x);
        }
      }
    }
  }
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    mn[v] = __reduce_min_sync(0xffffffffu, mn[v]);
    mx[v] = __reduce_max_sync(0xffffffffu, mx[v]);
  }
  if (lane == 0) {
    int32_t* o = out + static_cast<int64_t>(h) * 8 * n_slots + slot;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      o[(2 * v) * n_slots] = mn[v];
      o[(2 * v + 1) * n_slots] = mx[v];
    }
  }
}

}  // namespace

cudaError_t launch_mask_minmax(const int32_t* sri, int n_mask_heads, int64_t T,
                               const int32_t* cu, int n_seqs, int block_n, int32_t* out,
                               int64_t n_slots, cudaStream_t stream) {
  const int64_t warps = n_slots * n_mask_heads;
  const int64_t blocks = (warps + kWarps - 1) / kWarps;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(blocks));
  if (block_n == 128)
    return launch_pdl(mask_block_minmax_kernel<128>, grid, dim3(kThreads), 0, stream, sri,
                      n_mask_heads, T, cu, n_seqs, out, n_slots);
  return launch_pdl(mask_block_minmax_kernel<64>, grid, dim3(kThreads), 0, stream, sri,
                    n_mask_heads, T, cu, n_seqs, out, n_slots);
}

}  // namespace fm
