// rope_varlen.cu -- fused, in-place QK RoPE over packed samples.
//
// Unsloth packing blog, section "Fused QK RoPE Triton kernel with packing":
// one launch rotates q and k together, Y = X*cos + rotate_half(X)*sin, with
// positions restarting at every sample boundary; backward flips the sign of
// sin.  The community change cited there (one program per group of heads)
// is kept: a thread owns one token and eight frequency pairs, computes the
// eight (cos, sin) pairs once and applies them to a group of heads.
//
// Memory: every q/k element is read once and written once with 16-byte
// accesses (8 bf16).  For one head, eight consecutive threads cover the
// first half-row (128 B) and the second half-row of a token, so each warp
// access touches whole 128-byte lines.
//
// The angle (double-float, Cody-Waite reduction) and the rotation of a chunk
// pair live in rope_device.cuh, shared with the attention kernel's fused Q
// prologue.
#include <cuda_bf16.h>

#include "fm_device.cuh"
#include "rope_device.cuh"
#include "fm_internal.h"

namespace fm {
namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 8;  // 256 threads x 8 = 2048 threads resident per SM

template <typename IdxT, int D>
__global__ void __launch_bounds__(kThreads) rope_qk_varlen_kernel(
    __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ k, IdxT n_threads_x, int hq,
    int hkv, IdxT q_stride, IdxT k_stride, const int32_t* __restrict__ cu, int n_seqs,
    float sin_sign, int heads_per_group, const __grid_constant__ RopeFreqs freqs) {
  constexpr int kChunks = D / 16;  // 16-byte chunks per half row
  pdl_trigger();
  pdl_wait();
  const IdxT gid = static_cast<IdxT>(blockIdx.x) * kThreads + threadIdx.x;
  if (gid >= n_threads_x) return;
  const IdxT t = gid / kChunks;
  const int c = static_cast<int>(gid % kChunks);

  // sample of token t: largest s with cu[s] <= t
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<IdxT>(__ldg(cu + mid)) <= t) lo = mid; else hi = mid - 1;
  }
  long long pos_ll = static_cast<long long>(t) - __ldg(cu + lo);
  pos_ll = pos_ll < 0 ? 0 : pos_ll;
  const float pos = static_cast<float>(pos_ll);

  float cs[8], sn[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    rope_cos_sin(pos, freqs.hi[c * 8 + i], freqs.lo[c * 8 + i], sin_sign, cs[i], sn[i]);

  const int h_begin = blockIdx.y * heads_per_group;
  const int h_total = hq + hkv;
  const int h_end = min(h_begin + heads_per_group, h_total);
#pragma unroll 4
  for (int h = h_begin; h < h_end; ++h) {
    __nv_bfloat16* row = (h < hq) ? q + t * q_stride + static_cast<IdxT>(h) * D
                                  : k + t * k_stride + static_cast<IdxT>(h - hq) * D;
    uint4* p1 = reinterpret_cast<uint4*>(row + c * 8);
    uint4* p2 = reinterpret_cast<uint4*>(row + D / 2 + c * 8);
    const uint4 x1 = *p1;
    const uint4 x2 = *p2;
    uint4 y1, y2;
    rope_rotate8(x1, x2, cs, sn, y1, y2);
    *p1 = y1;
    *p2 = y2;
  }
}

// Heads per thread: eight amortise the eight (cos, sin) pairs best, but a
// grid of few CTAs (a short batch, or the key heads alone) then ends in a
// partial wave of long CTAs.  Eight when that still gives at least four
// waves of resident CTAs, else four (measured best for short grids; two
// and one lose to the extra angle arithmetic).  Grid y is limited to 65535
// groups; eight heads per group always fit the head counts the C ABI
// accepts.
int heads_per_group(int64_t blocks_x, int n_heads, int num_sms) {
  const int64_t wave = static_cast<int64_t>(num_sms) * kCtasPerSm;
  const int g = (blocks_x * ((n_heads + 7) / 8) >= 4 * wave) ? 8 : 4;
  return ((n_heads + g - 1) / g > 65535) ? 8 : g;
}

template <typename IdxT, int D>
cudaError_t launch_typed(void* q, void* k, int64_t T, int hq, int hkv, int64_t q_stride,
                         int64_t k_stride, const int32_t* cu, int n_seqs, const RopeFreqs& fr,
                         bool backward, int num_sms, cudaStream_t stream) {
  const int64_t n = T * (D / 16);
  const int64_t blocks_x = (n + kThreads - 1) / kThreads;
  const int hpg = heads_per_group(blocks_x, hq + hkv, num_sms);
  const int groups = (hq + hkv + hpg - 1) / hpg;
  if (blocks_x > 0x7FFFFFFFLL || groups > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid(static_cast<unsigned>(blocks_x), static_cast<unsigned>(groups));
  return launch_pdl(rope_qk_varlen_kernel<IdxT, D>, grid, dim3(kThreads), 0, stream,
                    static_cast<__nv_bfloat16*>(q), static_cast<__nv_bfloat16*>(k),
                    static_cast<IdxT>(n), hq, hkv, static_cast<IdxT>(q_stride),
                    static_cast<IdxT>(k_stride), cu, n_seqs, backward ? -1.0f : 1.0f, hpg, fr);
}

}  // namespace

cudaError_t launch_rope(void* q, void* k, int64_t T, int hq, int hkv, int head_dim,
                        int64_t q_stride, int64_t k_stride, const int32_t* cu, int n_seqs,
                        const RopeFreqs& freqs, bool backward, bool use_int64, int num_sms,
                        cudaStream_t stream) {
  if (head_dim == 128) {
    return use_int64 ? launch_typed<int64_t, 128>(q, k, T, hq, hkv, q_stride, k_stride, cu,
                                                  n_seqs, freqs, backward, num_sms, stream)
                     : launch_typed<int32_t, 128>(q, k, T, hq, hkv, q_stride, k_stride, cu,
                                                  n_seqs, freqs, backward, num_sms, stream);
  }
  return use_int64 ? launch_typed<int64_t, 64>(q, k, T, hq, hkv, q_stride, k_stride, cu, n_seqs,
                                               freqs, backward, num_sms, stream)
                   : launch_typed<int32_t, 64>(q, k, T, hq, hkv, q_stride, k_stride, cu, n_seqs,
                                               freqs, backward, num_sms, stream);
}

}  // namespace fm
