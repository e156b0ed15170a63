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
// Angle accuracy: positions reach 65535 and more, where an fp32 product
// p * f is off by up to ~4e-3 rad.  The angle is therefore formed as a
// double-float: f = f_hi + f_lo (host, double precision), p * f_hi split
// exactly with an FMA (two-product), then reduced modulo 2*pi by the
// Cody-Waite method with a two-part 2*pi whose first part multiplies exactly
// inside the FMA.  The reduced |r| <= pi + tiny goes to the hardware
// sin/cos, whose absolute error there is about 2^-21.
#include <cuda_bf16.h>

#include "fm_device.cuh"
#include "fm_internal.h"

namespace fm {
namespace {

// 2*pi split: kTwoPiHi = fp32(2*pi), kTwoPiLo = fp32(2*pi - kTwoPiHi).
constexpr float kTwoPiHi = 6.28318548202514648f;
constexpr float kTwoPiLo = -1.74845553146951715e-07f;
constexpr float kInvTwoPi = 0.159154936671257019f;
constexpr int kHeadsPerGroup = 8;
constexpr int kThreads = 256;

template <typename IdxT, int D>
__global__ void __launch_bounds__(kThreads) rope_qk_varlen_kernel(
    __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ k, IdxT n_threads_x, int hq,
    int hkv, IdxT q_stride, IdxT k_stride, const int32_t* __restrict__ cu, int n_seqs,
    float sin_sign, const __grid_constant__ RopeFreqs freqs) {
  constexpr int kChunks = D / 16;  // 16-byte chunks per half row
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
  for (int i = 0; i < 8; ++i) {
    const float fh = freqs.hi[c * 8 + i];
    const float fl = freqs.lo[c * 8 + i];
    const float a_hi = pos * fh;
    const float a_err = fmaf(pos, fh, -a_hi);  // exact remainder of pos * fh
    const float a_lo = fmaf(pos, fl, a_err);
    const float kq = rintf(a_hi * kInvTwoPi);
    float r = fmaf(-kq, kTwoPiHi, a_hi);  // exact product inside the FMA
    r = fmaf(-kq, kTwoPiLo, r);
    r += a_lo;
    float s, co;
    __sincosf(r, &s, &co);
    cs[i] = co;
    sn[i] = s * sin_sign;
  }

  const int h_begin = blockIdx.y * kHeadsPerGroup;
  const int h_total = hq + hkv;
  const int h_end = min(h_begin + kHeadsPerGroup, h_total);
#pragma unroll 4
  for (int h = h_begin; h < h_end; ++h) {
    __nv_bfloat16* row = (h < hq) ? q + t * q_stride + static_cast<IdxT>(h) * D
                                  : k + t * k_stride + static_cast<IdxT>(h - hq) * D;
    uint4* p1 = reinterpret_cast<uint4*>(row + c * 8);
    uint4* p2 = reinterpret_cast<uint4*>(row + D / 2 + c * 8);
    const uint4 x1 = *p1;
    const uint4 x2 = *p2;
    const uint32_t a[4] = {x1.x, x1.y, x1.z, x1.w};
    const uint32_t b[4] = {x2.x, x2.y, x2.z, x2.w};
    uint32_t y1[4], y2[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float2 u = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a[w]));
      const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b[w]));
      const float c0 = cs[2 * w], c1 = cs[2 * w + 1];
      const float s0 = sn[2 * w], s1 = sn[2 * w + 1];
      // first half: x1*cos - x2*sin ; second half: x2*cos + x1*sin
      y1[w] = pack_bf16x2(fmaf(u.x, c0, -v.x * s0), fmaf(u.y, c1, -v.y * s1));
      y2[w] = pack_bf16x2(fmaf(v.x, c0, u.x * s0), fmaf(v.y, c1, u.y * s1));
    }
    *p1 = make_uint4(y1[0], y1[1], y1[2], y1[3]);
    *p2 = make_uint4(y2[0], y2[1], y2[2], y2[3]);
  }
}

template <typename IdxT, int D>
cudaError_t launch_typed(void* q, void* k, int64_t T, int hq, int hkv, int64_t q_stride,
                         int64_t k_stride, const int32_t* cu, int n_seqs, const RopeFreqs& fr,
                         bool backward, cudaStream_t stream) {
  const int64_t n = T * (D / 16);
  const int64_t blocks_x = (n + kThreads - 1) / kThreads;
  const int groups = (hq + hkv + kHeadsPerGroup - 1) / kHeadsPerGroup;
  if (blocks_x > 0x7FFFFFFFLL || groups > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid(static_cast<unsigned>(blocks_x), static_cast<unsigned>(groups));
  rope_qk_varlen_kernel<IdxT, D><<<grid, kThreads, 0, stream>>>(
      static_cast<__nv_bfloat16*>(q), static_cast<__nv_bfloat16*>(k), static_cast<IdxT>(n), hq,
      hkv, static_cast<IdxT>(q_stride), static_cast<IdxT>(k_stride), cu, n_seqs,
      backward ? -1.0f : 1.0f, fr);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope(void* q, void* k, int64_t T, int hq, int hkv, int head_dim,
                        int64_t q_stride, int64_t k_stride, const int32_t* cu, int n_seqs,
                        const RopeFreqs& freqs, bool backward, bool use_int64,
                        cudaStream_t stream) {
  if (head_dim == 128) {
    return use_int64 ? launch_typed<int64_t, 128>(q, k, T, hq, hkv, q_stride, k_stride, cu,
                                                  n_seqs, freqs, backward, stream)
                     : launch_typed<int32_t, 128>(q, k, T, hq, hkv, q_stride, k_stride, cu,
                                                  n_seqs, freqs, backward, stream);
  }
  return use_int64 ? launch_typed<int64_t, 64>(q, k, T, hq, hkv, q_stride, k_stride, cu, n_seqs,
                                               freqs, backward, stream)
                   : launch_typed<int32_t, 64>(q, k, T, hq, hkv, q_stride, k_stride, cu, n_seqs,
                                               freqs, backward, stream);
}

}  // namespace fm
