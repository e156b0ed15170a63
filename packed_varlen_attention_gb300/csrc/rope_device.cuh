// rope_device.cuh -- the RoPE rotation of one pair of 8-channel chunks.
//
// Unsloth packing blog, section "Fused QK RoPE Triton kernel with packing":
// Y = X*cos + rotate_half(X)*sin, where channel i < D/2 pairs with channel
// i + D/2 and the angle of channel i at position p is p * theta^(-2i/D).
// Backward flips the sign of sin.
//
// Shared by the stand-alone RoPE kernel and the attention kernel's fused Q
// prologue, so that both produce the same bits for the same token.
//
// Angle accuracy: positions reach 65535 and more, where an fp32 product
// p * f is off by up to ~4e-3 rad.  The angle is therefore formed as a
// double-float: f = f_hi + f_lo (host, double precision), p * f_hi split
// exactly with an FMA (two-product), then reduced modulo 2*pi by the
// Cody-Waite method with a two-part 2*pi whose first part multiplies exactly
// inside the FMA.  The reduced |r| <= pi + tiny goes to the hardware
// sin/cos, whose absolute error there is about 2^-21.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "fm_device.cuh"

namespace fm {

// 2*pi split: kTwoPiHi = fp32(2*pi), kTwoPiLo = fp32(2*pi - kTwoPiHi).
constexpr float kRopeTwoPiHi = 6.28318548202514648f;
constexpr float kRopeTwoPiLo = -1.74845553146951715e-07f;
constexpr float kRopeInvTwoPi = 0.159154936671257019f;

// cos(p * f) and sin_sign * sin(p * f) for f = fh + fl.
__device__ __forceinline__ void rope_cos_sin(float pos, float fh, float fl, float sin_sign,
                                             float& co, float& sn) {
  const float a_hi = pos * fh;
  const float a_err = fmaf(pos, fh, -a_hi);  // exact remainder of pos * fh
  const float a_lo = fmaf(pos, fl, a_err);
  const float kq = rintf(a_hi * kRopeInvTwoPi);
  float r = fmaf(-kq, kRopeTwoPiHi, a_hi);  // exact product inside the FMA
  r = fmaf(-kq, kRopeTwoPiLo, r);
  r += a_lo;
  float s, c;
  __sincosf(r, &s, &c);
  co = c;
  sn = s * sin_sign;
}

// x1: eight consecutive channels of the first half row, x2: their partners
// in the second half; cs/sn: cos and (signed) sin of the eight angles.
// First half: x1*cos - x2*sin; second half: x2*cos + x1*sin.
__device__ __forceinline__ void rope_rotate8(const uint4& x1, const uint4& x2,
                                             const float (&cs)[8], const float (&sn)[8],
                                             uint4& y1, uint4& y2) {
  const uint32_t a[4] = {x1.x, x1.y, x1.z, x1.w};
  const uint32_t b[4] = {x2.x, x2.y, x2.z, x2.w};
  uint32_t o1[4], o2[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float2 u = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a[w]));
    const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b[w]));
    const float c0 = cs[2 * w], c1 = cs[2 * w + 1];
    const float s0 = sn[2 * w], s1 = sn[2 * w + 1];
    o1[w] = pack_bf16x2(fmaf(u.x, c0, -v.x * s0), fmaf(u.y, c1, -v.y * s1));
    o2[w] = pack_bf16x2(fmaf(v.x, c0, u.x * s0), fmaf(v.y, c1, u.y * s1));
  }
  y1 = make_uint4(o1[0], o1[1], o1[2], o1[3]);
  y2 = make_uint4(o2[0], o2[1], o2[2], o2[3]);
}

}  // namespace fm
