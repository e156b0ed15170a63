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
// access touches whole 128-byte lines.  A thread first issues the loads of
// all its heads, then finds its sample and computes the angles while they
// are in flight.  Launch shape measured on GB300 (q + k of 8192 to 131072
// tokens, 40 to 64 heads, L2 flushed): groups of 8 heads in 128-thread CTAs
// beat 256-thread CTAs and groups of 2 to 10 heads, and loading after the
// sample search, by 5 to 15 %.
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

constexpr int kThreads = 128;
// Heads per thread: the eight (cos, sin) pairs a thread computes serve a
// group of eight heads.  The C ABI limits q + k heads to 8 * 65535, so the
// groups always fit grid y.
constexpr int kGroup = 8;

template <typename IdxT, int D>
__global__ void __launch_bounds__(kThreads) rope_qk_varlen_kernel(
    __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ k, IdxT n_threads_x, int hq,
    int hkv, IdxT q_stride, IdxT k_stride, const int32_t* __restrict__ cu, int n_seqs,
    float sin_sign, const __grid_constant__ RopeFreqs freqs) {
  constexpr int kChunks = D / 16;  // 16-byte chunks per half row
  pdl_trigger();
  pdl_wait();
  const IdxT gid = static_cast<IdxT>(blockIdx.x) * kThreads + threadIdx.x;
  if (gid >= n_threads_x) return;
  const IdxT t = gid / kChunks;
  const int c = static_cast<int>(gid % kChunks);
  const int h_begin = blockIdx.y * kGroup;
  const int h_end = min(h_begin + kGroup, hq + hkv);

  // The group's head rows first: their loads do not depend on the position,
  // so they are in flight while the sample search and the angles run.
  auto row_of = [&](int h) -> __nv_bfloat16* {
    return (h < hq) ? q + t * q_stride + static_cast<IdxT>(h) * D
                    : k + t * k_stride + static_cast<IdxT>(h - hq) * D;
  };
  uint4 x1[kGroup], x2[kGroup];
#pragma unroll
  for (int j = 0; j < kGroup; ++j) {
    if (h_begin + j < h_end) {
      const __nv_bfloat16* row = row_of(h_begin + j);
      x1[j] = *reinterpret_cast<const uint4*>(row + c * 8);
      x2[j] = *reinterpret_cast<const uint4*>(row + D / 2 + c * 8);
    }
  }

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

#pragma unroll
  for (int j = 0; j < kGroup; ++j) {
    if (h_begin + j < h_end) {
      __nv_bfloat16* row = row_of(h_begin + j);
      uint4 y1, y2;
      rope_rotate8(x1[j], x2[j], cs, sn, y1, y2);
      *reinterpret_cast<uint4*>(row + c * 8) = y1;
      *reinterpret_cast<uint4*>(row + D / 2 + c * 8) = y2;
    }
  }
}

template <typename IdxT, int D>
cudaError_t launch_typed(void* q, void* k, int64_t T, int hq, int hkv, int64_t q_stride,
                         int64_t k_stride, const int32_t* cu, int n_seqs, const RopeFreqs& fr,
                         bool backward, cudaStream_t stream) {
  const int64_t n = T * (D / 16);
  const int64_t blocks_x = (n + kThreads - 1) / kThreads;
  const int groups = (hq + hkv + kGroup - 1) / kGroup;
  if (blocks_x > 0x7FFFFFFFLL || groups > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid(static_cast<unsigned>(blocks_x), static_cast<unsigned>(groups));
  return launch_pdl(rope_qk_varlen_kernel<IdxT, D>, grid, dim3(kThreads), 0, stream,
                    static_cast<__nv_bfloat16*>(q), static_cast<__nv_bfloat16*>(k),
                    static_cast<IdxT>(n), hq, hkv, static_cast<IdxT>(q_stride),
                    static_cast<IdxT>(k_stride), cu, n_seqs, backward ? -1.0f : 1.0f, fr);
}

}  // namespace

cudaError_t launch_rope(void* q, void* k, int64_t T, int hq, int hkv, int head_dim,
                        int64_t q_stride, int64_t k_stride, const int32_t* cu, int n_seqs,
                        const RopeFreqs& freqs, bool backward, bool use_int64, int num_sms,
                        cudaStream_t stream) {
  (void)num_sms;  // the grid covers every (token chunk, head group) once
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
