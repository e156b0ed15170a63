// fm_api.cu -- the C ABI: argument validation, TMA descriptor encoding and
// kernel launches.  Nothing here allocates device memory or synchronises,
// except the two documented read-back helpers.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fm_internal.h"

namespace {

using fm::AttnParams;

constexpr int kMaxDevices = 64;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

struct DeviceInfo {
  bool known = false;
  bool supported = false;
  int num_sms = 0;
};

// Current device must be sm_103 (GB300); SM count cached per device.
fm_status device_info(int* num_sms) {
  static DeviceInfo info[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& d = info[dev];
  if (!d.known) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FM_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.num_sms = sms;
    d.known = true;
  }
  if (!d.supported) return FM_ERR_UNSUPPORTED;
  if (num_sms) *num_sms = d.num_sms;
  return FM_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

fm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FM_OK : FM_ERR_CUDA; }

// 2-D bf16 tensor map over [rows][cols] (cols contiguous) with a
// 64-column x box_rows box and 128-byte swizzle; out-of-range rows read 0.
bool make_map(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
              uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

int fm_version(void) { return 100; }

const char* fm_status_string(int status) {
  switch (status) {
    case FM_OK: return "FM_OK";
    case FM_ERR_INVALID_ARG: return "FM_ERR_INVALID_ARG";
    case FM_ERR_UNSUPPORTED: return "FM_ERR_UNSUPPORTED";
    case FM_ERR_ALIGNMENT: return "FM_ERR_ALIGNMENT";
    case FM_ERR_WORKSPACE: return "FM_ERR_WORKSPACE";
    case FM_ERR_CUDA: return "FM_ERR_CUDA";
    case FM_ERR_TIMEOUT: return "FM_ERR_TIMEOUT";
    case FM_ERR_DEVICE_DATA: return "FM_ERR_DEVICE_DATA";
    default: return "FM_ERR_UNKNOWN";
  }
}

fm_status fm_rope_qk_varlen(void* q, void* k, int64_t total_tokens, int n_heads_q,
                            int n_heads_kv, int head_dim, int64_t q_token_stride,
                            int64_t k_token_stride, const int32_t* cu_seqlens, int n_seqs,
                            double theta, int backward, uint32_t flags, void* stream) {
  if (total_tokens < 0 || n_heads_q < 1 || n_heads_kv < 0 || n_seqs < 1) return FM_ERR_INVALID_ARG;
  if (q == nullptr || cu_seqlens == nullptr || (n_heads_kv > 0 && k == nullptr))
    return FM_ERR_INVALID_ARG;
  if (!(theta > 0.0) || !std::isfinite(theta)) return FM_ERR_INVALID_ARG;
  if (flags & ~FM_FLAG_FORCE_INT64) return FM_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return FM_ERR_UNSUPPORTED;
  if (q_token_stride < static_cast<int64_t>(n_heads_q) * head_dim) return FM_ERR_INVALID_ARG;
  if (n_heads_kv > 0 && k_token_stride < static_cast<int64_t>(n_heads_kv) * head_dim)
    return FM_ERR_INVALID_ARG;
  if (!aligned(q, 16) || q_token_stride % 8 != 0) return FM_ERR_ALIGNMENT;
  if (n_heads_kv > 0 && (!aligned(k, 16) || k_token_stride % 8 != 0)) return FM_ERR_ALIGNMENT;
  if (n_heads_q + n_heads_kv > 8 * 65535) return FM_ERR_UNSUPPORTED;
  if (total_tokens == 0) return FM_OK;
  int num_sms = 0;
  fm_status st = device_info(&num_sms);
  if (st != FM_OK) return st;

  fm::RopeFreqs fr;
  std::memset(&fr, 0, sizeof(fr));
  for (int i = 0; i < head_dim / 2; ++i) {
    const double f = std::pow(theta, -2.0 * i / head_dim);
    fr.hi[i] = static_cast<float>(f);
    fr.lo[i] = static_cast<float>(f - static_cast<double>(fr.hi[i]));
  }
  const bool use64 = fm_rope_index_bits(total_tokens, n_heads_kv, head_dim, q_token_stride,
                                        k_token_stride, flags) == 64;
  return from_cuda(fm::launch_rope(q, k, total_tokens, n_heads_q, n_heads_kv, head_dim,
                                   q_token_stride, k_token_stride, cu_seqlens, n_seqs, fr,
                                   backward != 0, use64, num_sms,
                                   static_cast<cudaStream_t>(stream)));
}

int fm_rope_index_bits(int64_t total_tokens, int n_heads_kv, int head_dim,
                       int64_t q_token_stride, int64_t k_token_stride, uint32_t flags) {
  if (total_tokens < 0 || n_heads_kv < 0 || head_dim <= 0 || q_token_stride < 0 ||
      k_token_stride < 0)
    return -1;
  const int64_t lim = int64_t(1) << 31;
  const bool use64 = (flags & FM_FLAG_FORCE_INT64) != 0 || total_tokens * q_token_stride >= lim ||
                     (n_heads_kv > 0 && total_tokens * k_token_stride >= lim) ||
                     total_tokens * (head_dim / 16) >= lim;
  return use64 ? 64 : 32;
}

int fm_attn_index_bits(int64_t total_tokens, int n_heads_q, int n_heads_kv, int head_dim,
                       uint32_t flags) {
  if (total_tokens < 0 || n_heads_q < 0 || n_heads_kv < 0 || head_dim <= 0) return -1;
  const int64_t lim = int64_t(1) << 31;
  const bool use64 = (flags & FM_FLAG_FORCE_INT64) != 0 ||
                     total_tokens * n_heads_q * head_dim >= lim ||
                     total_tokens * n_heads_kv * head_dim >= lim;
  return use64 ? 64 : 32;
}

int64_t fm_num_kv_tiles_bound(int64_t total_tokens, int n_seqs, int block_n) {
  if (total_tokens < 0 || n_seqs < 0 || block_n <= 0) return -1;
  return total_tokens / block_n + n_seqs;
}

fm_status fm_mask_block_minmax(const int32_t* startend_row_indices, int n_mask_heads,
                               int64_t total_tokens, const int32_t* cu_seqlens, int n_seqs,
                               int block_n, int32_t* block_minmax,
                               int64_t block_minmax_capacity, void* stream) {
  if (startend_row_indices == nullptr || cu_seqlens == nullptr || block_minmax == nullptr)
    return FM_ERR_INVALID_ARG;
  if (n_mask_heads < 1 || n_seqs < 1 || total_tokens < 0 || total_tokens > INT32_MAX)
    return FM_ERR_INVALID_ARG;
  if (block_n != 64 && block_n != 128) return FM_ERR_UNSUPPORTED;
  const int64_t n_slots = fm_num_kv_tiles_bound(total_tokens, n_seqs, block_n);
  if (block_minmax_capacity < n_slots * 8 * n_mask_heads) return FM_ERR_WORKSPACE;
  if (!aligned(startend_row_indices, 4) || !aligned(block_minmax, 4)) return FM_ERR_ALIGNMENT;
  fm_status st = device_info(nullptr);
  if (st != FM_OK) return st;
  return from_cuda(fm::launch_mask_minmax(startend_row_indices, n_mask_heads, total_tokens,
                                          cu_seqlens, n_seqs, block_n, block_minmax, n_slots,
                                          static_cast<cudaStream_t>(stream)));
}

size_t fm_attn_fwd_workspace_size(int64_t total_tokens, int n_seqs, int n_heads_q, int block_m) {
  if (total_tokens < 0 || n_seqs < 0 || n_heads_q < 1 || (block_m != 64 && block_m != 128))
    return 0;
  return fm::attn_workspace_bytes(total_tokens, n_seqs, block_m);
}

}  // extern "C"

namespace {

// Frequencies theta^(-2i/D) as double-float pairs (hi + lo).
void rope_freqs(double theta, int head_dim, fm::RopeFreqs* fr) {
  std::memset(fr, 0, sizeof(*fr));
  for (int i = 0; i < head_dim / 2; ++i) {
    const double f = std::pow(theta, -2.0 * i / head_dim);
    fr->hi[i] = static_cast<float>(f);
    fr->lo[i] = static_cast<float>(f - static_cast<double>(fr->hi[i]));
  }
}

// The scheduler's part of the forward parameters: samples, mask statistics,
// tile sizes and the workspace tables (shared by the attention calls and
// fm_attn_fwd_plan, so that a plan and the calls that reuse it agree).
void set_schedule_params(AttnParams& p, int64_t total_tokens, int n_heads_q, int n_heads_kv,
                         const int32_t* cu_seqlens, int n_seqs,
                         const int32_t* startend_row_indices, int n_mask_heads,
                         const int32_t* block_minmax, int causal, int block_m, int block_n,
                         void* workspace) {
  const int64_t n_qslots = total_tokens / block_m + n_seqs;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.cu = cu_seqlens;
  p.sri = startend_row_indices;
  p.minmax = block_minmax;
  p.ws = reinterpret_cast<fm::AttnWorkspaceHeader*>(ws);
  uint8_t* tail = ws + sizeof(fm::AttnWorkspaceHeader);
  p.slot_info = reinterpret_cast<int2*>(tail);
  p.order = reinterpret_cast<int2*>(tail + n_qslots * sizeof(int2));
  p.cost = reinterpret_cast<int*>(tail + 2 * n_qslots * sizeof(int2));
  p.T = total_tokens;
  p.n_qslots = n_qslots;
  p.n_kv_slots = fm_num_kv_tiles_bound(total_tokens, n_seqs, block_n);
  p.n_seqs = n_seqs;
  p.hq = n_heads_q;
  p.hkv = n_heads_kv;
  p.hm = n_mask_heads;
  p.block_m = block_m;
  p.block_n = block_n;
  p.causal = causal != 0;
  // Work items of two q heads that share a key/value head and the mask (one
  // Q tile each): both softmax warpgroups then see the same blocks, where two
  // consecutive Q tiles of one head differ in their last key tiles.
  p.head_pairs = n_mask_heads <= 1 && (n_heads_q / n_heads_kv) % 2 == 0;
}

// Validation shared by the attention forward calls and fm_attn_fwd_plan:
// samples, mask arguments (n_mask_heads is set to 0 without a mask), tile
// sizes and workspace.
fm_status check_schedule_args(int64_t total_tokens, int n_heads_q, int n_heads_kv,
                              const int32_t* cu_seqlens, int n_seqs,
                              const int32_t* startend_row_indices,
                              int& n_mask_heads, const int32_t* block_minmax, int block_m,
                              int block_n, const void* workspace, size_t workspace_bytes) {
  if (cu_seqlens == nullptr || workspace == nullptr) return FM_ERR_INVALID_ARG;
  if (total_tokens < 0 || total_tokens > INT32_MAX - 256 || n_seqs < 1) return FM_ERR_INVALID_ARG;
  if (n_heads_q < 1 || n_heads_kv < 1 || n_heads_q % n_heads_kv != 0) return FM_ERR_INVALID_ARG;
  if (startend_row_indices != nullptr) {
    if (n_mask_heads != 1 && n_mask_heads != n_heads_q) return FM_ERR_INVALID_ARG;
    if (block_minmax == nullptr) return FM_ERR_INVALID_ARG;
  } else {
    if (block_minmax != nullptr) return FM_ERR_INVALID_ARG;
    n_mask_heads = 0;
  }
  if ((block_m != 64 && block_m != 128) || (block_n != 64 && block_n != 128))
    return FM_ERR_UNSUPPORTED;
  if (!aligned(workspace, 256)) return FM_ERR_ALIGNMENT;
  if (workspace_bytes < fm::attn_workspace_bytes(total_tokens, n_seqs, block_m))
    return FM_ERR_WORKSPACE;
  const int64_t n_qslots = total_tokens / block_m + n_seqs;
  if (n_qslots * n_heads_q >= (int64_t(1) << 31)) return FM_ERR_UNSUPPORTED;
  return FM_OK;
}

// fm_attn_fwd_varlen and fm_attn_fwd_varlen_rope: validation, tensor maps,
// parameters and launches.  With `theta` > 0 the keys are rotated in place
// first and every Q tile is rotated in shared memory after its load.
fm_status attn_fwd_impl(const void* q, void* k_rot_in_place, const void* k, const void* v,
                        int64_t total_tokens, int n_heads_q, int n_heads_kv, int head_dim,
                        const int32_t* cu_seqlens, int n_seqs,
                        const int32_t* startend_row_indices, int n_mask_heads,
                        const int32_t* block_minmax, int causal, float softmax_scale,
                        int block_m, int block_n, double theta, void* out, float* lse,
                        void* q_rot, int64_t* block_class_counts, void* workspace,
                        size_t workspace_bytes, uint32_t flags, void* stream) {
  const bool fused_rope = theta != 0.0;
  if (fused_rope && (!(theta > 0.0) || !std::isfinite(theta))) return FM_ERR_INVALID_ARG;
  if (fused_rope && (k_rot_in_place == nullptr || k_rot_in_place != k)) return FM_ERR_INVALID_ARG;
  if (!fused_rope && q_rot != nullptr) return FM_ERR_INVALID_ARG;
  if (q_rot != nullptr && !aligned(q_rot, 16)) return FM_ERR_ALIGNMENT;
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || lse == nullptr)
    return FM_ERR_INVALID_ARG;
  if (flags & ~(FM_FLAG_FORCE_INT64 | FM_FLAG_REUSE_PLAN)) return FM_ERR_INVALID_ARG;
  fm_status st = check_schedule_args(total_tokens, n_heads_q, n_heads_kv, cu_seqlens, n_seqs,
                                     startend_row_indices, n_mask_heads, block_minmax, block_m,
                                     block_n, workspace, workspace_bytes);
  if (st != FM_OK) return st;
  if (!(softmax_scale >= 0.0f) || !std::isfinite(softmax_scale)) return FM_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return FM_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lse, 4))
    return FM_ERR_ALIGNMENT;
  if (block_class_counts != nullptr && !aligned(block_class_counts, 8)) return FM_ERR_ALIGNMENT;
  if (total_tokens == 0) return FM_OK;
  int num_sms = 0;
  st = device_info(&num_sms);
  if (st != FM_OK) return st;

  CUtensorMap tq, tk, tv;
  const uint64_t T = static_cast<uint64_t>(total_tokens);
  if (!make_map(&tq, q, static_cast<uint64_t>(n_heads_q) * head_dim, T, 128) ||
      !make_map(&tk, k, static_cast<uint64_t>(n_heads_kv) * head_dim, T, block_n) ||
      !make_map(&tv, v, static_cast<uint64_t>(n_heads_kv) * head_dim, T, block_n))
    return FM_ERR_CUDA;

  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  set_schedule_params(p, total_tokens, n_heads_q, n_heads_kv, cu_seqlens, n_seqs,
                      startend_row_indices, n_mask_heads, block_minmax, causal, block_m, block_n,
                      workspace);
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.lse = lse;
  p.class_counts = block_class_counts;
  p.head_dim = head_dim;
  p.reuse_plan = (flags & FM_FLAG_REUSE_PLAN) != 0;
  const double scale = softmax_scale > 0.0f ? softmax_scale : 1.0 / std::sqrt(double(head_dim));
  p.scale_log2 = static_cast<float>(scale * 1.4426950408889634);
  p.timeout_ns = 1000000000ull;

  const int64_t lim = int64_t(1) << 31;
  const bool use64 =
      fm_attn_index_bits(total_tokens, n_heads_q, n_heads_kv, head_dim, flags) == 64;

  // (the planner initialises the workspace header itself: no memset; with
  // FM_FLAG_REUSE_PLAN the kernel checks the stored plan's sizes instead)
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!fused_rope) return from_cuda(fm::launch_attn_fwd(p, tq, tk, tv, use64, num_sms, s));

  fm::RopeArgs ra;
  rope_freqs(theta, head_dim, &ra.freqs);
  ra.q_rot = q_rot;
  // keys in place (the stand-alone RoPE kernel over the key heads only)
  const int64_t kstride = static_cast<int64_t>(n_heads_kv) * head_dim;
  const bool rope64 = use64 || total_tokens * (head_dim / 16) >= lim;
  cudaError_t e = fm::launch_rope(k_rot_in_place, nullptr, total_tokens, n_heads_kv, 0, head_dim,
                                  kstride, 0, cu_seqlens, n_seqs, ra.freqs, false, rope64,
                                  num_sms, s);
  if (e != cudaSuccess) return FM_ERR_CUDA;
  return from_cuda(fm::launch_attn_fwd(p, tq, tk, tv, use64, num_sms, s, &ra));
}

}  // namespace

extern "C" {

fm_status fm_attn_fwd_varlen(const void* q, const void* k, const void* v, int64_t total_tokens,
                             int n_heads_q, int n_heads_kv, int head_dim,
                             const int32_t* cu_seqlens, int n_seqs,
                             const int32_t* startend_row_indices, int n_mask_heads,
                             const int32_t* block_minmax, int causal, float softmax_scale,
                             int block_m, int block_n, void* out, float* lse,
                             int64_t* block_class_counts, void* workspace,
                             size_t workspace_bytes, uint32_t flags, void* stream) {
  return attn_fwd_impl(q, nullptr, k, v, total_tokens, n_heads_q, n_heads_kv, head_dim,
                       cu_seqlens, n_seqs, startend_row_indices, n_mask_heads, block_minmax,
                       causal, softmax_scale, block_m, block_n, 0.0, out, lse, nullptr,
                       block_class_counts, workspace, workspace_bytes, flags, stream);
}

fm_status fm_attn_fwd_varlen_rope(const void* q, void* k, const void* v, int64_t total_tokens,
                                  int n_heads_q, int n_heads_kv, int head_dim,
                                  const int32_t* cu_seqlens, int n_seqs, double theta,
                                  const int32_t* startend_row_indices, int n_mask_heads,
                                  const int32_t* block_minmax, int causal, float softmax_scale,
                                  int block_m, int block_n, void* out, float* lse, void* q_rot,
                                  int64_t* block_class_counts, void* workspace,
                                  size_t workspace_bytes, uint32_t flags, void* stream) {
  if (!(theta > 0.0) || !std::isfinite(theta) || k == nullptr) return FM_ERR_INVALID_ARG;
  return attn_fwd_impl(q, k, k, v, total_tokens, n_heads_q, n_heads_kv, head_dim, cu_seqlens,
                       n_seqs, startend_row_indices, n_mask_heads, block_minmax, causal,
                       softmax_scale, block_m, block_n, theta, out, lse, q_rot,
                       block_class_counts, workspace, workspace_bytes, flags, stream);
}

fm_status fm_attn_fwd_plan(int64_t total_tokens, int n_heads_q, int n_heads_kv,
                           const int32_t* cu_seqlens, int n_seqs,
                           const int32_t* startend_row_indices, int n_mask_heads,
                           const int32_t* block_minmax, int causal, int block_m, int block_n,
                           void* workspace, size_t workspace_bytes, void* stream) {
  fm_status st = check_schedule_args(total_tokens, n_heads_q, n_heads_kv, cu_seqlens, n_seqs,
                                     startend_row_indices, n_mask_heads, block_minmax, block_m,
                                     block_n, workspace, workspace_bytes);
  if (st != FM_OK) return st;
  if (total_tokens == 0) return FM_OK;
  int num_sms = 0;
  st = device_info(&num_sms);
  if (st != FM_OK) return st;
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  set_schedule_params(p, total_tokens, n_heads_q, n_heads_kv, cu_seqlens, n_seqs,
                      startend_row_indices, n_mask_heads, block_minmax, causal, block_m, block_n,
                      workspace);
  return from_cuda(fm::launch_attn_plan(p, static_cast<cudaStream_t>(stream)));
}

size_t fm_attn_bwd_workspace_size(int64_t total_tokens, int n_seqs, int n_heads_q) {
  if (total_tokens < 0 || n_seqs < 0 || n_heads_q < 1) return 0;
  return fm::attn_bwd_workspace_bytes(total_tokens, n_seqs, n_heads_q);
}

fm_status fm_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* out,
                             const void* dout, const float* lse, int64_t total_tokens,
                             int n_heads_q, int n_heads_kv, int head_dim,
                             const int32_t* cu_seqlens, int n_seqs,
                             const int32_t* startend_row_indices, int n_mask_heads,
                             const int32_t* block_minmax, int causal, float softmax_scale,
                             void* dq, void* dk, void* dv, void* workspace,
                             size_t workspace_bytes, uint32_t flags, void* stream) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || dout == nullptr ||
      lse == nullptr || dq == nullptr || dk == nullptr || dv == nullptr ||
      cu_seqlens == nullptr || workspace == nullptr)
    return FM_ERR_INVALID_ARG;
  if (total_tokens < 0 || total_tokens > INT32_MAX - 256 || n_seqs < 1) return FM_ERR_INVALID_ARG;
  if (n_heads_q < 1 || n_heads_kv < 1 || n_heads_q % n_heads_kv != 0) return FM_ERR_INVALID_ARG;
  if (flags & ~FM_FLAG_FORCE_INT64) return FM_ERR_INVALID_ARG;
  if (startend_row_indices != nullptr) {
    if (n_mask_heads != 1 && n_mask_heads != n_heads_q) return FM_ERR_INVALID_ARG;
    if (block_minmax == nullptr) return FM_ERR_INVALID_ARG;
  } else {
    if (block_minmax != nullptr) return FM_ERR_INVALID_ARG;
    n_mask_heads = 0;
  }
  if (!(softmax_scale >= 0.0f) || !std::isfinite(softmax_scale)) return FM_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return FM_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(workspace, 256))
    return FM_ERR_ALIGNMENT;
  if (workspace_bytes < fm::attn_bwd_workspace_bytes(total_tokens, n_seqs, n_heads_q))
    return FM_ERR_WORKSPACE;
  const int64_t n_slots = total_tokens / 128 + n_seqs;
  if (n_slots * n_heads_q >= (int64_t(1) << 31)) return FM_ERR_UNSUPPORTED;
  if (total_tokens == 0) return FM_OK;
  int num_sms = 0;
  fm_status st = device_info(&num_sms);
  if (st != FM_OK) return st;

  fm::BwdMaps m;
  const uint64_t T = static_cast<uint64_t>(total_tokens);
  const uint64_t qc = static_cast<uint64_t>(n_heads_q) * head_dim;
  const uint64_t kc = static_cast<uint64_t>(n_heads_kv) * head_dim;
  if (!make_map(&m.q128, q, qc, T, 128) || !make_map(&m.do128, dout, qc, T, 128) ||
      !make_map(&m.k128, k, kc, T, 128) || !make_map(&m.v128, v, kc, T, 128) ||
      !make_map(&m.q64, q, qc, T, 64) || !make_map(&m.do64, dout, qc, T, 64) ||
      !make_map(&m.k64, k, kc, T, 64) || !make_map(&m.v64, v, kc, T, 64))
    return FM_ERR_CUDA;

  fm::AttnBwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.dout = dout;
  p.lse = lse;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.cu = cu_seqlens;
  p.sri = startend_row_indices;
  p.minmax = block_minmax;
  fm::attn_bwd_bind_workspace(p, workspace, total_tokens, n_seqs, n_heads_q);
  p.T = total_tokens;
  p.n_res_slots = n_slots;
  p.n_kv_slots = fm_num_kv_tiles_bound(total_tokens, n_seqs, 128);
  p.n_seqs = n_seqs;
  p.hq = n_heads_q;
  p.hkv = n_heads_kv;
  p.hm = n_mask_heads;
  p.head_dim = head_dim;
  p.causal = causal != 0;
  const double scale = softmax_scale > 0.0f ? softmax_scale : 1.0 / std::sqrt(double(head_dim));
  p.scale = static_cast<float>(scale);
  p.scale_log2 = static_cast<float>(scale * 1.4426950408889634);
  p.timeout_ns = 1000000000ull;

  const bool use64 =
      fm_attn_index_bits(total_tokens, n_heads_q, n_heads_kv, head_dim, flags) == 64;

  // (the backward planners initialise the workspace header: no memset)
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return from_cuda(fm::launch_attn_bwd(p, m, use64, num_sms, s));
}

fm_status fm_attn_fwd_num_work_items(const void* workspace, int64_t* host_items, void* stream) {
  if (workspace == nullptr || host_items == nullptr) return FM_ERR_INVALID_ARG;
  const auto* hdr = static_cast<const fm::AttnWorkspaceHeader*>(workspace);
  int32_t n = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&n, &hdr->n_tile_items, sizeof(n), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FM_ERR_CUDA;
  *host_items = n;
  return FM_OK;
}

fm_status fm_get_device_error(const void* workspace, int32_t* host_err, void* stream) {
  if (host_err == nullptr) return FM_ERR_INVALID_ARG;
  if (workspace == nullptr) {
    // the allocation-free entry point's array on the current device
    fm_status st = FM_OK;
    workspace = fm::noalloc_scratch_address(&st);
    if (st != FM_OK) return st;
  }
  const auto* hdr = static_cast<const fm::AttnWorkspaceHeader*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_err, &hdr->error_word, sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FM_ERR_CUDA;
  return FM_OK;
}

fm_status fm_get_device_timeout_info(const void* workspace, int32_t* host_info, void* stream) {
  if (host_info == nullptr) return FM_ERR_INVALID_ARG;
  if (workspace == nullptr) {
    fm_status st = FM_OK;
    workspace = fm::noalloc_scratch_address(&st);
    if (st != FM_OK) return st;
  }
  const auto* hdr = static_cast<const fm::AttnWorkspaceHeader*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_info, hdr->diag, sizeof(hdr->diag), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FM_ERR_CUDA;
  return FM_OK;
}

fm_status fm_debug_bounded_wait(int32_t* device_status, uint64_t timeout_ns, void* stream) {
  if (device_status == nullptr || timeout_ns == 0 || timeout_ns > 1000000000ull)
    return FM_ERR_INVALID_ARG;
  fm_status st = device_info(nullptr);
  if (st != FM_OK) return st;
  return from_cuda(
      fm::launch_bounded_wait_probe(device_status, timeout_ns, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
