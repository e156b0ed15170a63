// attn_fwd_noalloc.cu -- fm_attn_fwd_varlen_noalloc: the attention forward
// pass for callers that cannot allocate device memory.
//
// Who needs it: a plugin or custom operator that is handed only its input and
// output buffers by a host framework (no allocator handle to ask for a
// workspace), code running under a framework's caching allocator that owns
// the whole device memory pool (a private cudaMalloc would take memory the
// pool believes is free), and latency-critical paths that must not call
// cudaMalloc (it may synchronise the device and has no latency bound).
//
// How: the scheduler scratch that fm_attn_fwd_varlen normally takes from the
// caller lives here in one file-scope __device__ array of kScratchBytes bytes.
// Every GPU that loads this library holds that array until the process exits.
// The array is shared by every call on a device and keeps the last call's
// contents; each call's planner first initialises the part that must start
// at zero (work counter, error word), exactly as with a caller workspace.
// Calls that overlap on the GPU (different streams without ordering) race
// on the array and give wrong results: order them on one stream.  The array
// starts with the same header as a caller workspace, so fm_get_device_error
// and fm_get_device_timeout_info read its error word when given NULL.
#include <mutex>

#include "fm_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// Up to 32768 Q-tile slots (floor(T / block_m) + n_seqs), e.g. 4M tokens at
// block_m = 128: 256-byte header, 20 bytes per slot.
constexpr int64_t kMaxQSlots = 32768;
constexpr size_t kScratchBytes = sizeof(fm::AttnWorkspaceHeader) + kMaxQSlots * 20;
static_assert(kScratchBytes % 256 == 0, "scratch size is a multiple of 256 bytes");

}  // namespace

static __device__ __align__(256) uint8_t g_attn_scratch[kScratchBytes];

namespace fm {

// Device address of g_attn_scratch, resolved once per device.
void* noalloc_scratch_address(fm_status* st) {
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    *st = FM_ERR_CUDA;
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    *st = FM_ERR_UNSUPPORTED;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || p == nullptr) {
      *st = FM_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  *st = FM_OK;
  return addr[dev];
}

}  // namespace fm

extern "C" fm_status fm_attn_fwd_varlen_noalloc(
    const void* q, const void* k, const void* v, int64_t total_tokens, int n_heads_q,
    int n_heads_kv, int head_dim, const int32_t* cu_seqlens, int n_seqs,
    const int32_t* startend_row_indices, int n_mask_heads, const int32_t* block_minmax,
    int causal, float softmax_scale, int block_m, int block_n, void* out, float* lse,
    int64_t* block_class_counts, uint32_t flags, void* stream) {
  // the shared array holds whichever call ran last: no plan is reused here
  if (flags & FM_FLAG_REUSE_PLAN) return FM_ERR_INVALID_ARG;
  if (total_tokens < 0 || n_seqs < 1 || (block_m != 64 && block_m != 128))
    return total_tokens < 0 || n_seqs < 1 ? FM_ERR_INVALID_ARG : FM_ERR_UNSUPPORTED;
  if (total_tokens / block_m + n_seqs > kMaxQSlots) return FM_ERR_WORKSPACE;
  if (fm::attn_workspace_bytes(total_tokens, n_seqs, block_m) > kScratchBytes)
    return FM_ERR_WORKSPACE;
  fm_status st = FM_OK;
  void* scratch = fm::noalloc_scratch_address(&st);
  if (st != FM_OK) return st;
  return fm_attn_fwd_varlen(q, k, v, total_tokens, n_heads_q, n_heads_kv, head_dim, cu_seqlens,
                            n_seqs, startend_row_indices, n_mask_heads, block_minmax, causal,
                            softmax_scale, block_m, block_n, out, lse, block_class_counts,
                            scratch, kScratchBytes, flags, stream);
}
