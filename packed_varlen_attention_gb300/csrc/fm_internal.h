// fm_internal.h -- launchers shared between the C ABI (fm_api.cu) and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/fm.h"

namespace fm {

// Launches `kernel` as a programmatic dependent launch: its CTAs may be
// scheduled while the previous kernel on `stream` finishes, so its launch
// latency and set-up overlap that kernel's tail.  Every kernel launched this
// way calls pdl_wait() before its first global-memory access, which keeps
// stream order for memory; kernels that call pdl_trigger() let the next one
// start early in turn.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kMaxHalfDim = 64;  // head_dim <= 128

// Inverse RoPE frequencies theta^(-2i/D) as double-float pairs (hi + lo).
struct RopeFreqs {
  float hi[kMaxHalfDim];
  float lo[kMaxHalfDim];
};

// Fused Q rotation of the attention forward pass: frequencies and the
// optional output of the rotated q ([T][Hq][D] bf16, may be q itself).
struct RopeArgs {
  RopeFreqs freqs;
  void* q_rot;
};

cudaError_t launch_rope(void* q, void* k, int64_t T, int hq, int hkv, int head_dim,
                        int64_t q_stride, int64_t k_stride, const int32_t* cu, int n_seqs,
                        const RopeFreqs& freqs, bool backward, bool use_int64, int num_sms,
                        cudaStream_t stream);

cudaError_t launch_mask_minmax(const int32_t* sri, int n_mask_heads, int64_t T,
                               const int32_t* cu, int n_seqs, int block_n, int32_t* out,
                               int64_t n_slots, cudaStream_t stream);

// Workspace header of the attention forward pass.
struct AttnWorkspaceHeader {
  uint32_t work_counter;  // next work item (atomic)
  int32_t n_qtiles;       // real Q tiles found by the planner
  int32_t n_items;        // work items: (pair of Q tiles) x Hq
  int32_t error_word;     // FM_DEVERR_* bits
  int32_t diag[4];        // first expired wait: set flag, barrier, parity, block << 8 | warp
  int32_t n_tile_items;   // n_qtiles * Hq
  uint32_t work_counter_kv;  // backward: next key/value work item (atomic)
  int32_t bwd_q_tiles;       // backward: real 128-row tiles (planner)
  int32_t bwd_kv_tiles;      // backward: the same count for the key/value pass
  // forward plan: the sizes it was made for (plan_n_seqs = 0: no valid plan),
  // one 16-byte group read with one load; plan_tiles = block_m | block_n << 12
  // | head_pairs << 24
  int32_t plan_T, plan_n_seqs, plan_hq, plan_tiles;
  uint32_t exit_counter;  // forward: CTAs done claiming (the last one resets the counters)
  int32_t pad[47];
};
static_assert(sizeof(AttnWorkspaceHeader) == 256, "header is 256 bytes");
static_assert(offsetof(AttnWorkspaceHeader, n_items) == 8 &&
                  offsetof(AttnWorkspaceHeader, error_word) == 12 &&
                  offsetof(AttnWorkspaceHeader, plan_T) % 16 == 0,
              "the attention kernel reads the header in 16-byte groups");

constexpr int kCostBins = 1024;  // scheduler histogram bins (cost = non-F KV tiles)

struct AttnParams {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;
  const int32_t* cu;
  const int32_t* sri;
  const int32_t* minmax;
  int64_t* class_counts;
  AttnWorkspaceHeader* ws;
  int* cost;         // [n_qslots]
  int2* slot_info;   // [n_qslots] (sample, q tile)
  int2* order;       // [n_qslots] work order (sample, q tile)
  int64_t T;
  int64_t n_qslots;
  int64_t n_kv_slots;
  int n_seqs;
  int hq, hkv, hm;
  int head_dim;
  int block_m, block_n;
  int causal;
  int reuse_plan;  // skip the planner: the workspace holds the work order already
  int head_pairs;  // a work item is one Q tile for two q heads of one key/value head
  float scale_log2;
  uint64_t timeout_ns;
};

size_t attn_workspace_bytes(int64_t T, int n_seqs, int block_m);

// Device address of the allocation-free entry point's scheduler array on the
// current device (resolved once per device); nullptr with *st set on failure.
void* noalloc_scratch_address(fm_status* st);

// rope == nullptr: q is already rotated; otherwise every Q tile is rotated
// in shared memory after its load (positions restart at each sample start).
cudaError_t launch_attn_fwd(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, bool use_int64, int num_sms,
                            cudaStream_t stream, const RopeArgs* rope = nullptr);

// The forward scheduler alone (the planner kernels of launch_attn_fwd).
cudaError_t launch_attn_plan(const AttnParams& p, cudaStream_t stream);

cudaError_t launch_bounded_wait_probe(int32_t* status, uint64_t timeout_ns, cudaStream_t stream);

// Attention backward: 128-row resident tiles, 64-row streamed tiles, block
// statistics of 128-column key tiles.
struct AttnBwdParams {
  const void* q;
  const void* k;
  const void* v;
  const void* out;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  const int32_t* cu;
  const int32_t* sri;
  const int32_t* minmax;
  AttnWorkspaceHeader* ws;
  int* order_q;   // [n_res_slots] tile slots in processing order (dQ pass)
  int* order_kv;  // the same for the key/value pass
  float* nlse2;   // [Hq][T]: -lse * log2(e), -inf for rows with no unmasked key
  float* ndelta;  // [Hq][T]: -(dout . out) per row
  int64_t T;
  int64_t n_res_slots;  // floor(T / 128) + n_seqs: 128-row tile slots
  int64_t n_kv_slots;   // slots of the block statistics (same formula)
  int n_seqs;
  int hq, hkv, hm;
  int head_dim;
  int causal;
  float scale;
  float scale_log2;
  uint64_t timeout_ns;
  int num_sms;  // CTAs of the persistent passes (the planner's balance test)
};

// Tensor maps of the backward pass: 128-row and 64-row boxes of q, k, v, dout.
struct BwdMaps {
  CUtensorMap q128, do128, k128, v128;
  CUtensorMap q64, do64, k64, v64;
};

size_t attn_bwd_workspace_bytes(int64_t T, int n_seqs, int n_heads_q);
size_t attn_bwd_clear_bytes();
void attn_bwd_bind_workspace(AttnBwdParams& p, void* workspace, int64_t T, int n_seqs,
                             int n_heads_q);

cudaError_t launch_attn_bwd(const AttnBwdParams& p, const BwdMaps& maps, bool use_int64,
                            int num_sms, cudaStream_t stream);

}  // namespace fm
