/*
 * fm.h -- C ABI of libfm: packed variable-length FlashMask attention and
 * packed QK RoPE for NVIDIA GB300 (sm_103a).
 *
 * Every entry point takes plain pointers and sizes.  Device pointers are
 * CUDA device addresses of the current device; host pointers are marked.
 * The caller owns every buffer (inputs, outputs, workspace) and the stream;
 * the library never allocates device memory, never synchronises the stream
 * (except fm_get_device_error, which reads one word back) and keeps no
 * state beyond cached device attributes and resolved driver entry points.
 * `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 * stream.  All kernels are enqueued on `stream` in call order, as
 * programmatic dependent launches: a kernel may begin its set-up while the
 * previous kernel on the stream finishes, and touches no global memory
 * before that kernel has completed, so stream order holds for every buffer.
 * The calls may be captured in a CUDA graph; make the first call on a device
 * outside capture (it caches device attributes and sets kernel attributes).
 *
 * Packed layout (Unsloth packing blog, section "Why padding is needed";
 * Varlen-Packing technical document, section 1.1): documents are
 * concatenated along the token axis with no padding, T tokens in all;
 * cu_seqlens is int32[n_seqs + 1] on the device with cu[0] = 0,
 * cu[n_seqs] = T and cu non-decreasing.  Sample s owns tokens
 * [cu[s], cu[s+1]).  Malformed cu_seqlens never makes a kernel read or write
 * outside the buffers described here (indices are clamped), but the results
 * are then unspecified and fm_attn_fwd_varlen sets FM_DEVERR_DATA.
 *
 * Tensors are bfloat16, token-major: q[T][Hq][D], k and v[T][Hkv][D].
 *
 * Errors: every call validates its arguments on the host first and returns
 * before any launch when they are invalid; a failed launch returns
 * FM_ERR_CUDA.  Kernels never trap: conditions only the device can see are
 * written to a device error word (see fm_get_device_error).
 */
#ifndef FM_H_
#define FM_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FM_API __attribute__((visibility("default")))
#else
#define FM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fm_status {
  FM_OK = 0,
  FM_ERR_INVALID_ARG = 1,  /* null pointer, negative size, inconsistent sizes */
  FM_ERR_UNSUPPORTED = 2,  /* head_dim / tile shape / device not supported    */
  FM_ERR_ALIGNMENT = 3,    /* a pointer or stride breaks the 16-byte rule     */
  FM_ERR_WORKSPACE = 4,    /* output or workspace capacity too small          */
  FM_ERR_CUDA = 5,         /* a CUDA runtime / driver call failed             */
  FM_ERR_TIMEOUT = 6,      /* a bounded device wait ran out (see below)       */
  FM_ERR_DEVICE_DATA = 7   /* the device saw malformed cu_seqlens             */
} fm_status;

/* Bits of the device error word. */
#define FM_DEVERR_TIMEOUT 0x1u /* a pipeline wait exceeded its limit      */
#define FM_DEVERR_DATA 0x2u    /* malformed cu_seqlens seen on the device, or a
                                  reused plan made for other sizes          */

/* Flags. */
#define FM_FLAG_FORCE_INT64 0x1u /* use the 64-bit index specialisation */
#define FM_FLAG_REUSE_PLAN 0x2u  /* attention forward: use the work order already
                                    in the workspace (see fm_attn_fwd_plan) */

/*
 * fm_rope_qk_varlen -- rotary position embedding of q and k, in place, with
 * positions restarting at every packed sample.
 *
 * Unsloth packing blog, section "Fused QK RoPE Triton kernel with packing":
 * one launch rotates both q and k (no clones, no transposes), with
 * Y = X*cos + rotate_half(X)*sin, rotate_half(X) = X @ R, R = [[0, I], [-I, 0]];
 * the backward pass is the same rotation with sin -> -sin.  Section
 * "Uncontaminated packing": position ids reset per sample, so token t of
 * sample s has position p = t - cu[s].  Channel i pairs with channel
 * i + D/2; the angle of pair i is p * theta^(-2i/D).
 *
 *   q, k            device bf16, rotated in place.  Token t, head h of q is
 *                   at q + t*q_token_stride + h*head_dim (elements); heads
 *                   are contiguous.  q and k may be views into one fused
 *                   buffer as long as they do not overlap.
 *   total_tokens    T >= 0 (T = 0 is a no-op).
 *   n_heads_q/kv    >= 1 (n_heads_kv = 0 skips k, which may then be NULL).
 *   head_dim        64 or 128.
 *   *_token_stride  elements between consecutive tokens, >= heads*head_dim,
 *                   multiple of 8 (16 bytes).
 *   cu_seqlens      device int32[n_seqs + 1]; n_seqs >= 1.  A sample may be
 *                   at most 2^24 tokens long (positions are exact in fp32).
 *   theta           RoPE base, > 0.
 *   backward        0: forward rotation, 1: inverse rotation (sin -> -sin).
 *   flags           FM_FLAG_FORCE_INT64 or 0 (64-bit offsets are also chosen
 *                   automatically when an element offset reaches 2^31).
 *   q, k must be 16-byte aligned.
 */
FM_API fm_status fm_rope_qk_varlen(void* q, void* k, int64_t total_tokens, int n_heads_q,
                            int n_heads_kv, int head_dim, int64_t q_token_stride,
                            int64_t k_token_stride, const int32_t* cu_seqlens, int n_seqs,
                            double theta, int backward, uint32_t flags, void* stream);

/*
 * fm_rope_index_bits / fm_attn_index_bits -- the index width (32 or 64) that
 * fm_rope_qk_varlen / the attention calls (forward, fused-RoPE forward,
 * backward) choose for these sizes; -1 on negative sizes.
 *
 * Unsloth packing blog, section "Int64 indexing for Triton kernels": 32-bit
 * offsets overflow at long contexts, while always-64-bit indexing slows
 * training slightly, so the width is a compile-time specialisation chosen
 * per call.  Offsets are 32-bit unless an element offset can reach 2^31
 * (RoPE: T * token stride of q or k, or T * head_dim / 16 threads;
 * attention: T * Hq * D or T * Hkv * D), or FM_FLAG_FORCE_INT64 asks for
 * 64-bit; both widths give identical results.
 */
FM_API int fm_rope_index_bits(int64_t total_tokens, int n_heads_kv, int head_dim,
                              int64_t q_token_stride, int64_t k_token_stride, uint32_t flags);
FM_API int fm_attn_index_bits(int64_t total_tokens, int n_heads_q, int n_heads_kv, int head_dim,
                              uint32_t flags);

/*
 * fm_num_kv_tiles_bound -- number of per-tile slots used by the block
 * statistics layout below: floor(T / block_n) + n_seqs.
 *
 * Tiles are sample-local: tile j of sample s covers key columns
 * [cu[s] + j*block_n, min(cu[s] + (j+1)*block_n, cu[s+1])) and lives in slot
 * floor(cu[s] / block_n) + s + j.  Distinct tiles never share a slot and no
 * slot reaches the bound; slots that hold no tile are filled with
 * (INT32_MAX, INT32_MIN) pairs.  Returns -1 on invalid arguments.
 */
FM_API int64_t fm_num_kv_tiles_bound(int64_t total_tokens, int n_seqs, int block_n);

/*
 * fm_mask_block_minmax -- FlashMask preprocessing: the eight per-key-tile
 * extreme vectors.
 *
 * PaddleNLP FlashMask article, section 2.2: the mask is given column by
 * column as LTS/LTE (rows [LTS_j, LTE_j) masked on and below the diagonal)
 * and UTS/UTE (rows [UTS_j, UTE_j) masked above it), global row indices.
 * Section 3.1: split the columns by the attention kernel's key tile and take
 * the minimum and maximum of each vector over every tile.
 *
 *   startend_row_indices  device int32[n_mask_heads][4][T], vectors in the
 *                         order LTS, LTE, UTS, UTE.
 *   n_mask_heads          >= 1.
 *   block_n               key tile width, 64 or 128.
 *   block_minmax          device int32[n_mask_heads][8][n_slots] output,
 *                         n_slots = fm_num_kv_tiles_bound(T, n_seqs, block_n);
 *                         the eight rows are LTS min, LTS max, LTE min,
 *                         LTE max, UTS min, UTS max, UTE min, UTE max.
 *   block_minmax_capacity elements available at block_minmax; must be at
 *                         least n_mask_heads * 8 * n_slots.
 */
FM_API fm_status fm_mask_block_minmax(const int32_t* startend_row_indices, int n_mask_heads,
                               int64_t total_tokens, const int32_t* cu_seqlens, int n_seqs,
                               int block_n, int32_t* block_minmax,
                               int64_t block_minmax_capacity, void* stream);

/*
 * fm_attn_fwd_workspace_size -- bytes of device workspace that
 * fm_attn_fwd_varlen needs for these sizes (scheduler tables, counters and
 * the device error word).  Returns 0 on invalid arguments.
 */
FM_API size_t fm_attn_fwd_workspace_size(int64_t total_tokens, int n_seqs, int n_heads_q, int block_m);

/*
 * fm_attn_fwd_varlen -- FlashMask attention forward over packed samples.
 *
 * PaddleNLP FlashMask article, section 3: FlashAttention-2 tiling (Q tiles
 * of block_m rows, key/value tiles of block_n columns, online softmax, S and
 * P kept on chip) in which every (Q tile, KV tile) block is classified from
 * the eight statistics (section 3.2) as fully masked (skipped), partially
 * masked (element mask applied) or unmasked (no mask arithmetic); section
 * 3.3: the result equals attention under the dense mask.  For every sample
 * s, q head h and row i of s:
 *     o_i   = sum_j softmax_j(scale * q_i . k_j) v_j   over unmasked keys j of s
 *     lse_i = log sum_j exp(scale * q_i . k_j)         (natural log)
 * with key/value head h / (Hq / Hkv).  Element (i, j), i >= j (diagonal
 * included) is masked iff LTS_j <= i < LTE_j; element i < j is masked iff
 * causal or UTS_j <= i < UTE_j; keys of other samples are always masked.
 * A row with no unmasked key gets o = 0 and lse = -inf.  Section 3.4 names
 * softmax_lse as an input of the backward operator, hence the lse output.
 *
 * Scheduling (Varlen-Packing technical document, section 2, describes the
 * fixed grid (seq_count, n_head, ceil(max_seq_len / block_m)) that this call
 * does not use): work items are only the real Q tiles of every sample
 * (times Hq heads), ordered by the number of blocks they must compute and
 * pulled by a persistent grid of one CTA per SM.  A work item is one Q
 * tile for two q heads that share a key/value head and the mask (when
 * Hq / Hkv is even and n_mask_heads <= 1), else two consecutive Q tiles of
 * one q head; either way one CTA computes both with each K/V tile loaded
 * once.
 *
 *   q                 device bf16 [T][Hq][D], contiguous, 16-byte aligned.
 *   k, v              device bf16 [T][Hkv][D], contiguous, 16-byte aligned.
 *   n_heads_q         Hq >= 1;  n_heads_kv: Hkv >= 1 with Hq % Hkv == 0.
 *   head_dim          64 or 128.
 *   cu_seqlens        device int32[n_seqs + 1], n_seqs >= 1.
 *   startend_row_indices  device int32[n_mask_heads][4][T] (LTS, LTE, UTS,
 *                     UTE) or NULL for no interval mask (then n_mask_heads
 *                     is ignored and block_minmax must be NULL).
 *   n_mask_heads      1 (shared by every head) or Hq (mask head h for q head h).
 *   block_minmax      device output of fm_mask_block_minmax with the same
 *                     cu_seqlens, startend_row_indices and block_n.
 *   causal            nonzero: the whole upper triangle is masked.
 *   softmax_scale     > 0, or 0 for 1/sqrt(head_dim).
 *   block_m, block_n  Q / KV tile sizes, each 64 or 128.
 *   out               device bf16 [T][Hq][D], 16-byte aligned (written).
 *   lse               device float [Hq][T] (written).
 *   block_class_counts  optional device int64[3]; when not NULL, the counts
 *                     of fully masked, partially masked and unmasked blocks
 *                     over all (sample, Q tile, KV tile, q head) are ADDED
 *                     to it.
 *   workspace         device buffer of workspace_bytes >=
 *                     fm_attn_fwd_workspace_size(T, n_seqs, Hq, block_m),
 *                     256-byte aligned; its contents need no initialisation
 *                     and are overwritten.  Calls that share a workspace must
 *                     be ordered on one stream.
 *   flags             FM_FLAG_FORCE_INT64, FM_FLAG_REUSE_PLAN, both or 0.
 *                     Without FM_FLAG_REUSE_PLAN the call first runs the
 *                     scheduler (fm_attn_fwd_plan) into `workspace`; with it
 *                     the call launches the attention kernel alone, on the
 *                     work order already there (see fm_attn_fwd_plan).
 */
FM_API fm_status fm_attn_fwd_varlen(const void* q, const void* k, const void* v, int64_t total_tokens,
                             int n_heads_q, int n_heads_kv, int head_dim,
                             const int32_t* cu_seqlens, int n_seqs,
                             const int32_t* startend_row_indices, int n_mask_heads,
                             const int32_t* block_minmax, int causal, float softmax_scale,
                             int block_m, int block_n, void* out, float* lse,
                             int64_t* block_class_counts, void* workspace,
                             size_t workspace_bytes, uint32_t flags, void* stream);

/*
 * fm_attn_fwd_plan -- the scheduler of fm_attn_fwd_varlen alone: the work
 * items (the real Q tiles of every sample, times Hq) and their order, largest
 * first by the number of blocks that are not fully masked, written into
 * `workspace` together with the sizes they were made for.
 *
 * Varlen-Packing technical document, section 2: a fixed grid over
 * ceil(max_seq_len / block_m) tiles per sample leaves most of its blocks
 * empty on packed batches; this work list holds real tiles only.  The list
 * depends on cu_seqlens and the sizes, not on q, k or v, so the layers of a
 * model that share one packed batch can share one plan: plan once, then pass
 * FM_FLAG_REUSE_PLAN to every fm_attn_fwd_varlen / fm_attn_fwd_varlen_rope
 * call on this workspace (the calls need not repeat the scheduler's two
 * launches).  A call with the flag checks on the device that the plan was
 * made for the same total_tokens, n_seqs, n_heads_q, block_m, block_n and
 * work-item form (see fm_attn_fwd_varlen, Scheduling);
 * if not (or once fm_attn_bwd_varlen has used the workspace, or a call on
 * the plan has set a device error) it computes nothing and sets
 * FM_DEVERR_DATA.  It cannot check cu_seqlens itself: the plan must come
 * from the same cu_seqlens values.  The mask statistics only set the order
 * (the attention kernel classifies every block itself), so a plan stays
 * correct for other masks over the same samples.
 *
 * Arguments as fm_attn_fwd_varlen (same meaning and rules).  The device
 * error word and timeout record of `workspace` are cleared.
 */
FM_API fm_status fm_attn_fwd_plan(int64_t total_tokens, int n_heads_q, int n_heads_kv,
                                  const int32_t* cu_seqlens, int n_seqs,
                                  const int32_t* startend_row_indices, int n_mask_heads,
                                  const int32_t* block_minmax, int causal, int block_m,
                                  int block_n, void* workspace, size_t workspace_bytes,
                                  void* stream);

/*
 * fm_attn_fwd_varlen_noalloc -- fm_attn_fwd_varlen for callers that cannot
 * allocate device memory.  The pages have no counterpart: this entry point
 * exists for integration only.
 *
 * Same arguments and results as fm_attn_fwd_varlen, without workspace and
 * workspace_bytes.  Callers without an allocator handle (a plugin that only
 * receives its input and output buffers), callers whose device memory is
 * owned by a framework's caching allocator, and latency-critical paths that
 * must not call cudaMalloc (it may synchronise the device) can use it: the
 * scheduler scratch lives in a fixed array inside the library (a little
 * under 0.7 MB, held by every GPU that loads the library until the process
 * exits).  Limit: floor(T / block_m) + n_seqs <= 32768 Q-tile slots, else
 * FM_ERR_WORKSPACE is returned before any launch.  The first call on a
 * device resolves the array's device address (with that device current);
 * make that first call before any stream capture.  All calls on a device
 * share the array and each call clears what must start at zero; calls that
 * overlap on the GPU race on it, so order them on one stream.  Nothing is
 * allocated or freed.  The device error word and the timeout record of the
 * last call on the current device are read with fm_get_device_error /
 * fm_get_device_timeout_info given workspace == NULL.  Every call runs the
 * scheduler: FM_FLAG_REUSE_PLAN gives FM_ERR_INVALID_ARG.
 */
FM_API fm_status fm_attn_fwd_varlen_noalloc(const void* q, const void* k, const void* v,
                                            int64_t total_tokens, int n_heads_q, int n_heads_kv,
                                            int head_dim, const int32_t* cu_seqlens, int n_seqs,
                                            const int32_t* startend_row_indices,
                                            int n_mask_heads, const int32_t* block_minmax,
                                            int causal, float softmax_scale, int block_m,
                                            int block_n, void* out, float* lse,
                                            int64_t* block_class_counts, uint32_t flags,
                                            void* stream);

/*
 * fm_attn_fwd_varlen_rope -- fm_attn_fwd_varlen with the QK RoPE fused into
 * the attention prologue.
 *
 * Unsloth packing blog, section "Fused QK RoPE Triton kernel with packing":
 * the rotation Y = X*cos + rotate_half(X)*sin with positions restarting at
 * every sample start (section "Uncontaminated packing"), fused to save
 * memory traffic.  Here the queries are never rotated in HBM: every Q tile
 * is rotated in shared memory right after its load, before the QK^T MMAs
 * read it.  The keys are rotated in place first (one pass over k only),
 * because every key tile is read by many Q tiles and the backward pass needs
 * the rotated keys.  The result (out, lse, block counts) is bit-identical to
 * fm_rope_qk_varlen(q, k, ..., backward = 0) followed by fm_attn_fwd_varlen:
 * both use the same rotation arithmetic (frequencies theta^(-2i/D),
 * channel i paired with i + D/2, angle in extended precision).
 *
 * Arguments as fm_attn_fwd_varlen, plus:
 *   k        device bf16 [T][Hkv][D]: rotated IN PLACE (read and written).
 *   theta    RoPE base, > 0 and finite (e.g. 10000, 500000, 1e6).
 *   q        device bf16 [T][Hq][D], NOT rotated: left unchanged unless
 *            q_rot == q.
 *   q_rot    optional device bf16 [T][Hq][D], 16-byte aligned: when not NULL
 *            the rotated queries are written there (every token inside a
 *            sample, every head), as the backward pass needs them.  May be
 *            q itself (rotation in place).  NULL: nothing is written.
 * Errors: as fm_attn_fwd_varlen; theta <= 0, non-finite or k == NULL give
 * FM_ERR_INVALID_ARG, an unaligned q_rot FM_ERR_ALIGNMENT.
 */
FM_API fm_status fm_attn_fwd_varlen_rope(const void* q, void* k, const void* v,
                                         int64_t total_tokens, int n_heads_q, int n_heads_kv,
                                         int head_dim, const int32_t* cu_seqlens, int n_seqs,
                                         double theta, const int32_t* startend_row_indices,
                                         int n_mask_heads, const int32_t* block_minmax,
                                         int causal, float softmax_scale, int block_m,
                                         int block_n, void* out, float* lse, void* q_rot,
                                         int64_t* block_class_counts, void* workspace,
                                         size_t workspace_bytes, uint32_t flags, void* stream);

/*
 * fm_attn_bwd_workspace_size -- bytes of device workspace that
 * fm_attn_bwd_varlen needs for these sizes: counters and the device error
 * word, the scheduler's tables (floor(T / 128) + n_seqs tile slots) and two
 * float arrays of Hq * T.  Returns 0 on invalid arguments.
 */
FM_API size_t fm_attn_bwd_workspace_size(int64_t total_tokens, int n_seqs, int n_heads_q);

/*
 * fm_attn_bwd_varlen -- FlashMask attention backward over packed samples.
 *
 * PaddleNLP FlashMask article, section 3.4: the backward operator takes q,
 * k, v, the column intervals, out, softmax_lse and the gradient of out, and
 * returns the gradients of q, k and v; section 3.3: the block-skipping
 * kernel equals dense-mask attention, so these are the gradients of the
 * attention defined at fm_attn_fwd_varlen (same mask rules).  With
 * p_ij = exp(scale * q_i . k_j - lse_i) over unmasked pairs of a sample,
 * delta_i = dout_i . out_i and ds_ij = p_ij (dout_i . v_j - delta_i):
 *     dq_i = scale * sum_j ds_ij k_j
 *     dk_j = scale * sum over q heads of the group and rows i of ds_ij q_i
 *     dv_j = sum over q heads of the group and rows i of p_ij dout_i
 * Rows with lse = -inf (no unmasked key) contribute nothing.  Fully masked
 * blocks are skipped using the block statistics (section 3.2).  Every
 * gradient row is owned by one CTA (no atomics): results are bitwise
 * reproducible from run to run.
 *
 *   q, k, v, cu_seqlens, n_heads_q, n_heads_kv, head_dim,
 *   startend_row_indices, n_mask_heads, causal, softmax_scale: as for
 *                     fm_attn_fwd_varlen (the values of the forward call).
 *   out, lse          device outputs of that forward call: bf16 [T][Hq][D]
 *                     and float [Hq][T].
 *   dout              device bf16 [T][Hq][D], 16-byte aligned.
 *   block_minmax      device output of fm_mask_block_minmax with block_n =
 *                     128 (NULL when startend_row_indices is NULL).
 *   dq                device bf16 [T][Hq][D] (written).
 *   dk, dv            device bf16 [T][Hkv][D] (written).
 *   workspace         device buffer of workspace_bytes >=
 *                     fm_attn_bwd_workspace_size(T, n_seqs, Hq), 256-byte aligned; no
 *                     initialisation needed.  Calls that share a workspace
 *                     must be ordered on one stream.  fm_get_device_error
 *                     reads its error word.
 *   flags             FM_FLAG_FORCE_INT64 or 0.
 * Pointers to tensors must be 16-byte aligned, lse 4-byte aligned.
 */
FM_API fm_status fm_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* out,
                                    const void* dout, const float* lse, int64_t total_tokens,
                                    int n_heads_q, int n_heads_kv, int head_dim,
                                    const int32_t* cu_seqlens, int n_seqs,
                                    const int32_t* startend_row_indices, int n_mask_heads,
                                    const int32_t* block_minmax, int causal, float softmax_scale,
                                    void* dq, void* dk, void* dv, void* workspace,
                                    size_t workspace_bytes, uint32_t flags, void* stream);

/*
 * fm_attn_fwd_num_work_items -- after fm_attn_fwd_varlen has completed on
 * `stream`, copies to *host_items the number of work items its scheduler
 * built (real Q tiles times Hq).  Synchronises `stream`.
 */
FM_API fm_status fm_attn_fwd_num_work_items(const void* workspace, int64_t* host_items, void* stream);

/*
 * fm_get_device_error -- synchronises `stream` and copies the device error
 * word of the last fm_attn_fwd_varlen or fm_attn_bwd_varlen that used
 * `workspace` into *host_err (a bit set of FM_DEVERR_*; 0 when clean).
 * workspace == NULL reads the word of the last fm_attn_fwd_varlen_noalloc
 * call on the current device (its array inside the library).
 */
FM_API fm_status fm_get_device_error(const void* workspace, int32_t* host_err, void* stream);

/*
 * fm_get_device_timeout_info -- synchronises `stream` and copies four int32
 * describing the first pipeline wait that ran out in the last call that used
 * `workspace`: {1 if one did (else 0), barrier index, phase parity,
 * block << 8 | warp}.  Barrier indices are internal to each kernel; this is
 * a diagnostic for bug reports, not an interface to act on.  workspace ==
 * NULL: the last fm_attn_fwd_varlen_noalloc call on the current device.
 */
FM_API fm_status fm_get_device_timeout_info(const void* workspace, int32_t* host_info, void* stream);

/*
 * fm_debug_bounded_wait -- runs the pipeline's bounded mbarrier wait once on
 * a barrier that nothing ever arrives at, with a limit of timeout_ns, and
 * writes the resulting status (FM_ERR_TIMEOUT when the limit expired) to
 * device int32 *device_status.  Used to check the timeout path without
 * hanging a GPU.  timeout_ns must be in (0, 10^9].
 */
FM_API fm_status fm_debug_bounded_wait(int32_t* device_status, uint64_t timeout_ns, void* stream);

/* Human-readable name of a status code. */
FM_API const char* fm_status_string(int status);

/* Library ABI version (major * 100 + minor). */
FM_API int fm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FM_H_ */
