"""Python binding of libfm (packed variable-length FlashMask attention, GB300).

Argument marshalling only: every step runs in the CUDA kernels of
``libfm.so`` (built in place by ``packed_varlen_attention_gb300.build``).
PyTorch supplies device memory and the current stream.  There is no CPU
fallback: if the library is missing or the device is not sm_103, every call
raises.

Entry points (same names as the C ABI in ``include/fm.h``):

* ``rope_qk_varlen``       fused in-place QK RoPE, positions reset per sample
* ``mask_block_minmax``    FlashMask per-key-tile min/max of LTS/LTE/UTS/UTE
* ``attn_fwd_varlen``      FlashMask attention forward (out, lse)
* ``attn_fwd_varlen_rope``  the same with the QK RoPE fused into its prologue
* ``attn_fwd_plan``        the forward's scheduler alone (a plan that the layers
                           of one packed batch reuse with ``reuse_plan=True``)
* ``attn_bwd_varlen``      FlashMask attention backward (dq, dk, dv)
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

__all__ = [
    "FMError",
    "rope_qk_varlen",
    "num_kv_tiles_bound",
    "rope_index_bits",
    "attn_index_bits",
    "mask_block_minmax",
    "attn_fwd_workspace_size",
    "attn_fwd_varlen",
    "attn_fwd_varlen_noalloc",
    "attn_fwd_varlen_rope",
    "attn_fwd_num_work_items",
    "attn_bwd_workspace_size",
    "attn_bwd_varlen",
    "attn_fwd_plan",
    "get_device_error",
    "get_device_timeout_info",
    "debug_bounded_wait",
    "status_string",
    "version",
    "library_path",
    "EXPORTED_SYMBOLS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libfm.so")
_LIB = None

FM_FLAG_FORCE_INT64 = 0x1
FM_FLAG_REUSE_PLAN = 0x2
FM_DEVERR_TIMEOUT = 0x1
FM_DEVERR_DATA = 0x2

_c_i64 = ctypes.c_int64
_c_int = ctypes.c_int
_c_u32 = ctypes.c_uint32
_c_vp = ctypes.c_void_p

_SIGNATURES = {
    "fm_rope_qk_varlen": (_c_int, [_c_vp, _c_vp, _c_i64, _c_int, _c_int, _c_int, _c_i64, _c_i64,
                                   _c_vp, _c_int, ctypes.c_double, _c_int, _c_u32, _c_vp]),
    "fm_num_kv_tiles_bound": (_c_i64, [_c_i64, _c_int, _c_int]),
    "fm_rope_index_bits": (_c_int, [_c_i64, _c_int, _c_int, _c_i64, _c_i64, _c_u32]),
    "fm_attn_index_bits": (_c_int, [_c_i64, _c_int, _c_int, _c_int, _c_u32]),
    "fm_mask_block_minmax": (_c_int, [_c_vp, _c_int, _c_i64, _c_vp, _c_int, _c_int, _c_vp,
                                      _c_i64, _c_vp]),
    "fm_attn_fwd_workspace_size": (ctypes.c_size_t, [_c_i64, _c_int, _c_int, _c_int]),
    "fm_attn_fwd_varlen": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_int, _c_int, _c_int, _c_vp,
                                    _c_int, _c_vp, _c_int, _c_vp, _c_int, ctypes.c_float, _c_int,
                                    _c_int, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_size_t, _c_u32,
                                    _c_vp]),
    "fm_attn_fwd_plan": (_c_int, [_c_i64, _c_int, _c_int, _c_vp, _c_int, _c_vp, _c_int, _c_vp,
                                  _c_int, _c_int, _c_int, _c_vp, ctypes.c_size_t, _c_vp]),
    "fm_attn_fwd_varlen_noalloc": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_int, _c_int, _c_int,
                                            _c_vp, _c_int, _c_vp, _c_int, _c_vp, _c_int,
                                            ctypes.c_float, _c_int, _c_int, _c_vp, _c_vp, _c_vp,
                                            _c_u32, _c_vp]),
    "fm_attn_fwd_varlen_rope": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_int, _c_int, _c_int,
                                         _c_vp, _c_int, ctypes.c_double, _c_vp, _c_int, _c_vp,
                                         _c_int, ctypes.c_float, _c_int, _c_int, _c_vp, _c_vp,
                                         _c_vp, _c_vp, _c_vp, ctypes.c_size_t, _c_u32, _c_vp]),
    "fm_attn_fwd_num_work_items": (_c_int, [_c_vp, ctypes.POINTER(_c_i64), _c_vp]),
    "fm_attn_bwd_workspace_size": (ctypes.c_size_t, [_c_i64, _c_int, _c_int]),
    "fm_attn_bwd_varlen": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_int,
                                    _c_int, _c_int, _c_vp, _c_int, _c_vp, _c_int, _c_vp, _c_int,
                                    ctypes.c_float, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_size_t,
                                    _c_u32, _c_vp]),
    "fm_get_device_error": (_c_int, [_c_vp, ctypes.POINTER(ctypes.c_int32), _c_vp]),
    "fm_get_device_timeout_info": (_c_int, [_c_vp, ctypes.POINTER(ctypes.c_int32), _c_vp]),
    "fm_debug_bounded_wait": (_c_int, [_c_vp, ctypes.c_uint64, _c_vp]),
    "fm_status_string": (ctypes.c_char_p, [_c_int]),
    "fm_version": (_c_int, []),
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)


class FMError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                "libfm.so is not built; run `python -m packed_varlen_attention_gb300.build`")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def status_string(code: int) -> str:
    return _lib().fm_status_string(int(code)).decode()


def version() -> int:
    return int(_lib().fm_version())


def _check(fn: str, code: int):
    if code != 0:
        raise FMError(fn, code)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _flags(force_int64: bool, reuse_plan: bool = False) -> int:
    return (FM_FLAG_FORCE_INT64 if force_int64 else 0) | (FM_FLAG_REUSE_PLAN if reuse_plan else 0)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def rope_qk_varlen(q: torch.Tensor, k: Optional[torch.Tensor], cu_seqlens: torch.Tensor,
                   theta: float, backward: bool = False, force_int64: bool = False,
                   stream=None) -> None:
    """Rotate q [T, Hq, D] and k [T, Hkv, D] (bf16, CUDA) in place."""
    _need(q, "q", torch.bfloat16)
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    T, hq, d = q.shape
    if q.stride(2) != 1 or q.stride(1) != d:
        raise ValueError("q must have contiguous heads ([T, H, D] with stride (s, D, 1))")
    hkv, ks = 0, 0
    if k is not None:
        _need(k, "k", torch.bfloat16)
        if k.shape[0] != T or k.shape[2] != d or k.stride(2) != 1 or k.stride(1) != d:
            raise ValueError("k must be [T, Hkv, D] with contiguous heads")
        hkv, ks = k.shape[1], k.stride(0)
    _check("fm_rope_qk_varlen", _lib().fm_rope_qk_varlen(
        _ptr(q), _ptr(k), T, hq, hkv, d, q.stride(0), ks, _ptr(cu_seqlens),
        cu_seqlens.numel() - 1, float(theta), int(bool(backward)),
        FM_FLAG_FORCE_INT64 if force_int64 else 0, _stream(stream)))


def rope_index_bits(total_tokens: int, n_heads_kv: int, head_dim: int, q_token_stride: int,
                    k_token_stride: int, force_int64: bool = False) -> int:
    """Index width (32 or 64) rope_qk_varlen uses for these sizes."""
    return int(_lib().fm_rope_index_bits(total_tokens, n_heads_kv, head_dim, q_token_stride,
                                         k_token_stride, FM_FLAG_FORCE_INT64 if force_int64 else 0))


def attn_index_bits(total_tokens: int, n_heads_q: int, n_heads_kv: int, head_dim: int,
                    force_int64: bool = False) -> int:
    """Index width (32 or 64) the attention calls use for these sizes."""
    return int(_lib().fm_attn_index_bits(total_tokens, n_heads_q, n_heads_kv, head_dim,
                                         FM_FLAG_FORCE_INT64 if force_int64 else 0))


def num_kv_tiles_bound(total_tokens: int, n_seqs: int, block_n: int) -> int:
    return int(_lib().fm_num_kv_tiles_bound(total_tokens, n_seqs, block_n))


def mask_block_minmax(startend_row_indices: torch.Tensor, cu_seqlens: torch.Tensor,
                      block_n: int, out: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
    """Per-key-tile statistics int32 [Hm, 8, n_slots] of the column intervals."""
    _need(startend_row_indices, "startend_row_indices", torch.int32)
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    sri = startend_row_indices
    if sri.dim() != 3 or sri.shape[1] != 4 or not sri.is_contiguous():
        raise ValueError("startend_row_indices must be contiguous int32 [Hm, 4, T]")
    hm, _, T = sri.shape
    n_seqs = cu_seqlens.numel() - 1
    n_slots = num_kv_tiles_bound(T, n_seqs, block_n)
    if out is None:
        out = torch.empty((hm, 8, n_slots), dtype=torch.int32, device=sri.device)
    _need(out, "out", torch.int32)
    _check("fm_mask_block_minmax", _lib().fm_mask_block_minmax(
        _ptr(sri), hm, T, _ptr(cu_seqlens), n_seqs, block_n, _ptr(out), out.numel(),
        _stream(stream)))
    return out


def attn_fwd_workspace_size(total_tokens: int, n_seqs: int, n_heads_q: int, block_m: int) -> int:
    return int(_lib().fm_attn_fwd_workspace_size(total_tokens, n_seqs, n_heads_q, block_m))


def attn_fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
                    startend_row_indices: Optional[torch.Tensor] = None,
                    block_minmax: Optional[torch.Tensor] = None, causal: bool = False,
                    softmax_scale: float = 0.0, block_m: int = 128, block_n: int = 128,
                    out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                    class_counts: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None, force_int64: bool = False,
                    reuse_plan: bool = False,
                    stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """FlashMask attention forward. Returns (out [T, Hq, D] bf16, lse [Hq, T] fp32).

    ``reuse_plan``: launch the attention kernel alone, on the work order that
    ``attn_fwd_plan`` (or an earlier call without the flag) left in
    ``workspace`` for the same ``cu_seqlens`` and sizes.
    """
    if reuse_plan and workspace is None:
        raise ValueError("reuse_plan needs the workspace that holds the plan")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous [T, H, D]")
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    T, hq, d = q.shape
    hkv = k.shape[1]
    n_seqs = cu_seqlens.numel() - 1
    hm = 0
    if startend_row_indices is not None:
        _need(startend_row_indices, "startend_row_indices", torch.int32)
        hm = startend_row_indices.shape[0]
        if block_minmax is None:
            raise ValueError("block_minmax (from mask_block_minmax) is required with a mask")
        _need(block_minmax, "block_minmax", torch.int32)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((hq, T), dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes = attn_fwd_workspace_size(T, n_seqs, hq, block_m)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if class_counts is not None:
        _need(class_counts, "class_counts", torch.int64)
    _check("fm_attn_fwd_varlen", _lib().fm_attn_fwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), T, hq, hkv, d, _ptr(cu_seqlens), n_seqs,
        _ptr(startend_row_indices), hm, _ptr(block_minmax), int(bool(causal)),
        float(softmax_scale), block_m, block_n, _ptr(out), _ptr(lse), _ptr(class_counts),
        _ptr(workspace), workspace.numel(), _flags(force_int64, reuse_plan),
        _stream(stream)))
    return out, lse


def attn_fwd_plan(cu_seqlens: torch.Tensor, total_tokens: int, n_heads_q: int, n_heads_kv: int,
                  startend_row_indices: Optional[torch.Tensor] = None,
                  block_minmax: Optional[torch.Tensor] = None, causal: bool = False,
                  block_m: int = 128, block_n: int = 128,
                  workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The forward scheduler alone: writes the work order for these samples
    into ``workspace`` (allocated when None) and returns it, for attention
    calls given ``reuse_plan=True``."""
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    n_seqs = cu_seqlens.numel() - 1
    hm = 0
    if startend_row_indices is not None:
        _need(startend_row_indices, "startend_row_indices", torch.int32)
        hm = startend_row_indices.shape[0]
        if block_minmax is None:
            raise ValueError("block_minmax (from mask_block_minmax) is required with a mask")
        _need(block_minmax, "block_minmax", torch.int32)
    if workspace is None:
        nbytes = attn_fwd_workspace_size(total_tokens, n_seqs, n_heads_q, block_m)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=cu_seqlens.device)
    _check("fm_attn_fwd_plan", _lib().fm_attn_fwd_plan(
        total_tokens, n_heads_q, n_heads_kv, _ptr(cu_seqlens), n_seqs,
        _ptr(startend_row_indices), hm,
        _ptr(block_minmax), int(bool(causal)), block_m, block_n, _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return workspace


def attn_fwd_varlen_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                            cu_seqlens: torch.Tensor,
                            startend_row_indices: Optional[torch.Tensor] = None,
                            block_minmax: Optional[torch.Tensor] = None, causal: bool = False,
                            softmax_scale: float = 0.0, block_m: int = 128, block_n: int = 128,
                            out: Optional[torch.Tensor] = None,
                            lse: Optional[torch.Tensor] = None,
                            class_counts: Optional[torch.Tensor] = None,
                            force_int64: bool = False,
                            stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """``attn_fwd_varlen`` for callers that cannot allocate device memory.

    The library keeps the scheduler scratch in a fixed device array of its own
    (limit: T // block_m + n_seqs <= 32768), so no workspace is passed.  Pass
    ``out`` and ``lse`` as well to keep this call free of allocations; the
    first call on a device should come before any stream capture, and calls
    must not overlap on the GPU (they share the array).
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous [T, H, D]")
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    T, hq, d = q.shape
    hm = 0
    if startend_row_indices is not None:
        _need(startend_row_indices, "startend_row_indices", torch.int32)
        hm = startend_row_indices.shape[0]
        if block_minmax is None:
            raise ValueError("block_minmax (from mask_block_minmax) is required with a mask")
        _need(block_minmax, "block_minmax", torch.int32)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((hq, T), dtype=torch.float32, device=q.device)
    if class_counts is not None:
        _need(class_counts, "class_counts", torch.int64)
    _check("fm_attn_fwd_varlen_noalloc", _lib().fm_attn_fwd_varlen_noalloc(
        _ptr(q), _ptr(k), _ptr(v), T, hq, k.shape[1], d, _ptr(cu_seqlens),
        cu_seqlens.numel() - 1, _ptr(startend_row_indices), hm, _ptr(block_minmax),
        int(bool(causal)), float(softmax_scale), block_m, block_n, _ptr(out), _ptr(lse),
        _ptr(class_counts), FM_FLAG_FORCE_INT64 if force_int64 else 0, _stream(stream)))
    return out, lse


def attn_fwd_varlen_rope(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                         cu_seqlens: torch.Tensor, theta: float,
                         startend_row_indices: Optional[torch.Tensor] = None,
                         block_minmax: Optional[torch.Tensor] = None, causal: bool = False,
                         softmax_scale: float = 0.0, block_m: int = 128, block_n: int = 128,
                         out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                         q_rot: Optional[torch.Tensor] = None,
                         class_counts: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None, force_int64: bool = False,
                         reuse_plan: bool = False,
                         stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Attention forward with the QK RoPE fused into its prologue.

    ``q`` and ``k`` are NOT rotated on entry.  ``k`` is rotated in place;
    ``q`` is rotated tile by tile in shared memory and left unchanged, unless
    ``q_rot`` (written with the rotated queries) is ``q`` itself.  Returns
    (out, lse), bit-identical to ``rope_qk_varlen`` followed by
    ``attn_fwd_varlen``.  ``reuse_plan`` as in ``attn_fwd_varlen``.
    """
    if reuse_plan and workspace is None:
        raise ValueError("reuse_plan needs the workspace that holds the plan")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous [T, H, D]")
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    T, hq, d = q.shape
    n_seqs = cu_seqlens.numel() - 1
    hm = 0
    if startend_row_indices is not None:
        _need(startend_row_indices, "startend_row_indices", torch.int32)
        hm = startend_row_indices.shape[0]
        if block_minmax is None:
            raise ValueError("block_minmax (from mask_block_minmax) is required with a mask")
        _need(block_minmax, "block_minmax", torch.int32)
    if q_rot is not None:
        _need(q_rot, "q_rot", torch.bfloat16)
        if q_rot.shape != q.shape or not q_rot.is_contiguous():
            raise ValueError("q_rot must be a contiguous tensor shaped like q")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((hq, T), dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes = attn_fwd_workspace_size(T, n_seqs, hq, block_m)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if class_counts is not None:
        _need(class_counts, "class_counts", torch.int64)
    _check("fm_attn_fwd_varlen_rope", _lib().fm_attn_fwd_varlen_rope(
        _ptr(q), _ptr(k), _ptr(v), T, hq, k.shape[1], d, _ptr(cu_seqlens), n_seqs,
        float(theta), _ptr(startend_row_indices), hm, _ptr(block_minmax), int(bool(causal)),
        float(softmax_scale), block_m, block_n, _ptr(out), _ptr(lse), _ptr(q_rot),
        _ptr(class_counts), _ptr(workspace), workspace.numel(),
        _flags(force_int64, reuse_plan), _stream(stream)))
    return out, lse


def attn_bwd_workspace_size(total_tokens: int, n_seqs: int, n_heads_q: int) -> int:
    return int(_lib().fm_attn_bwd_workspace_size(total_tokens, n_seqs, n_heads_q))


def attn_bwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
                    dout: torch.Tensor, lse: torch.Tensor, cu_seqlens: torch.Tensor,
                    startend_row_indices: Optional[torch.Tensor] = None,
                    block_minmax: Optional[torch.Tensor] = None, causal: bool = False,
                    softmax_scale: float = 0.0, dq: Optional[torch.Tensor] = None,
                    dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None, force_int64: bool = False,
                    stream=None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """FlashMask attention backward. Returns (dq, dk, dv), bf16, shaped like q, k, v.

    ``block_minmax`` must come from ``mask_block_minmax(..., block_n=128)``.
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, n, torch.bfloat16)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous [T, H, D]")
    _need(lse, "lse", torch.float32)
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    T, hq, d = q.shape
    hkv = k.shape[1]
    n_seqs = cu_seqlens.numel() - 1
    hm = 0
    if startend_row_indices is not None:
        _need(startend_row_indices, "startend_row_indices", torch.int32)
        hm = startend_row_indices.shape[0]
        if block_minmax is None:
            raise ValueError("block_minmax (from mask_block_minmax, block_n=128) is required")
        _need(block_minmax, "block_minmax", torch.int32)
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    if workspace is None:
        workspace = torch.empty(attn_bwd_workspace_size(T, n_seqs, hq), dtype=torch.uint8,
                                device=q.device)
    _check("fm_attn_bwd_varlen", _lib().fm_attn_bwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), T, hq, hkv, d,
        _ptr(cu_seqlens), n_seqs, _ptr(startend_row_indices), hm, _ptr(block_minmax),
        int(bool(causal)), float(softmax_scale), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
        workspace.numel(), FM_FLAG_FORCE_INT64 if force_int64 else 0, _stream(stream)))
    return dq, dk, dv


def attn_fwd_num_work_items(workspace: torch.Tensor, stream=None) -> int:
    n = _c_i64(0)
    _check("fm_attn_fwd_num_work_items",
           _lib().fm_attn_fwd_num_work_items(_ptr(workspace), ctypes.byref(n), _stream(stream)))
    return int(n.value)


def get_device_error(workspace: Optional[torch.Tensor], stream=None) -> int:
    """Device error word (FM_DEVERR_* bits) of the last call that used
    ``workspace``; ``None``: the last ``attn_fwd_varlen_noalloc`` call on the
    current device."""
    e = ctypes.c_int32(0)
    _check("fm_get_device_error",
           _lib().fm_get_device_error(_ptr(workspace), ctypes.byref(e), _stream(stream)))
    return int(e.value)


def get_device_timeout_info(workspace: Optional[torch.Tensor], stream=None):
    """(expired, barrier, parity, block, warp) of the first wait that ran out
    (``workspace=None``: the last ``attn_fwd_varlen_noalloc`` call)."""
    info = (ctypes.c_int32 * 4)()
    _check("fm_get_device_timeout_info", _lib().fm_get_device_timeout_info(
        _ptr(workspace), info, _stream(stream)))
    return (int(info[0]), int(info[1]), int(info[2]), int(info[3]) >> 8, int(info[3]) & 0xFF)


def debug_bounded_wait(timeout_ns: int, stream=None) -> int:
    """Runs one bounded wait on a barrier nothing arrives at; returns its status."""
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _check("fm_debug_bounded_wait",
           _lib().fm_debug_bounded_wait(_ptr(status), int(timeout_ns), _stream(stream)))
    return int(status.item())
