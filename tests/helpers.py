"""Shared test plumbing: building/loading the library, tensors from workloads,
tolerance checks.  Test code only (never imported by the product)."""

from __future__ import annotations

import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Tolerances stated for the hot path: attention output max-abs 1e-2 and
# mean-abs 1e-3, LSE 1e-3, RoPE max-abs 8e-3.  Where the oracle value is so
# large that one bfloat16 ulp of the stored output exceeds the max-abs bound,
# the bound is that ulp (the output format cannot do better).
ATTN_MAX_ABS = 1e-2
ATTN_MEAN_ABS = 1e-3
LSE_ABS = 1e-3
ROPE_MAX_ABS = 8e-3


def ensure_library():
    import packed_varlen_attention_gb300 as fm
    if not os.path.exists(fm.library_path()):
        from packed_varlen_attention_gb300 import build
        build.build()
    return fm


def ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Spacing of bfloat16 numbers at |x| (8 significand bits)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.power(2.0, e - 7)


def check_close_bf16(got: np.ndarray, ref: np.ndarray, max_abs: float, mean_abs: float = None,
                     what: str = ""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = np.maximum(max_abs, ulp_bf16(ref))
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements over bound; worst at {i}: "
                             f"got {got[i]} ref {ref[i]} err {err[i]:.3e} bound {bound[i]:.3e}")
    if mean_abs is not None:
        assert err.mean() <= mean_abs, f"{what}: mean abs {err.mean():.3e} > {mean_abs}"
    return float(err.max()), float(err.mean())


def check_lse(got: np.ndarray, ref: np.ndarray, what: str = "lse"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    ninf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf_ref), f"{what}: -inf rows differ"
    fin = ~ninf_ref
    if fin.any():
        err = np.abs(got[fin] - ref[fin])
        assert err.max() <= LSE_ABS, f"{what}: max abs {err.max():.3e}"
        return float(err.max())
    return 0.0


def to_device_bf16(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_tensor_to_f64(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def kv_slot(cu: np.ndarray, s: int, j: int, block_n: int) -> int:
    """Slot of sample-local key tile j of sample s in the statistics layout."""
    return int(cu[s]) // block_n + s + j
