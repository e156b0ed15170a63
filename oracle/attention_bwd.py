"""Gradients of masked softmax attention over packed samples, float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

PaddleNLP FlashMask article, section 3.4: the backward operator takes q, k,
v, the column intervals (startend_row_indices), out, softmax_lse and the
output gradient, and returns the gradients of q, k and v.  Section 3.3: the
block-skipping kernel equals dense-mask attention, so the gradient is the
plain gradient of the oracle's forward pass (``attention.attention_forward``)
under the same dense mask.  Written out from the chain rule, for every
sample, q head h (key/value head g = h // (Hq / Hkv)) and unmasked pair
(i, j):

    p_ij   = exp(scale * q_i . k_j - lse_i)
    dv_j  += sum_i p_ij * do_i
    dp_ij  = do_i . v_j
    delta_i = sum_j p_ij * dp_ij  = do_i . o_i
    ds_ij  = p_ij * (dp_ij - delta_i)
    dq_i   = scale * sum_j ds_ij * k_j
    dk_j  += scale * sum_i ds_ij * q_i

dk and dv of a key/value head sum the contributions of all its q heads.
Reading (the pages do not say): rows with no unmasked key contribute nothing
(their p row is zero).

Pinned in ``tests/test_oracle_attention_bwd.py`` by central finite
differences of ``attention_forward``, which is itself pinned to the pages.
"""

from __future__ import annotations

from typing import Optional

import numpy as np

from .mask import dense_mask


def attention_backward(q: np.ndarray, k: np.ndarray, v: np.ndarray, dout: np.ndarray,
                       cu_seqlens: np.ndarray, sri: Optional[np.ndarray], causal: bool,
                       scale: Optional[float] = None, magnitudes: bool = False):
    """Returns (dq [T, Hq, D], dk [T, Hkv, D], dv [T, Hkv, D]) in float64.

    With ``magnitudes=True`` also returns the magnitude sums (mq, mk, mv) of
    the same shapes that bound how far rounded arithmetic can stray from
    these values (used only to derive test tolerances):
        e_i  = sum_d |do_id| (sum_j p_ij |v_jd|)
        mv_j = sum_i p_ij |do_i|
        mk_j = scale * sum_i (|ds_ij| + p_ij e_i) |q_i|
        mq_i = scale * sum_j (|ds_ij| + p_ij e_i) |k_j|
    summed over the q heads of a key/value head like the gradients.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(dout, dtype=np.float64)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    group = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    dq = np.zeros((T, Hq, D))
    dk = np.zeros((T, Hkv, D))
    dv = np.zeros((T, Hkv, D))
    if magnitudes:
        mq = np.zeros((T, Hq, D))
        mk = np.zeros((T, Hkv, D))
        mv = np.zeros((T, Hkv, D))
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        if b <= a:
            continue
        idx = np.arange(a, b)
        for h in range(Hq):
            g = h // group
            mh = None if sri is None else sri[h if sri.shape[0] > 1 else 0]
            masked = dense_mask(mh, idx, idx, causal)
            scores = scale * (q[a:b, h, :] @ k[a:b, g, :].T)
            scores = np.where(masked, -np.inf, scores)
            m = scores.max(axis=1)
            empty = ~np.isfinite(m)
            m_safe = np.where(empty, 0.0, m)
            e = np.exp(scores - m_safe[:, None])
            l = e.sum(axis=1)
            p = e / np.where(empty, 1.0, l)[:, None]
            p[empty] = 0.0
            o = p @ v[a:b, g, :]
            dp = do[a:b, h, :] @ v[a:b, g, :].T
            delta = (do[a:b, h, :] * o).sum(axis=1)
            ds = p * (dp - delta[:, None])
            dv[a:b, g, :] += p.T @ do[a:b, h, :]
            dq[a:b, h, :] = scale * (ds @ k[a:b, g, :])
            dk[a:b, g, :] += scale * (ds.T @ q[a:b, h, :])
            if magnitudes:
                eo = (np.abs(do[a:b, h, :]) * (p @ np.abs(v[a:b, g, :]))).sum(axis=1)
                w = np.abs(ds) + p * eo[:, None]
                mv[a:b, g, :] += p.T @ np.abs(do[a:b, h, :])
                mk[a:b, g, :] += scale * (w.T @ np.abs(q[a:b, h, :]))
                mq[a:b, h, :] = scale * (w @ np.abs(k[a:b, g, :]))
    if magnitudes:
        return dq, dk, dv, mq, mk, mv
    return dq, dk, dv


def row_delta(out: np.ndarray, dout: np.ndarray) -> np.ndarray:
    """delta[h, i] = do_i . o_i (the row term of ds), float64 [Hq, T]."""
    o = np.asarray(out, dtype=np.float64)
    do = np.asarray(dout, dtype=np.float64)
    return np.einsum("thd,thd->ht", do, o)
