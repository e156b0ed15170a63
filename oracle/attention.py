"""Masked softmax attention over packed samples, float64 (test infrastructure).

PaddleNLP FlashMask article, section 3.3: block skipping leaves the result
equal to attention under the equivalent dense mask, so the oracle computes
that plain definition: for every packed sample s, q head h and row i of s,

    s_ij  = scale * q_i . k_j        for unmasked keys j of sample s
    lse_i = log sum_j exp(s_ij)      (natural log)
    o_i   = sum_j exp(s_ij - lse_i) v_j

with the mask of ``oracle.mask.dense_mask``.  Grouped-query heads share
key/value head ``h // (Hq / Hkv)``.  Section 3.4 lists ``softmax_lse`` among
the backward operator's inputs, so the forward pass also returns lse.

Reading (the pages do not say): a row with no unmasked key gets o = 0 and
lse = -inf.

The dense mask is built one slab of rows at a time from the column
intervals; no T x T array is ever allocated.
"""

from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

from .mask import dense_mask


def attention_forward(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                      cu_seqlens: np.ndarray, sri: Optional[np.ndarray],
                      causal: bool, scale: Optional[float] = None,
                      rows: Optional[Sequence[int]] = None,
                      heads: Optional[Sequence[int]] = None,
                      slab: int = 256):
    """Reference forward pass.

    q: [T, Hq, D], k/v: [T, Hkv, D] (any float dtype, promoted to float64).
    sri: int [Hm][4][T] with Hm in {1, Hq}, or None.
    rows: optional subset of global rows to evaluate (others left NaN).
    heads: optional subset of q heads to evaluate (others left NaN).

    Returns (out [T, Hq, D] float64, lse [Hq, T] float64).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    group = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    out = np.full((T, Hq, D), np.nan)
    lse = np.full((Hq, T), np.nan)
    want = None
    if rows is not None:
        want = np.zeros(T, dtype=bool)
        want[np.asarray(rows, dtype=np.int64)] = True
    head_list = range(Hq) if heads is None else heads
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        if b <= a:
            continue
        cols = np.arange(a, b)
        for r0 in range(a, b, slab):
            r = np.arange(r0, min(r0 + slab, b))
            if want is not None:
                r = r[want[r]]
                if r.size == 0:
                    continue
            for h in head_list:
                mh = None if sri is None else sri[h if sri.shape[0] > 1 else 0]
                masked = dense_mask(mh, r, cols, causal)
                kv = h // group
                scores = scale * (q[r, h, :] @ k[a:b, kv, :].T)
                scores = np.where(masked, -np.inf, scores)
                m = scores.max(axis=1)
                empty = ~np.isfinite(m)
                m_safe = np.where(empty, 0.0, m)
                p = np.exp(scores - m_safe[:, None])
                l = p.sum(axis=1)
                o = (p @ v[a:b, kv, :]) / np.where(empty, 1.0, l)[:, None]
                o[empty] = 0.0
                out[r, h, :] = o
                lse[h, r] = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, l)))
    return out, lse


def effective_pairs(cu_seqlens: np.ndarray, sri: Optional[np.ndarray], causal: bool,
                    mask_head: int = 0, slab: int = 1024) -> int:
    """Number of unmasked (query, key) pairs of one mask head."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    total = 0
    mh = None if sri is None else sri[mask_head]
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        cols = np.arange(a, b)
        for r0 in range(a, b, slab):
            r = np.arange(r0, min(r0 + slab, b))
            total += int((~dense_mask(mh, r, cols, causal)).sum())
    return total
