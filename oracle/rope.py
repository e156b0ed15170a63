"""RoPE with per-sample position reset, float64 (test infrastructure only).

Unsloth packing blog, section "Fused QK RoPE Triton kernel with packing":
the rotation is ``Y = Q*cos + rotate_half(Q)*sin`` where
``rotate_half(Q) = Q @ R`` and ``R = [[0, I], [-I, 0]]``; the backward pass
is the same expression with ``R^T = -R``, i.e. ``sin -> -sin``.  Section
"Uncontaminated packing": position ids restart at every packed sample.

Reading (the pages print neither the frequencies nor the pairing): channel i
of the first half pairs with channel i + D/2 (the half-split pairing that the
block matrix R fixes), and the angle of pair i at position p is
``p * theta ** (-2 i / D)``, the standard RoPE frequencies, with theta the
base each workload names.
"""

from __future__ import annotations

import numpy as np


def frequencies(head_dim: int, theta: float) -> np.ndarray:
    """Inverse frequencies ``theta ** (-2 i / D)`` for i in [0, D/2)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def positions(cu_seqlens: np.ndarray, total_tokens: int) -> np.ndarray:
    """Position of every packed token inside its own sample: ``t - cu[s]``."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    pos = np.empty(total_tokens, dtype=np.int64)
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        pos[a:b] = np.arange(b - a)
    return pos


def rotate_half(x: np.ndarray) -> np.ndarray:
    """``x @ R`` with ``R = [[0, I], [-I, 0]]``: ``[x1, x2] -> [-x2, x1]``."""
    half = x.shape[-1] // 2
    return np.concatenate([-x[..., half:], x[..., :half]], axis=-1)


def rope_apply(x: np.ndarray, cu_seqlens: np.ndarray, theta: float,
               backward: bool = False, tokens=None) -> np.ndarray:
    """Rotate ``x`` of shape [T, H, D] (float64); ``backward`` flips sin.

    With ``tokens`` (global token indices), ``x`` holds only those tokens'
    rows, [len(tokens), H, D], and each row keeps its own position.
    """
    x = np.asarray(x, dtype=np.float64)
    _, _, D = x.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    pos = positions(cu, int(cu[-1]))
    if tokens is not None:
        pos = pos[np.asarray(tokens, dtype=np.int64)]
    ang = pos[:, None].astype(np.float64) * frequencies(D, theta)[None, :]
    cos = np.cos(ang)
    sin = np.sin(ang)
    if backward:
        sin = -sin
    cos = np.concatenate([cos, cos], axis=-1)[:, None, :]
    sin = np.concatenate([sin, sin], axis=-1)[:, None, :]
    return x * cos + rotate_half(x) * sin


def rope_backward(dy: np.ndarray, cu_seqlens: np.ndarray, theta: float) -> np.ndarray:
    """Gradient of the rotation w.r.t. its input: ``dY*cos + dY @ R^T * sin``."""
    return rope_apply(dy, cu_seqlens, theta, backward=True)
