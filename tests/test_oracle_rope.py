"""Pins for the oracle's RoPE (Unsloth packing blog, fused QK RoPE section)."""

import numpy as np

from oracle import rope as orope


def _x(T, H, D, seed=0):
    return np.random.default_rng(seed).standard_normal((T, H, D))


def test_position_zero_is_identity():
    x = _x(4, 3, 16)
    cu = np.array([0, 1, 2, 3, 4], dtype=np.int32)  # every token at position 0
    assert np.array_equal(orope.rope_apply(x, cu, 1e4), x)


def test_positions_reset_per_sample():
    cu = np.array([0, 3, 3, 7, 8], dtype=np.int32)
    assert orope.positions(cu, 8).tolist() == [0, 1, 2, 0, 1, 2, 3, 0]


def test_matches_complex_rotation():
    """Pair (x_i, x_{i+D/2}) as the complex number x_i + i x_{i+D/2}.

    Multiplying it by exp(i * p * theta^(-2i/D)) is the same rotation written
    without rotate_half; a sign or half-swap error in rotate_half breaks it.
    """
    T, H, D, theta = 9, 2, 32, 500000.0
    x = _x(T, H, D, 1)
    cu = np.array([0, 4, 9], dtype=np.int32)
    y = orope.rope_apply(x, cu, theta)
    pos = np.array([0, 1, 2, 3, 0, 1, 2, 3, 4], dtype=np.float64)
    inv = np.array([theta ** (-2.0 * i / D) for i in range(D // 2)])
    z = x[..., : D // 2] + 1j * x[..., D // 2:]
    w = z * np.exp(1j * pos[:, None, None] * inv[None, None, :])
    assert np.allclose(y[..., : D // 2], w.real, atol=1e-12)
    assert np.allclose(y[..., D // 2:], w.imag, atol=1e-12)


def test_first_pair_frequency_is_one():
    D = 64
    x = np.zeros((2, 1, D))
    x[1, 0, 0] = 1.0   # unit vector on pair 0 at position 1
    y = orope.rope_apply(x, np.array([0, 2], dtype=np.int32), 1e4)
    assert np.isclose(y[1, 0, 0], np.cos(1.0)) and np.isclose(y[1, 0, D // 2], np.sin(1.0))


def test_pairwise_norm_preserved():
    x = _x(20, 3, 64, 2)
    cu = np.array([0, 7, 20], dtype=np.int32)
    y = orope.rope_apply(x, cu, 1e6)
    nx = x[..., :32] ** 2 + x[..., 32:] ** 2
    ny = y[..., :32] ** 2 + y[..., 32:] ** 2
    assert np.allclose(nx, ny, rtol=1e-12, atol=1e-12)


def test_backward_undoes_forward():
    """The blog's backward rule (sin -> -sin) is the inverse rotation."""
    x = _x(30, 2, 128, 3)
    cu = np.array([0, 11, 30], dtype=np.int32)
    y = orope.rope_apply(x, cu, 1e4)
    assert np.allclose(orope.rope_backward(y, cu, 1e4), x, atol=1e-12)


def test_backward_matches_finite_differences():
    """d/dx sum(w * rope(x)) equals rope_backward(w), the blog's dC/dY rule."""
    T, H, D = 5, 1, 8
    rng = np.random.default_rng(4)
    x = rng.standard_normal((T, H, D))
    w = rng.standard_normal((T, H, D))
    cu = np.array([0, 2, 5], dtype=np.int32)
    g = orope.rope_backward(w, cu, 100.0)
    eps = 1e-6
    num = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp = x.copy()
        xm = x.copy()
        xp[idx] += eps
        xm[idx] -= eps
        num[idx] = ((w * orope.rope_apply(xp, cu, 100.0)).sum()
                    - (w * orope.rope_apply(xm, cu, 100.0)).sum()) / (2 * eps)
    assert np.allclose(num, g, atol=1e-7)
