"""Pins of the float64 attention-gradient oracle.

The gradient of L = sum(dout * attention_forward(q, k, v)) is checked
against central finite differences of the (separately pinned) forward
oracle on tiny packed inputs, for every mask style, GQA and fully masked
rows; plus two closed-form cases.  A dropped term (the delta row term), a
wrong sign, a missing scale or a transposed operand each fail one of these.
"""

import numpy as np
import pytest

from oracle import attention as oat
from oracle import attention_bwd as ob
from workloads import gen


def loss(q, k, v, dout, cu, sri, causal):
    o, _ = oat.attention_forward(q, k, v, cu, sri, causal)
    return float((dout * o).sum())


def finite_diff(fn, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + h
        fp = fn()
        x[i] = old - h
        fm = fn()
        x[i] = old
        g[i] = (fp - fm) / (2 * h)
    return g


CASES = [
    # lens, Hq, Hkv, mask, causal
    ([5, 7], 2, 1, "causal_document", True),
    ([9], 2, 2, "none", False),
    ([4, 6, 3], 4, 2, "window", True),
    ([8, 5], 2, 1, "bidir_prefix", False),
    ([6, 6], 2, 2, "random", False),
    ([7, 4], 2, 1, "random", True),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_gradient_matches_finite_differences(case):
    lens, hq, hkv, mask, causal = CASES[case]
    wl = gen.make_custom(lens, n_heads_q=hq, n_heads_kv=hkv, head_dim=4, mask=mask,
                         causal=causal, window=3, seed=case, tensors=False)
    rng = np.random.default_rng(100 + case)
    T = wl.total_tokens
    q = rng.standard_normal((T, hq, 4))
    k = rng.standard_normal((T, hkv, 4))
    v = rng.standard_normal((T, hkv, 4))
    do = rng.standard_normal((T, hq, 4))
    cu, sri = wl.cu_seqlens, wl.startend_row_indices
    dq, dk, dv = ob.attention_backward(q, k, v, do, cu, sri, causal)
    f = lambda: loss(q, k, v, do, cu, sri, causal)
    np.testing.assert_allclose(dq, finite_diff(f, q), atol=1e-7, rtol=1e-6)
    np.testing.assert_allclose(dk, finite_diff(f, k), atol=1e-7, rtol=1e-6)
    np.testing.assert_allclose(dv, finite_diff(f, v), atol=1e-7, rtol=1e-6)


def test_fully_masked_rows_have_zero_gradient():
    wl = gen.make_custom([6], n_heads_q=1, n_heads_kv=1, head_dim=4, mask="none", causal=True,
                         tensors=False)
    sri = np.zeros((1, 4, 6), dtype=np.int32)
    sri[0, 0, :] = 0          # every row of every column masked below the diagonal
    sri[0, 1, :] = 6
    rng = np.random.default_rng(0)
    x = [rng.standard_normal((6, 1, 4)) for _ in range(4)]
    dq, dk, dv = ob.attention_backward(*x, wl.cu_seqlens, sri, True)
    assert not dq.any() and not dk.any() and not dv.any()


def test_single_key_closed_form():
    # one token: p = 1, o = v, so dv = dout and dq = dk = 0 (ds = p (dp - dp) = 0)
    rng = np.random.default_rng(1)
    q, k, v, do = (rng.standard_normal((1, 1, 8)) for _ in range(4))
    dq, dk, dv = ob.attention_backward(q, k, v, do, np.array([0, 1]), None, True)
    np.testing.assert_allclose(dv, do, atol=1e-15)
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15


def test_row_delta_is_rowsum_of_p_times_dp():
    wl = gen.make_custom([10, 6], n_heads_q=2, n_heads_kv=1, head_dim=8, mask="causal_document",
                         seed=3, tensors=False)
    rng = np.random.default_rng(2)
    T = wl.total_tokens
    q, do = rng.standard_normal((T, 2, 8)), rng.standard_normal((T, 2, 8))
    k, v = rng.standard_normal((T, 1, 8)), rng.standard_normal((T, 1, 8))
    o, lse = oat.attention_forward(q, k, v, wl.cu_seqlens, wl.startend_row_indices, True)
    delta = ob.row_delta(o, do)
    # do_i . o_i = sum_j p_ij (do_i . v_j) with p from lse
    for h in range(2):
        for i in range(T):
            s = 0 if i < 10 else 10
            e = 10 if i < 10 else 16
            js = np.arange(s, i + 1)
            p = np.exp((q[i, h] @ k[js, 0].T) / np.sqrt(8) - lse[h, i])
            assert abs(delta[h, i] - (p * (v[js, 0] @ do[i, h])).sum()) < 1e-12


def test_magnitude_sums_bound_the_gradients():
    # |sum of terms| <= sum of |terms|; with dout >= 0 the dv sum has no
    # cancellation and equals its magnitude sum
    wl = gen.make_custom([9, 14], n_heads_q=4, n_heads_kv=2, head_dim=8, mask="window",
                         window=5, seed=4, tensors=False)
    rng = np.random.default_rng(9)
    T = wl.total_tokens
    q, do = rng.standard_normal((T, 4, 8)), rng.standard_normal((T, 4, 8))
    k, v = rng.standard_normal((T, 2, 8)), rng.standard_normal((T, 2, 8))
    cu, sri = wl.cu_seqlens, wl.startend_row_indices
    dq, dk, dv, mq, mk, mv = ob.attention_backward(q, k, v, do, cu, sri, True, magnitudes=True)
    assert np.all(mq >= np.abs(dq) - 1e-12)
    assert np.all(mk >= np.abs(dk) - 1e-12)
    assert np.all(mv >= np.abs(dv) - 1e-12)
    g = ob.attention_backward(q, k, v, np.abs(do), cu, sri, True, magnitudes=True)
    np.testing.assert_allclose(g[2], g[5], rtol=1e-12)
    # the gradients themselves do not depend on the option
    np.testing.assert_array_equal(ob.attention_backward(q, k, v, do, cu, sri, True)[0], dq)
