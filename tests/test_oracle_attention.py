"""Pins for the oracle's masked attention (FlashMask article, sections 3.3-3.4)."""

import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import attention as oat
from oracle import mask as om
from workloads import gen


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _brute(q, k, v, cu, sri, causal, scale):
    """Triple loop with math.exp; the mask cell test is written out per cell."""
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    out = np.zeros((T, Hq, D))
    lse = np.zeros((Hq, T))
    seg = np.zeros(T, dtype=int)
    for s in range(len(cu) - 1):
        seg[cu[s]:cu[s + 1]] = s
    for h in range(Hq):
        kh = h // (Hq // Hkv)
        mh = None if sri is None else sri[h if sri.shape[0] > 1 else 0]
        for i in range(T):
            keys = []
            for j in range(T):
                if seg[j] != seg[i]:
                    continue
                if i >= j:
                    hidden = mh is not None and mh[0][j] <= i < mh[1][j]
                else:
                    hidden = causal or (mh is not None and mh[2][j] <= i < mh[3][j])
                if not hidden:
                    keys.append(j)
            if not keys:
                lse[h, i] = -math.inf
                continue
            sc = [scale * sum(q[i, h, d] * k[j, kh, d] for d in range(D)) for j in keys]
            mx = max(sc)
            w = [math.exp(x - mx) for x in sc]
            tot = sum(w)
            lse[h, i] = mx + math.log(tot)
            for d in range(D):
                out[i, h, d] = sum(w[n] * v[keys[n], kh, d] for n in range(len(keys))) / tot
    return out, lse


def test_single_key_returns_its_value():
    q = _rand((1, 1, 8), 0)
    k = _rand((1, 1, 8), 1)
    v = _rand((1, 1, 8), 2)
    o, lse = oat.attention_forward(q, k, v, np.array([0, 1]), None, causal=True, scale=0.3)
    assert np.allclose(o[0, 0], v[0, 0])
    assert np.isclose(lse[0, 0], 0.3 * float(q[0, 0] @ k[0, 0]))


def test_bidirectional_single_sample_is_textbook_softmax():
    T, D = 11, 16
    q, k, v = _rand((T, 2, D), 3), _rand((T, 2, D), 4), _rand((T, 2, D), 5)
    o, lse = oat.attention_forward(q, k, v, np.array([0, T]), None, causal=False)
    for h in range(2):
        s = q[:, h] @ k[:, h].T / math.sqrt(D)
        assert np.allclose(o[:, h], softmax(s, axis=1) @ v[:, h], atol=1e-12)
        assert np.allclose(lse[h], logsumexp(s, axis=1), atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("causal", [False, True])
def test_matches_brute_force_loop(seed, causal):
    wl = gen.make_custom([3, 1, 6, 2], n_heads_q=4, n_heads_kv=2, head_dim=4, mask="random",
                         causal=causal, seed=seed, n_mask_heads=(4 if seed % 2 else 1),
                         tensors=False)
    T = wl.total_tokens
    q, k, v = _rand((T, 4, 4), 10 + seed), _rand((T, 2, 4), 20 + seed), _rand((T, 2, 4), 30 + seed)
    o, lse = oat.attention_forward(q, k, v, wl.cu_seqlens, wl.startend_row_indices, causal,
                                   scale=0.7)
    bo, blse = _brute(q, k, v, wl.cu_seqlens, wl.startend_row_indices, causal, 0.7)
    assert np.allclose(o, bo, atol=1e-12)
    assert np.array_equal(np.isinf(lse), np.isinf(blse))
    fin = np.isfinite(blse)
    assert np.allclose(lse[fin], blse[fin], atol=1e-12)


def test_fully_masked_row_convention():
    sri = np.zeros((1, 4, 3), dtype=np.int32)
    sri[0, 1] = 3   # LTS = 0, LTE = 3: every lower cell hidden
    sri[0, 3] = 3
    q, k, v = _rand((3, 1, 4), 0), _rand((3, 1, 4), 1), _rand((3, 1, 4), 2)
    o, lse = oat.attention_forward(q, k, v, np.array([0, 3]), sri, causal=True)
    assert np.all(o == 0.0) and np.all(np.isneginf(lse))


def test_causal_document_encodings_agree():
    """Three encodings of the same causal-document mask give equal results:
    samples from cu_seqlens + causal; one sample + LTS = doc end intervals;
    samples + intervals."""
    lens = [5, 9, 1, 7]
    wl = gen.make_custom(lens, n_heads_q=2, n_heads_kv=1, head_dim=8, tensors=False)
    T = wl.total_tokens
    q, k, v = _rand((T, 2, 8), 7), _rand((T, 1, 8), 8), _rand((T, 1, 8), 9)
    a = oat.attention_forward(q, k, v, wl.cu_seqlens, None, True)
    b = oat.attention_forward(q, k, v, np.array([0, T]), wl.startend_row_indices, True)
    c = oat.attention_forward(q, k, v, wl.cu_seqlens, wl.startend_row_indices, True)
    for x, y in ((a, b), (a, c)):
        assert np.allclose(x[0], y[0], rtol=0, atol=1e-13)
        assert np.allclose(x[1], y[1], rtol=0, atol=1e-13)


def test_prefix_lm_encodings_agree():
    from workloads.gen import bidir_prefix_intervals
    lens = [12, 9, 16]
    cu = np.array([0, 12, 21, 37], dtype=np.int32)
    kinds = ["bidir", "prefix_lm", "prefix_lm"]
    s1 = bidir_prefix_intervals(cu, kinds, 37, alt=False)
    s2 = bidir_prefix_intervals(cu, kinds, 37, alt=True)
    q, k, v = _rand((37, 1, 8), 1), _rand((37, 1, 8), 2), _rand((37, 1, 8), 3)
    a = oat.attention_forward(q, k, v, cu, s1, False)
    b = oat.attention_forward(q, k, v, cu, s2, False)
    assert np.allclose(a[0], b[0], atol=1e-14) and np.allclose(a[1], b[1], atol=1e-14)
    # the prefix-LM sample: rows of the prefix never see keys after the prefix
    a0 = 21
    m = om.dense_mask(s1[0], np.arange(a0, 37), np.arange(a0, 37), False)
    P = 16 // 4
    assert not m[:, :P].any()
    for i in range(16):
        for j in range(P, 16):
            assert m[i, j] == (i < j)
    assert sum(lens) == 37


def test_gqa_head_mapping_equals_expanded_heads():
    wl = gen.make_custom([6, 4], n_heads_q=4, n_heads_kv=2, head_dim=8, tensors=False)
    T = wl.total_tokens
    q, k, v = _rand((T, 4, 8), 1), _rand((T, 2, 8), 2), _rand((T, 2, 8), 3)
    a = oat.attention_forward(q, k, v, wl.cu_seqlens, wl.startend_row_indices, True)
    ke, ve = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    b = oat.attention_forward(q, ke, ve, wl.cu_seqlens, wl.startend_row_indices, True)
    assert np.array_equal(a[0], b[0])


def test_row_subset_matches_full():
    wl = gen.make_custom([40, 300], n_heads_q=2, n_heads_kv=1, head_dim=8, tensors=False)
    T = wl.total_tokens
    q, k, v = _rand((T, 2, 8), 1), _rand((T, 1, 8), 2), _rand((T, 1, 8), 3)
    full = oat.attention_forward(q, k, v, wl.cu_seqlens, wl.startend_row_indices, True)
    rows = [0, 39, 40, 41, 299, 339]
    part = oat.attention_forward(q, k, v, wl.cu_seqlens, wl.startend_row_indices, True, rows=rows)
    assert np.array_equal(full[0][rows], part[0][rows])


def test_effective_pairs_tiny_workload():
    """Docs [32, 96, 128], causal: sum n(n+1)/2 = 528 + 4656 + 8256."""
    wl = gen.make_workload(1, tensors=False)
    assert oat.effective_pairs(wl.cu_seqlens, wl.startend_row_indices, True) == 13440
