"""Host packing and collation utility (packed_varlen_attention_gb300.packing).

Pinned against the oracle's dense mask (a separate restatement of the
column-interval rule) and against brute-force predicates of each mask
pattern written out here from its definition:

* causal:            row i sees column j iff j <= i
* bidirectional:     every pair of the sample is visible
* prefix-LM (p):     j <= i, or both i and j inside the prefix
* shared question:   j <= i and (j in the prompt or j in the answer of i)
* sliding window w:  j <= i < j + w

The collated (global) intervals must give, over the whole pack, the block
diagonal of the per-sample masks with every cross-sample pair masked (the
ZeroPadding offset rule of the FlashMask article, section 6.7).
"""

import numpy as np
import pytest

from oracle import mask as om
from packed_varlen_attention_gb300 import packing as pk


def visible_matrix(n, pred):
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    return np.vectorize(pred)(i, j)


def sample_mask(sri, n, causal):
    """Dense mask of one sample on its own (local coordinates)."""
    full = pk._expand_local(sri, n, 1)[0]
    return om.dense_mask(full, np.arange(n), np.arange(n), causal)


# -------------------------------------------------------------- greedy packing

def test_greedy_pack_example():
    # room 10, input order: 7 -> A; 5 -> B (no room in A); 3 -> A (full);
    # 4 -> B; 2 -> C (A full, B has 1 left); 6 -> C.
    # Longest first (7, 6, 5, 4, 3, 2): 7 -> A; 6 -> B; 5 -> C; 4 -> B;
    # 3 -> A; 2 -> C.
    lens = [7, 5, 3, 4, 2, 6]
    assert pk.greedy_pack(lens, 10) == [[0, 2], [1, 3], [4, 5]]
    assert pk.greedy_pack(lens, 10, longest_first=True) == [[0, 2], [5, 3], [1, 4]]


@pytest.mark.parametrize("seed", range(5))
def test_greedy_pack_properties(seed):
    rng = np.random.default_rng(seed)
    lens = list(rng.integers(0, 700, size=60))
    cap = 1024
    packs = pk.greedy_pack(lens, cap)
    flat = sorted(i for p in packs for i in p)
    assert flat == list(range(len(lens)))            # every sample exactly once
    assert all(sum(lens[i] for i in p) <= cap for p in packs)
    # first fit: when sample i was placed, no earlier pack had room for it
    used = []
    where = {i: k for k, p in enumerate(packs) for i in p}
    for i in range(len(lens)):
        k = where[i]
        while len(used) <= k:
            used.append(0)
        for q in range(k):
            assert used[q] + lens[i] > cap
        used[k] += lens[i]


def test_greedy_pack_rejects():
    with pytest.raises(ValueError):
        pk.greedy_pack([5, 11], 10)
    with pytest.raises(ValueError):
        pk.greedy_pack([-1], 10)
    with pytest.raises(ValueError):
        pk.greedy_pack([1], 0)


# ------------------------------------------------------ per-sample patterns

@pytest.mark.parametrize("n", [1, 7, 40])
def test_causal_and_bidirectional(n):
    assert np.array_equal(~sample_mask(pk.intervals_causal(n), n, False),
                          visible_matrix(n, lambda i, j: j <= i))
    assert np.array_equal(~sample_mask(pk.intervals_causal(n), n, True),
                          visible_matrix(n, lambda i, j: j <= i))
    assert np.array_equal(~sample_mask(pk.intervals_bidirectional(n), n, False),
                          np.ones((n, n), dtype=bool))


@pytest.mark.parametrize("n,p", [(10, 0), (10, 4), (10, 10), (33, 17)])
def test_prefix_lm(n, p):
    got = ~sample_mask(pk.intervals_prefix_lm(n, p), n, False)
    want = visible_matrix(n, lambda i, j: (j <= i) or (i < p and j < p))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("prompt,answers", [(5, [3, 4]), (1, [1, 1, 1]), (12, [0, 7, 2, 9]), (0, [6])])
def test_shared_question(prompt, answers):
    n = prompt + sum(answers)
    owner = np.full(n, -1)
    e = prompt
    for k, a in enumerate(answers):
        owner[e:e + a] = k
        e += a
    got = ~sample_mask(pk.intervals_shared_question(prompt, answers), n, True)
    want = visible_matrix(n, lambda i, j: j <= i and (owner[j] < 0 or owner[j] == owner[i]))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("n,w", [(20, 1), (20, 5), (20, 50)])
def test_sliding_window(n, w):
    got = ~sample_mask(pk.intervals_sliding_window(n, w), n, True)
    want = visible_matrix(n, lambda i, j: j <= i < j + w)
    assert np.array_equal(got, want)


# ------------------------------------------------------------- collation

def _random_samples(rng, k):
    lens, ivs = [], []
    for _ in range(k):
        kind = rng.integers(0, 6)
        if kind == 0:
            n = int(rng.integers(1, 40)); iv = pk.intervals_causal(n)
        elif kind == 1:
            n = int(rng.integers(1, 40)); iv = pk.intervals_bidirectional(n)
        elif kind == 2:
            n = int(rng.integers(1, 40)); iv = pk.intervals_prefix_lm(n, int(rng.integers(0, n + 1)))
        elif kind == 3:
            q = int(rng.integers(0, 15)); ans = list(rng.integers(0, 10, size=3))
            n = q + int(sum(ans)); iv = pk.intervals_shared_question(q, ans)
        elif kind == 4:
            n = int(rng.integers(1, 40)); iv = pk.intervals_sliding_window(n, int(rng.integers(1, 12)))
        else:
            n = int(rng.integers(0, 40)); iv = None     # no interval mask (causal)
        lens.append(n); ivs.append(iv)
    return lens, ivs


@pytest.mark.parametrize("seed", range(6))
def test_collate_is_block_diagonal_of_samples(seed):
    rng = np.random.default_rng(100 + seed)
    lens, ivs = _random_samples(rng, 7)
    toks = [rng.integers(0, 50000, size=n) for n in lens]
    packed = pk.collate(toks, ivs)
    T = packed.total_tokens
    cu = packed.cu_seqlens.astype(np.int64)
    assert cu[0] == 0 and list(np.diff(cu)) == lens and T == sum(lens)
    assert np.array_equal(packed.tokens, np.concatenate(toks))
    sri = packed.startend_row_indices
    assert sri.shape == (1, 4, T) and sri.dtype == np.int32
    for causal in (False, True):
        whole = om.dense_mask(sri[0], np.arange(T), np.arange(T), causal)
        seg = np.searchsorted(cu, np.arange(T), side="right") - 1
        whole |= seg[:, None] != seg[None, :]            # the cu_seqlens restriction
        want = np.ones((T, T), dtype=bool)
        for s, n in enumerate(lens):
            a = cu[s]
            want[a:a + n, a:a + n] = sample_mask(ivs[s], n, causal)
        assert np.array_equal(whole, want), causal


def test_collate_partial_vectors_and_heads():
    # [LTS] only, [LTS, LTE], per-head intervals: omitted vectors take the
    # defaults LTE = UTE = n, UTS = 0 before the offset
    a = np.array([[2, 3, 3]])                 # LTS of a 3-token sample
    b = np.array([[1, 1], [2, 2]])            # LTS, LTE of a 2-token sample
    c = np.stack([pk.intervals_causal(4)[0], pk.intervals_bidirectional(4)[0]])  # 2 heads
    p = pk.collate([np.zeros(3), np.zeros(2), np.zeros(4)], [a, b, c], n_mask_heads=2)
    sri = p.startend_row_indices
    assert p.cu_seqlens.tolist() == [0, 3, 5, 9]
    assert sri[0, :, 0:3].tolist() == [[2, 3, 3], [3, 3, 3], [0, 0, 0], [3, 3, 3]]
    assert sri[1, :, 0:3].tolist() == sri[0, :, 0:3].tolist()
    assert sri[0, :, 3:5].tolist() == [[4, 4], [5, 5], [3, 3], [5, 5]]
    assert sri[0, :, 5:9].tolist() == (c[0] + 5).tolist()
    assert sri[1, :, 5:9].tolist() == (c[1] + 5).tolist()


def test_collate_without_intervals_and_errors():
    p = pk.collate([np.arange(3), np.arange(0), np.arange(5)])
    assert p.startend_row_indices is None and p.cu_seqlens.tolist() == [0, 3, 3, 8]
    with pytest.raises(ValueError):
        pk.collate([np.zeros(3)], [np.zeros((1, 4, 2), dtype=np.int32)])   # wrong length
    with pytest.raises(ValueError):
        pk.collate([np.zeros(3)], [np.full((1, 1, 3), 4)])                  # bound beyond n
    with pytest.raises(ValueError):
        pk.collate([np.zeros(3), np.zeros(2)], [None])                      # one entry per sample
