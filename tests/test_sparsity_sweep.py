"""Sparsity-sweep workloads (FlashMask article, section 4.3): one segment,
structure expressed only through the column intervals.

Each mask is pinned against a brute-force predicate of its pattern through
the oracle's dense mask; along each family the block sparsity (fully masked
blocks over all blocks of the T x T grid, from the oracle's block classes)
must grow with the family parameter.
"""

import numpy as np
import pytest

from oracle import mask as om
from workloads import gen

T = 256


def predicate(family, param):
    if family in ("causal_document", "document"):
        doc = np.arange(T) // (T // param)
        if family == "causal_document":
            return lambda i, j: j <= i and doc[i] == doc[j]
        return lambda i, j: doc[i] == doc[j]
    g = T // 4
    q = g // 4
    rest = g - q
    alens = [rest // param] * param
    alens[-1] += rest - sum(alens)
    group = np.arange(T) // g
    owner = np.full(T, -1)
    for g0 in range(0, T, g):
        a0 = g0 + q
        for k, a in enumerate(alens):
            owner[a0:a0 + a] = k
            a0 += a
    return lambda i, j: j <= i and group[i] == group[j] and (owner[j] < 0 or owner[j] == owner[i])


@pytest.mark.parametrize("idx", range(len(gen.sparsity_sweep(T))))
def test_sweep_masks_match_their_pattern(idx):
    family, param, causal, sri = gen.sparsity_sweep(T)[idx]
    assert sri.shape == (1, 4, T)
    got = ~om.dense_mask(sri[0], np.arange(T), np.arange(T), causal)
    pred = predicate(family, param)
    want = np.array([[pred(i, j) for j in range(T)] for i in range(T)])
    assert np.array_equal(got, want), (family, param)


def test_sparsity_grows_along_each_family():
    # the sweep's answer lengths are multiples of the block width at its own
    # size (16384 tokens, 128-column blocks); the same holds for 4096 tokens
    # and 32-column blocks (answers of 768 / k tokens)
    n = 4096
    cu = np.array([0, n], dtype=np.int32)
    rho = {}
    for family, param, causal, sri in gen.sparsity_sweep(n):
        f, p, u = om.block_class_counts(cu, sri, 1, 32, 32, causal)
        rho.setdefault(family, []).append((param, f / (f + p + u)))
    for family, pts in rho.items():
        vals = [r for _, r in sorted(pts)]
        assert all(b >= a for a, b in zip(vals, vals[1:])), (family, vals)
        assert vals[-1] > vals[0], family
