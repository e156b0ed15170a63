"""Pins for the oracle's mask, block statistics and block classes.

Each check ties the oracle to something the FlashMask article prints or to
an independent brute-force construction, never to the oracle itself.
"""

import itertools

import numpy as np
import pytest

from fixtures import load
from oracle import mask as om
from workloads import gen


def _table():
    g = load("flashmask_16x16_causal.txt")
    n = g["n"]
    sri = np.zeros((1, 4, n), dtype=np.int32)
    sri[0, 0] = g["LTS"]
    sri[0, 1] = g["LTE"]
    sri[0, 2] = 0
    sri[0, 3] = n
    return g, sri


def _brute_mask(sri_h, n, causal):
    """Enumerate masked cells row by row from each column's two intervals."""
    m = [[False] * n for _ in range(n)]
    for j in range(n):
        for i in range(int(sri_h[0][j]), int(sri_h[1][j])):
            if i >= j:
                m[i][j] = True
        if causal:
            for i in range(0, j):
                m[i][j] = True
        else:
            for i in range(int(sri_h[2][j]), int(sri_h[3][j])):
                if i < j:
                    m[i][j] = True
    return np.array(m, dtype=bool)


def test_worked_table_column0():
    g, sri = _table()
    n = g["n"]
    m = om.dense_mask(sri[0], np.arange(n), np.arange(n), causal=True)
    lower_rows = [i for i in range(n) if m[i, 0]]
    assert lower_rows == g["col0_masked_rows"]
    # causal: every cell above the diagonal is masked, the diagonal is not
    for i in range(n):
        for j in range(i + 1, n):
            assert m[i, j]
    assert not m[0, 0]


def test_worked_table_matches_brute_force():
    g, sri = _table()
    n = g["n"]
    m = om.dense_mask(sri[0], np.arange(n), np.arange(n), causal=True)
    assert (m == _brute_mask(sri[0], n, True)).all()


def test_worked_table_tile0_minmax():
    g, sri = _table()
    cu = np.array([0, g["n"]], dtype=np.int32)
    st = om.block_minmax(sri, cu, g["block_n"])
    lts_min, lts_max, lte_min, lte_max = st[(0, 0, 0)][:4]
    assert (lts_min, lts_max) == (g["tile0_LTS_min"], g["tile0_LTS_max"])
    assert (lte_min, lte_max) == (g["tile0_LTE_min"], g["tile0_LTE_max"])


def test_worked_table_printed_classes():
    g, sri = _table()
    cu = np.array([0, g["n"]], dtype=np.int32)
    bm, bn = g["block_m"], g["block_n"]
    st = om.block_minmax(sri, cu, bn)
    for key in ("class_3_2", "class_1_1", "class_3_1"):
        _, a, b = key.split("_")
        qi, kj = int(a), int(b)
        got = om.classify_block(qi * bm, (qi + 1) * bm, kj * bn, (kj + 1) * bn,
                                st[(0, 0, kj)], causal=True)
        assert got == g[key], key


def _check_sound(sri, cu, bm, bn, causal, n_heads=1):
    """Fully masked blocks hold only masked cells; unmasked blocks none."""
    st = None if sri is None else om.block_minmax(sri, cu, bn)
    ctiles = om.tiles(cu, bn)
    for h in range(n_heads):
        mh = None if sri is None else sri[h]
        for s, _, r0, r1 in om.tiles(cu, bm):
            for s2, t, c0, c1 in ctiles:
                if s2 != s:
                    continue
                cls = om.classify_block(r0, r1, c0, c1, None if st is None else st[(h, s, t)],
                                        causal)
                m = om.dense_mask(mh, np.arange(r0, r1), np.arange(c0, c1), causal)
                if cls == om.FULL:
                    assert m.all(), (h, s, r0, c0)
                elif cls == om.UNMASKED:
                    assert not m.any(), (h, s, r0, c0)


def test_worked_table_classes_sound():
    g, sri = _table()
    cu = np.array([0, g["n"]], dtype=np.int32)
    _check_sound(sri, cu, g["block_m"], g["block_n"], True)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("causal", [False, True])
def test_random_intervals_classes_sound(seed, causal):
    wl = gen.make_custom([5, 17, 1, 9, 24], mask="random", causal=causal, seed=seed,
                         n_mask_heads=2, tensors=False)
    for bm, bn in [(4, 4), (8, 4), (4, 8), (16, 16)]:
        _check_sound(wl.startend_row_indices, wl.cu_seqlens, bm, bn, causal, n_heads=2)


def test_no_interval_mask_classes():
    cu = np.array([0, 10, 30], dtype=np.int32)
    _check_sound(None, cu, 4, 4, True)
    _check_sound(None, cu, 4, 4, False)
    f, p, u = om.block_class_counts(cu, None, 1, 4, 4, causal=False)
    assert f == 0 and p == 0 and u == 3 * 3 + 5 * 5


def test_interval_mask_exhaustive_small():
    """Every single-column pattern 0<=S<=E<=T of both triangles, T = 5."""
    n = 5
    intervals = [(a, b) for a in range(n + 1) for b in range(a, n + 1)]
    for j in range(n):
        for (lts, lte), (uts, ute) in itertools.product(intervals, intervals):
            sri = np.zeros((4, n), dtype=np.int32)
            sri[1, :] = n
            sri[3, :] = n
            sri[:, j] = [lts, lte, uts, ute]
            for causal in (False, True):
                m = om.dense_mask(sri, np.arange(n), np.array([j]), causal)[:, 0]
                b = _brute_mask(sri, n, causal)[:, j]
                assert (m == b).all()


def test_block_minmax_is_min_and_max():
    wl = gen.make_custom([7, 13, 3], mask="random", seed=3, tensors=False)
    st = om.block_minmax(wl.startend_row_indices, wl.cu_seqlens, 4)
    sri = wl.startend_row_indices
    for (h, s, t), v in st.items():
        c0 = int(wl.cu_seqlens[s]) + 4 * t
        c1 = min(c0 + 4, int(wl.cu_seqlens[s + 1]))
        for k in range(4):
            col = sorted(int(x) for x in sri[h, k, c0:c1])
            assert v[2 * k] == col[0] and v[2 * k + 1] == col[-1]


def test_tiny_workload_class_counts_closed_form():
    """Docs [32, 96, 128], Br = Bc = 64, causal document mask.

    Sample-local tiles: the 32-token doc is one straddling diagonal block; the
    96-token doc has two diagonal blocks, one lower block and one upper block;
    the 128-token doc likewise.  LTS = doc end makes every lower block
    unmasked, causality makes upper blocks fully masked and diagonal blocks
    partial: F = 2, P = 5, U = 2.
    """
    wl = gen.make_workload(1, tensors=False)
    f, p, u = om.block_class_counts(wl.cu_seqlens, wl.startend_row_indices, 1, 64, 64, True)
    assert (f, p, u) == (2, 5, 2)
