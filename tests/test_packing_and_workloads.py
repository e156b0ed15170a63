"""Closed forms of the pages (packing arithmetic) and workload-recipe checks."""

import numpy as np
import pytest

from fixtures import load
from oracle import packing as opk
from workloads import gen


def test_half_long_half_short_speedup():
    """Unsloth blog: batch of half L and half S samples -> 2L / (L + S)."""
    for L, S in [(1024, 64), (4096, 4096), (512, 1)]:
        lens = [L] * 4 + [S] * 4
        assert np.isclose(opk.padding_speedup(lens), 2 * L / (L + S))


def test_speedup_limits():
    """S -> 0 gives 2; 20 % long / 80 % short gives L / (0.2 L + 0.8 S) -> 5."""
    L = 10 ** 7
    assert np.isclose(opk.padding_speedup([L] * 5 + [1] * 5), 2.0, rtol=1e-6)
    lens = [L] * 2 + [1] * 8
    assert np.isclose(opk.padding_speedup(lens), L / (0.2 * L + 0.8 * 1))
    assert np.isclose(opk.padding_speedup(lens), 5.0, rtol=1e-5)


def test_varlen_document_example():
    g = load("varlen_grid_example.txt")
    lens = g["lengths"]
    assert opk.padded_tokens(lens) == g["padded_tokens"]
    assert opk.packed_tokens(lens) == g["real_tokens"]
    assert opk.varlen_grid_blocks(lens, g["n_head"], g["block_m"]) == g["grid_blocks"]
    assert -(-max(lens) // g["block_m"]) == g["grid_z"]
    # launching only real Q tiles: (1 + 1 + 32) tiles x 2 heads
    assert opk.real_q_tiles(lens, g["n_head"], g["block_m"]) == 68


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_workload_structure(cfg):
    wl = gen.make_workload(cfg, seed=0, tensors=False)
    cu = wl.cu_seqlens.astype(np.int64)
    assert cu[0] == 0 and cu[-1] == wl.total_tokens and np.all(np.diff(cu) >= 0)
    sri = wl.startend_row_indices
    T = wl.total_tokens
    assert sri.shape == (1, 4, T)
    assert np.all((0 <= sri) & (sri <= T))
    assert np.all(sri[0, 0] <= sri[0, 1]) and np.all(sri[0, 2] <= sri[0, 3])
    j = np.arange(T)
    # every recipe keeps lower intervals strictly below and upper ones above
    # the diagonal, so the per-triangle reading and the plain union agree
    assert np.all(sri[0, 0] > j)
    assert np.all((sri[0, 3] <= j) | (sri[0, 2] == 0) & (sri[0, 3] == T))
    if cfg == 2:
        assert T == 8192 and (wl.n_heads_q, wl.n_heads_kv, wl.head_dim) == (32, 8, 128)
        lens = wl.seq_lens[:-1]
        assert np.all(((64 <= lens) & (lens <= 512)) | ((2048 <= lens) & (lens <= 4096)))
    if cfg == 3:
        assert T <= 16384 and wl.n_seqs == 4
    if cfg == 4:
        assert T == 16384 and not wl.causal
    if cfg == 5:
        assert T == 131072 and wl.seq_lens[0] == 65536 and wl.force_int64


def test_generator_is_seeded():
    a = gen.make_workload(2, seed=3)
    b = gen.make_workload(2, seed=3)
    assert np.array_equal(a.cu_seqlens, b.cu_seqlens)
    assert np.array_equal(a.q_bits, b.q_bits) and np.array_equal(a.v_bits, b.v_bits)


def test_bf16_rounding():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 3.0e38], dtype=np.float32)
    back = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(x))
    assert back[0] == 1.0
    assert back[1] == 1.0            # tie -> even
    assert back[2] == 1.0 + 2 ** -7  # above the tie -> up
    assert back[3] == -2.5


# ----------------------------------------------------------------------------
# mask recipes against brute-force predicates written from the workload text
# (PaddleNLP FlashMask article, sections 5.1-5.2: the mask types)
# ----------------------------------------------------------------------------

from oracle import mask as om  # noqa: E402


def _segment_masks(wl, seg):
    """(masked, rows, cols) of segment ``seg`` from the recipe's intervals,
    through the oracle's dense-mask builder."""
    a, b = int(wl.cu_seqlens[seg]), int(wl.cu_seqlens[seg + 1])
    idx = np.arange(a, b)
    return om.dense_mask(wl.startend_row_indices[0], idx, idx, wl.causal), idx


def _shared_question_visible(groups, i, j):
    """Row i sees key j iff both are in one group, j <= i, and j is in the
    group's question or i and j are in the same answer."""
    for g0, qlen, alens in groups:
        gend = g0 + qlen + sum(alens)
        if not (g0 <= i < gend and g0 <= j < gend) or j > i:
            continue
        if j < g0 + qlen:
            return True
        a0 = g0 + qlen
        for alen in alens:
            if a0 <= i < a0 + alen and a0 <= j < a0 + alen:
                return True
            a0 += alen
        return False
    return False


def test_shared_question_recipe_small_exhaustive():
    groups_spec = [(3, [2, 1, 4]), (1, [1]), (4, [3, 3])]
    groups, lens, g0 = [], [], 0
    for qlen, alens in groups_spec:
        groups.append((g0, qlen, alens))
        lens.append(qlen + sum(alens))
        g0 += lens[-1]
    T = g0
    sri = gen.shared_question_intervals(groups, T)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    for s in range(len(lens)):
        idx = np.arange(cu[s], cu[s + 1])
        masked = om.dense_mask(sri[0], idx, idx, True)
        want = np.array([[_shared_question_visible(groups, i, j) for j in idx] for i in idx])
        assert np.array_equal(~masked, want), s


def test_shared_question_workload_matches_its_text():
    """Workload 3 in full: 4 groups of one question U[512, 1536] and four
    answers U[256, 768], total <= 16384, one segment per group; every
    (row, key) pair of every group against the predicate."""
    wl = gen.make_workload(3, seed=0, tensors=False)
    assert len(wl.groups) == 4 and wl.total_tokens <= 16384
    for s, (g0, qlen, alens) in enumerate(wl.groups):
        assert 512 <= qlen <= 1536 and len(alens) == 4
        assert all(256 <= x <= 768 for x in alens)
        assert wl.cu_seqlens[s] == g0 and wl.cu_seqlens[s + 1] == g0 + qlen + sum(alens)
        masked, idx = _segment_masks(wl, s)
        i, j = idx[:, None], idx[None, :]
        vis = (j <= i) & (j < g0 + qlen)
        a0 = g0 + qlen
        for alen in alens:
            ina = (i >= a0) & (i < a0 + alen) & (j >= a0) & (j < a0 + alen)
            vis |= ina & (j <= i)
            a0 += alen
        assert np.array_equal(~masked, vis), s


def test_sliding_window_recipe_small_exhaustive():
    lens = [3, 10, 7, 1]
    W = 4
    wl = gen.make_custom(lens, mask="window", window=W, tensors=False)
    for s in range(len(lens)):
        masked, idx = _segment_masks(wl, s)
        i, j = idx[:, None], idx[None, :]
        assert np.array_equal(~masked, (i - j >= 0) & (i - j < W)), s


def test_long_context_window_workload_matches_its_text():
    """Workload 5: a 65536-token document first, then documents U[512, 8192]
    (the last one truncated), causal document mask intersected with a
    4096-key window (row i sees key j iff same document and
    0 <= i - j < 4096); checked on row slabs at every document start and end,
    across the window edge and at random places."""
    wl = gen.make_workload(5, seed=0, tensors=False)
    cu = wl.cu_seqlens.astype(np.int64)
    lens = np.diff(cu)
    assert lens[0] == 65536 and np.all((lens[1:-1] >= 512) & (lens[1:-1] <= 8192))
    assert 1 <= lens[-1] <= 8192 and cu[-1] == 131072
    rng = np.random.default_rng(0)
    sri = wl.startend_row_indices[0]
    for s in range(wl.n_seqs):
        a, b = int(cu[s]), int(cu[s + 1])
        starts = {a, max(a, b - 96), min(b - 1, a + 4096 - 40), int(rng.integers(a, b))}
        for r0 in starts:
            rows = np.arange(r0, min(r0 + 96, b))
            cols = np.arange(a, b)
            masked = om.dense_mask(sri, rows, cols, True)
            d = rows[:, None] - cols[None, :]
            assert np.array_equal(~masked, (d >= 0) & (d < 4096)), (s, r0)


def test_headline_causal_document_matches_its_text():
    wl = gen.make_workload(2, seed=0, tensors=False)
    for s in range(wl.n_seqs):
        masked, idx = _segment_masks(wl, s)
        assert np.array_equal(~masked, idx[:, None] >= idx[None, :]), s


def test_bidirectional_prefix_lm_workload_matches_its_text():
    """Workload 4 (non-causal): even documents fully bidirectional; odd
    documents prefix-LM, the first floor(len / 4) tokens visible to the whole
    document and later keys only to rows at or after them."""
    for alt in (False, True):
        wl = gen.make_workload(4, seed=0, tensors=False, alt_mask=alt)
        assert not wl.causal
        for s in range(wl.n_seqs):
            masked, idx = _segment_masks(wl, s)
            a, b = int(wl.cu_seqlens[s]), int(wl.cu_seqlens[s + 1])
            i, j = idx[:, None], idx[None, :]
            if s % 2 == 0:
                want = np.ones(masked.shape, dtype=bool)
            else:
                want = (j < a + (b - a) // 4) | (j <= i)
            assert np.array_equal(~masked, want), (alt, s)
