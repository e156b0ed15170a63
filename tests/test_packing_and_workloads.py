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
