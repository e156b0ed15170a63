"""GPU parity: fm_mask_block_minmax, bit-exact against the oracle."""

import numpy as np
import pytest

from helpers import ensure_library, kv_slot
from oracle import mask as om
from workloads import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    return ensure_library()


def _check(fm, wl, block_n):
    import torch
    sri = torch.from_numpy(wl.startend_row_indices).cuda()
    cu = torch.from_numpy(wl.cu_seqlens).cuda()
    out = fm.mask_block_minmax(sri, cu, block_n).cpu().numpy()
    ref = om.block_minmax(wl.startend_row_indices, wl.cu_seqlens, block_n)
    hm = wl.startend_row_indices.shape[0]
    n_slots = fm.num_kv_tiles_bound(wl.total_tokens, wl.n_seqs, block_n)
    assert out.shape == (hm, 8, n_slots)
    used = np.zeros(n_slots, dtype=bool)
    for (h, s, j), v in ref.items():
        slot = kv_slot(wl.cu_seqlens, s, j, block_n)
        used[slot] = True
        assert tuple(int(x) for x in out[h, :, slot]) == v, (h, s, j)
    # slots that hold no tile carry the neutral (max, min) pairs
    gaps = out[:, :, ~used]
    assert np.all(gaps[:, 0::2] == np.iinfo(np.int32).max)
    assert np.all(gaps[:, 1::2] == np.iinfo(np.int32).min)


def test_worked_example_tile_statistics(fm):
    """The FlashMask article's 16x16 table at the smallest supported tile."""
    from fixtures import load
    g = load("flashmask_16x16_causal.txt")
    sri = np.zeros((1, 4, 64), dtype=np.int32)
    sri[0, 1, :] = 64
    sri[0, 3, :] = 64
    sri[0, 0, :16] = g["LTS"]
    sri[0, 1, :16] = g["LTE"]
    sri[0, 0, 16:] = 64
    wl = gen.make_custom([64], tensors=False)
    wl.startend_row_indices = sri
    _check(fm, wl, 64)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("block_n", [64, 128])
def test_minmax_configs(fm, cfg, block_n):
    wl = gen.make_workload(cfg, seed=cfg, tensors=False)
    _check(fm, wl, block_n)


@pytest.mark.parametrize("seed", range(3))
def test_minmax_random_intervals_multihead(fm, seed):
    wl = gen.make_custom([0, 1, 63, 64, 65, 0, 300, 7], mask="random", n_mask_heads=3,
                         seed=seed, tensors=False)
    for bn in (64, 128):
        _check(fm, wl, bn)
