"""bench.py's interval-based count of unmasked pairs equals the oracle's
dense-mask count (the FLOP accounting of the reported metric)."""

import numpy as np
import pytest

import bench
from oracle import attention as oat
from workloads import gen


@pytest.mark.parametrize("mask,causal", [("none", True), ("none", False),
                                         ("causal_document", True), ("window", True),
                                         ("bidir_prefix", False), ("random", False),
                                         ("random", True)])
def test_unmasked_pairs_match_oracle(mask, causal):
    wl = gen.make_custom([1, 77, 0, 300, 64, 129], mask=mask, causal=causal, window=50, seed=3,
                         tensors=False)
    sri = wl.startend_row_indices
    got = bench.unmasked_pairs(wl.cu_seqlens, None if sri is None else sri[0], causal)
    assert got == oat.effective_pairs(wl.cu_seqlens, sri, causal)


@pytest.mark.parametrize("cfg", [1, 3])
def test_workload_pairs(cfg):
    wl = gen.make_workload(cfg, seed=0, tensors=False)
    sri = wl.startend_row_indices
    assert bench.unmasked_pairs(wl.cu_seqlens, sri[0], wl.causal) == \
        oat.effective_pairs(wl.cu_seqlens, sri, wl.causal)


def test_tiny_workload_flops():
    wl = gen.make_workload(1, seed=0, tensors=False)
    assert bench.effective_flops(wl) == 4 * 64 * 13440
