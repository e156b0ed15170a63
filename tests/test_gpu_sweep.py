"""GPU: the sparsity-sweep masks (one segment, structure only in the column
intervals) on a 2048-token segment.

Block-class counts must equal the oracle's exactly and the attention output
must match the float64 oracle on sampled rows (FlashMask article, sections
3.2 and 4.3).
"""

import numpy as np
import pytest

from helpers import (ATTN_MAX_ABS, ATTN_MEAN_ABS, abs_v_magnitude, bf16_tensor_to_f64,
                     check_close_bf16, check_lse, ensure_library)
from oracle import attention as oat
from oracle import mask as om
from workloads import gen

pytestmark = pytest.mark.gpu

T, HQ, HKV, D = 2048, 4, 2, 128
POINTS = gen.sparsity_sweep(T)


@pytest.fixture(scope="module")
def fm():
    return ensure_library()


@pytest.fixture(scope="module")
def tensors():
    rng = np.random.default_rng(3)
    return tuple(gen.f32_to_bf16_bits(rng.standard_normal((T, h, D)).astype(np.float32))
                 for h in (HQ, HKV, HKV))


@pytest.mark.parametrize("idx", range(len(POINTS)))
def test_sweep_point(fm, tensors, idx):
    import torch
    family, param, causal, sri = POINTS[idx]
    dt = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()
    q, k, v = (dt(b) for b in tensors)
    cu = np.array([0, T], dtype=np.int32)
    cu_t = torch.from_numpy(cu).cuda()
    sri_t = torch.from_numpy(sri).cuda()
    mm = fm.mask_block_minmax(sri_t, cu_t, 128)
    counts = torch.zeros(3, dtype=torch.int64, device="cuda")
    ws = torch.empty(fm.attn_fwd_workspace_size(T, 1, HQ, 128), dtype=torch.uint8, device="cuda")
    out, lse = fm.attn_fwd_varlen(q, k, v, cu_t, sri_t, mm, causal=causal, class_counts=counts,
                                  workspace=ws)
    torch.cuda.synchronize()
    assert fm.get_device_error(ws) == 0
    assert counts.cpu().tolist() == list(om.block_class_counts(cu, sri, HQ, 128, 128, causal))
    rows = np.unique(np.concatenate([np.arange(0, 130), np.arange(T - 130, T),
                                     np.random.default_rng(idx).integers(0, T, 200)]))
    f64 = gen.bf16_bits_to_f64
    ro, rl = oat.attention_forward(f64(tensors[0]), f64(tensors[1]), f64(tensors[2]), cu, sri,
                                   causal, rows=rows)
    mag = abs_v_magnitude(lambda: tuple(f64(t) for t in tensors), cu, sri, causal, rows=rows)
    check_close_bf16(bf16_tensor_to_f64(out)[rows], ro[rows], ATTN_MAX_ABS, ATTN_MEAN_ABS,
                     what=f"{family} {param}", magnitude=mag)
    check_lse(lse.cpu().numpy().astype(np.float64)[:, rows], rl[:, rows], what=f"{family} {param}")
