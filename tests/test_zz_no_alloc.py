"""The allocation-free attention entry point (fm_attn_fwd_varlen_noalloc).

It serves callers that cannot allocate device memory: a plugin handed only
its input and output buffers, code whose device memory belongs to a
framework's caching allocator, latency-critical paths that must not call
cudaMalloc.  Its scheduler scratch is a fixed device array inside the
library, shared by all calls.  This file is collected last on purpose.
"""

import numpy as np
import pytest

from helpers import (ATTN_MAX_ABS, ATTN_MEAN_ABS, bf16_tensor_to_f64, check_close_bf16, check_lse,
                     ensure_library, to_device_bf16)
from workloads import gen

pytestmark = pytest.mark.gpu


def _inputs(wl):
    import torch
    q, k, v = (to_device_bf16(b) for b in (wl.q_bits, wl.k_bits, wl.v_bits))
    cu = torch.from_numpy(wl.cu_seqlens).cuda()
    sri = torch.from_numpy(wl.startend_row_indices).cuda()
    return q, k, v, cu, sri


@pytest.mark.parametrize("cfg", [2, 3])
def test_noalloc_matches_workspace_entry_twice(cfg):
    import torch
    fm = ensure_library()
    wl = gen.make_workload(cfg, seed=0)
    q, k, v, cu, sri = _inputs(wl)
    mm = fm.mask_block_minmax(sri, cu, wl.block_n)
    ref_counts = torch.zeros(3, dtype=torch.int64, device="cuda")
    ref_out, ref_lse = fm.attn_fwd_varlen(q, k, v, cu, sri, mm, causal=wl.causal,
                                          class_counts=ref_counts)
    torch.cuda.synchronize()
    ref_o = bf16_tensor_to_f64(ref_out)
    ref_l = ref_lse.cpu().numpy().astype(np.float64)
    out = torch.empty_like(q)
    lse = torch.empty_like(ref_lse)
    for _ in range(2):   # the second call reuses the array the first one left behind
        out.fill_(7.0)
        lse.fill_(7.0)
        counts = torch.zeros(3, dtype=torch.int64, device="cuda")
        fm.attn_fwd_varlen_noalloc(q, k, v, cu, sri, mm, causal=wl.causal, out=out, lse=lse,
                                   class_counts=counts)
        torch.cuda.synchronize()
        check_close_bf16(bf16_tensor_to_f64(out), ref_o, ATTN_MAX_ABS, ATTN_MEAN_ABS,
                         what="noalloc out")
        check_lse(lse.cpu().numpy().astype(np.float64), ref_l, what="noalloc lse")
        assert counts.cpu().tolist() == ref_counts.cpu().tolist()


def test_noalloc_rejects_sizes_over_its_limit():
    import torch
    fm = ensure_library()
    q = torch.zeros((8, 1, 128), dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 8], dtype=torch.int32, device="cuda")
    lib = fm._lib()
    # 32768 * 128 tokens + 1 sample = 32769 Q-tile slots > 32768: refused before any launch
    rc = lib.fm_attn_fwd_varlen_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), 32768 * 128, 1,
                                        1, 128, cu.data_ptr(), 1, None, 0, None, 1, 0.0, 128,
                                        128, q.data_ptr(), q.data_ptr(), None, 0, None)
    assert rc == 4   # FM_ERR_WORKSPACE
