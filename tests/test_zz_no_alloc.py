"""The allocation-free attention entry point (fm_attn_fwd_varlen_noalloc).

It serves callers that cannot allocate device memory: a plugin handed only
its input and output buffers, code whose device memory belongs to a
framework's caching allocator, latency-critical paths that must not call
cudaMalloc.  Its scheduler scratch is a fixed device array inside the
library, shared by all calls.  This file is collected last on purpose.

The entry point runs the same kernels as fm_attn_fwd_varlen on the same
inputs, so its outputs must be bit-identical to that call's; they are also
checked against the float64 oracle.  Calls of different sizes follow each
other so that state a larger call leaves in the shared array (header, work
list entries past the smaller call's end) is shown to be harmless.
"""

import numpy as np
import pytest

from helpers import (ATTN_MAX_ABS, ATTN_MEAN_ABS, abs_v_magnitude, bf16_tensor_to_f64,
                     check_close_bf16, check_lse, ensure_library, to_device_bf16, workload_inputs)
import oracle_runs
from oracle import attention as oat
from workloads import gen

FM_ERR_INVALID_ARG, FM_ERR_WORKSPACE, FM_ERR_CUDA = 1, 4, 5
FM_DEVERR_DATA = 2


def _inputs(wl):
    import torch
    q, k, v = (to_device_bf16(b) for b in (wl.q_bits, wl.k_bits, wl.v_bits))
    cu = torch.from_numpy(wl.cu_seqlens).cuda()
    sri = None
    if wl.startend_row_indices is not None:
        sri = torch.from_numpy(wl.startend_row_indices).cuda()
    return q, k, v, cu, sri


def _bits(t):
    import torch
    return t.contiguous().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def _run_pair(fm, wl, causal, ref, sri_np="default"):
    """Workspace entry point, then the allocation-free one into buffers
    poisoned with 7.0: identical bits, identical block counts, and both
    within tolerance of the oracle result ``ref``."""
    import torch
    q, k, v, cu, sri = _inputs(wl)
    mm = None if sri is None else fm.mask_block_minmax(sri, cu, wl.block_n)
    ref_counts = torch.zeros(3, dtype=torch.int64, device="cuda")
    ws_out, ws_lse = fm.attn_fwd_varlen(q, k, v, cu, sri, mm, causal=causal,
                                        class_counts=ref_counts)
    out = torch.full_like(q, 7.0)
    lse = torch.full_like(ws_lse, 7.0)
    counts = torch.zeros(3, dtype=torch.int64, device="cuda")
    fm.attn_fwd_varlen_noalloc(q, k, v, cu, sri, mm, causal=causal, out=out, lse=lse,
                               class_counts=counts)
    torch.cuda.synchronize()
    assert fm.get_device_error(None) == 0
    assert torch.equal(_bits(out), _bits(ws_out)), "out differs from the workspace entry point"
    assert torch.equal(_bits(lse), _bits(ws_lse)), "lse differs from the workspace entry point"
    assert counts.cpu().tolist() == ref_counts.cpu().tolist()
    sri_np = wl.startend_row_indices if isinstance(sri_np, str) else sri_np
    mag = abs_v_magnitude(workload_inputs(wl), wl.cu_seqlens, sri_np, causal)
    check_close_bf16(bf16_tensor_to_f64(out), ref[0], ATTN_MAX_ABS, ATTN_MEAN_ABS,
                     what="noalloc out", magnitude=mag)
    check_lse(lse.cpu().numpy().astype(np.float64), ref[1], what="noalloc lse")


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_and_oracle():
    """Two workloads of different sizes in a row, then the first again: every
    call bit-identical to the workspace entry point and within tolerance of
    the oracle."""
    fm = ensure_library()
    for cfg in (3, 2, 3):
        wl = gen.make_workload(cfg, seed=0)
        _run_pair(fm, wl, wl.causal, oracle_runs.forward_full(cfg, 0))


@pytest.mark.gpu
def test_noalloc_causal_without_intervals():
    """No interval mask (startend_row_indices = None), causal within each
    sample, on small packed samples with ragged tails."""
    import dataclasses
    fm = ensure_library()
    wl = gen.make_custom([1, 200, 129, 0, 700, 64], n_heads_q=4, n_heads_kv=2, head_dim=128,
                         mask="none", causal=True, seed=9)
    ref = oat.attention_forward(gen.bf16_bits_to_f64(wl.q_bits), gen.bf16_bits_to_f64(wl.k_bits),
                                gen.bf16_bits_to_f64(wl.v_bits), wl.cu_seqlens, None, True)
    _run_pair(fm, dataclasses.replace(wl, startend_row_indices=None), True, ref)


@pytest.mark.gpu
def test_noalloc_reports_malformed_cu_seqlens():
    """cu_seqlens whose entries lie in [0, T] but do not end at T: every index
    stays in bounds (the kernels clamp), the device error word read through
    workspace = NULL says FM_DEVERR_DATA, and the next clean call reads 0."""
    import torch
    fm = ensure_library()
    wl = gen.make_custom([300, 500, 200], n_heads_q=2, n_heads_kv=1, head_dim=128,
                         mask="none", causal=True, seed=3)
    q, k, v, _, _ = _inputs(wl)
    bad = torch.tensor([0, 300, 800], dtype=torch.int32, device="cuda")   # T = 1000
    out = torch.zeros_like(q)
    lse = torch.zeros((2, wl.total_tokens), dtype=torch.float32, device="cuda")
    fm.attn_fwd_varlen_noalloc(q, k, v, bad, causal=True, out=out, lse=lse)
    torch.cuda.synchronize()
    assert fm.get_device_error(None) & FM_DEVERR_DATA
    assert bool(torch.isfinite(out.float()).all())
    good = torch.from_numpy(wl.cu_seqlens).cuda()
    fm.attn_fwd_varlen_noalloc(q, k, v, good, causal=True, out=out, lse=lse)
    torch.cuda.synchronize()
    assert fm.get_device_error(None) == 0


@pytest.mark.gpu
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
    assert rc == FM_ERR_WORKSPACE


def test_noalloc_slot_limit_boundary_host_only():
    """floor(T / block_m) + n_seqs == 32768 passes the size check, 32769 does
    not.  q = NULL makes an accepted call fail validation before any launch
    (FM_ERR_INVALID_ARG, or FM_ERR_CUDA where no device exists), so this runs
    with or without a GPU and never launches a kernel."""
    fm = ensure_library()
    lib = fm._lib()
    cases = [  # T, n_seqs, block_m, refused for size
        (32767 * 128, 1, 128, False),
        (32767 * 128 + 127, 1, 128, False),
        (32766 * 64, 2, 64, False),
        (32768 * 128, 1, 128, True),
        (32766 * 128, 3, 128, True),
    ]
    for T, n_seqs, bm, refused in cases:
        rc = lib.fm_attn_fwd_varlen_noalloc(None, None, None, T, 1, 1, 128, None, n_seqs, None, 0,
                                            None, 1, 0.0, bm, 128, None, None, None, 0, None)
        if refused:
            assert rc == FM_ERR_WORKSPACE, (T, n_seqs, bm, rc)
        else:
            assert rc in (FM_ERR_INVALID_ARG, FM_ERR_CUDA), (T, n_seqs, bm, rc)
