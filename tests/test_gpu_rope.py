"""GPU parity: fm_rope_qk_varlen against the float64 oracle."""

import numpy as np
import pytest

from helpers import (ROPE_MAX_ABS, bf16_tensor_to_f64, check_close_bf16, ensure_library,
                     to_device_bf16)
from oracle import rope as orope
from workloads import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    return ensure_library()


def _run(fm, wl, backward=False, force_int64=False):
    import torch
    q = to_device_bf16(wl.q_bits)
    k = to_device_bf16(wl.k_bits)
    cu = torch.from_numpy(wl.cu_seqlens).cuda()
    fm.rope_qk_varlen(q, k, cu, wl.theta, backward=backward, force_int64=force_int64)
    torch.cuda.synchronize()
    return q, k


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_rope_full_configs(fm, cfg):
    wl = gen.make_workload(cfg, seed=cfg)
    q, k = _run(fm, wl)
    for got, bits, what in ((q, wl.q_bits, "q"), (k, wl.k_bits, "k")):
        ref = orope.rope_apply(gen.bf16_bits_to_f64(bits), wl.cu_seqlens, wl.theta)
        check_close_bf16(bf16_tensor_to_f64(got), ref, ROPE_MAX_ABS, what=f"cfg{cfg} {what}")


def test_rope_long_context_full(fm):
    """131072 tokens, positions up to 65535, int64 path; every token, in
    chunks of 8192 tokens."""
    wl = gen.make_workload(5, seed=0)
    q, k = _run(fm, wl, force_int64=True)
    T = wl.total_tokens
    for t0 in range(0, T, 8192):
        toks = np.arange(t0, min(t0 + 8192, T))
        for got, bits, what in ((q, wl.q_bits, "q"), (k, wl.k_bits, "k")):
            ref = orope.rope_apply(gen.bf16_bits_to_f64(bits[toks]), wl.cu_seqlens, wl.theta,
                                   tokens=toks)
            check_close_bf16(bf16_tensor_to_f64(got[t0:t0 + len(toks)]), ref, ROPE_MAX_ABS,
                             what=f"cfg5 {what} tokens {t0}+")


def test_rope_backward_matches_oracle(fm):
    wl = gen.make_custom([1, 300, 17, 2000], n_heads_q=4, n_heads_kv=2, head_dim=128,
                         theta=5e5, seed=3)
    q, k = _run(fm, wl, backward=True)
    ref = orope.rope_apply(gen.bf16_bits_to_f64(wl.q_bits), wl.cu_seqlens, wl.theta,
                           backward=True)
    check_close_bf16(bf16_tensor_to_f64(q), ref, ROPE_MAX_ABS, what="backward q")


def test_rope_int64_path_bit_identical(fm):
    wl = gen.make_workload(2, seed=2)
    q32, k32 = _run(fm, wl)
    q64, k64 = _run(fm, wl, force_int64=True)
    import torch
    assert torch.equal(q32.view(torch.int16), q64.view(torch.int16))
    assert torch.equal(k32.view(torch.int16), k64.view(torch.int16))


def test_rope_fused_qkv_buffer_strides(fm):
    """q and k as views of one [T, Hq + 2 Hkv, D] buffer (token stride > heads * D)."""
    import torch
    wl = gen.make_custom([5, 64, 1, 130], n_heads_q=4, n_heads_kv=2, head_dim=64, seed=5)
    T = wl.total_tokens
    qkv = torch.zeros((T, 8, 64), dtype=torch.bfloat16, device="cuda")
    qkv[:, 0:4] = to_device_bf16(wl.q_bits)
    qkv[:, 4:6] = to_device_bf16(wl.k_bits)
    qkv[:, 6:8] = to_device_bf16(wl.v_bits)
    cu = torch.from_numpy(wl.cu_seqlens).cuda()
    fm.rope_qk_varlen(qkv[:, 0:4], qkv[:, 4:6], cu, wl.theta)
    torch.cuda.synchronize()
    ref_q = orope.rope_apply(gen.bf16_bits_to_f64(wl.q_bits), wl.cu_seqlens, wl.theta)
    ref_k = orope.rope_apply(gen.bf16_bits_to_f64(wl.k_bits), wl.cu_seqlens, wl.theta)
    check_close_bf16(bf16_tensor_to_f64(qkv[:, 0:4]), ref_q, ROPE_MAX_ABS, what="fused q")
    check_close_bf16(bf16_tensor_to_f64(qkv[:, 4:6]), ref_k, ROPE_MAX_ABS, what="fused k")
    # v untouched
    assert np.array_equal(qkv[:, 6:8].contiguous().view(torch.int16).cpu().numpy(),
                          wl.v_bits.view(np.int16))


def test_rope_position_zero_tokens_unchanged(fm):
    import torch
    wl = gen.make_custom([1] * 40, n_heads_q=2, n_heads_kv=1, head_dim=128, seed=1)
    q, k = _run(fm, wl)
    assert np.array_equal(q.view(torch.int16).cpu().numpy(), wl.q_bits.view(np.int16))
