"""GPU parity: fm_attn_fwd_varlen_rope (QK RoPE fused into the attention
prologue) against the unfused path and against the float64 oracle.

* Bitwise: the fused call must give exactly the bits of fm_rope_qk_varlen
  followed by fm_attn_fwd_varlen on the same inputs -- out, lse, the block
  counts, the keys rotated in place and (with q_rot) the rotated queries --
  while q itself stays unchanged.
* Oracle: out / lse within the attention tolerances of the float64 oracle
  applied to RoPE(q), RoPE(k) stored as bfloat16 (the rotated tensors the
  attention consumes are bfloat16 in both paths).
"""

import numpy as np
import pytest

from helpers import (ATTN_MAX_ABS, ATTN_MEAN_ABS, abs_v_magnitude, bf16_tensor_to_f64,
                     check_close_bf16, check_lse, ensure_library, to_device_bf16, workload_inputs)
import oracle_runs
from oracle import attention as oat
from oracle import rope as orope
from workloads import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    return ensure_library()


def _inputs(fm, wl, block_n):
    import torch
    q, k, v = (to_device_bf16(b) for b in (wl.q_bits, wl.k_bits, wl.v_bits))
    cu = torch.from_numpy(np.ascontiguousarray(wl.cu_seqlens)).cuda()
    sri = mm = None
    if wl.startend_row_indices is not None:
        sri = torch.from_numpy(np.ascontiguousarray(wl.startend_row_indices)).cuda()
        mm = fm.mask_block_minmax(sri, cu, block_n)
    return q, k, v, cu, sri, mm


def run_unfused(fm, wl, block_m, block_n, causal, force_int64=False):
    import torch
    q, k, v, cu, sri, mm = _inputs(fm, wl, block_n)
    fm.rope_qk_varlen(q, k, cu, wl.theta, force_int64=force_int64)
    counts = torch.zeros(3, dtype=torch.int64, device="cuda")
    out, lse = fm.attn_fwd_varlen(q, k, v, cu, sri, mm, causal=causal, block_m=block_m,
                                  block_n=block_n, class_counts=counts, force_int64=force_int64)
    torch.cuda.synchronize()
    return dict(out=out, lse=lse, counts=counts, q=q, k=k)


def run_fused(fm, wl, block_m, block_n, causal, q_rot="separate", force_int64=False):
    import torch
    q, k, v, cu, sri, mm = _inputs(fm, wl, block_n)
    q_in = q.clone()
    qr = None
    if q_rot == "separate":
        qr = torch.full_like(q, float("nan"))
    elif q_rot == "in_place":
        qr = q
    counts = torch.zeros(3, dtype=torch.int64, device="cuda")
    ws = torch.empty(fm.attn_fwd_workspace_size(wl.total_tokens, wl.n_seqs, wl.n_heads_q, block_m),
                     dtype=torch.uint8, device="cuda")
    out, lse = fm.attn_fwd_varlen_rope(q, k, v, cu, wl.theta, sri, mm, causal=causal,
                                       block_m=block_m, block_n=block_n, q_rot=qr,
                                       class_counts=counts, workspace=ws, force_int64=force_int64)
    torch.cuda.synchronize()
    assert fm.get_device_error(ws) == 0
    return dict(out=out, lse=lse, counts=counts, q=q, q_in=q_in, k=k, q_rot=qr)


def _bits(t):
    import torch
    return t.contiguous().view(torch.int16)


def assert_bitwise(fm, wl, block_m, block_n, causal, q_rot="separate", force_int64=False):
    import torch
    a = run_unfused(fm, wl, block_m, block_n, causal, force_int64)
    b = run_fused(fm, wl, block_m, block_n, causal, q_rot, force_int64)
    assert torch.equal(_bits(a["out"]), _bits(b["out"])), "out differs from the unfused path"
    assert torch.equal(a["lse"].view(torch.int32), b["lse"].view(torch.int32)), "lse differs"
    assert a["counts"].tolist() == b["counts"].tolist()
    assert torch.equal(_bits(a["k"]), _bits(b["k"])), "keys rotated in place differ"
    if q_rot == "separate":
        assert torch.equal(_bits(b["q"]), _bits(b["q_in"])), "q was modified"
        assert torch.equal(_bits(a["q"]), _bits(b["q_rot"])), "q_rot differs from RoPE(q)"
    elif q_rot == "in_place":
        assert torch.equal(_bits(a["q"]), _bits(b["q"])), "q rotated in place differs"
    else:
        assert torch.equal(_bits(b["q"]), _bits(b["q_in"])), "q was modified"
    return b


LENS = [1, 77, 128, 300, 5, 513, 0, 260, 64]


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("blocks", [(128, 128), (64, 64), (128, 64), (64, 128)])
@pytest.mark.parametrize("mask,causal", [("causal_document", True), ("none", False),
                                         ("window", True), ("bidir_prefix", False)])
def test_fused_equals_unfused_small(fm, head_dim, blocks, mask, causal):
    wl = gen.make_custom(LENS, n_heads_q=4, n_heads_kv=2, head_dim=head_dim, mask=mask,
                         causal=causal, window=100, seed=17, theta=1.0e4)
    assert_bitwise(fm, wl, blocks[0], blocks[1], causal)


@pytest.mark.parametrize("q_rot", ["separate", "in_place", None])
@pytest.mark.parametrize("blocks", [(128, 128), (64, 64)])
def test_fused_q_rot_modes(fm, q_rot, blocks):
    wl = gen.make_custom([700, 33, 1500, 129], n_heads_q=8, n_heads_kv=2, head_dim=128,
                         mask="causal_document", seed=5, theta=5.0e5)
    assert_bitwise(fm, wl, blocks[0], blocks[1], True, q_rot=q_rot)


def test_fused_rows_with_no_visible_key(fm):
    """Items whose blocks are all fully masked never load their Q tile: their
    rotated queries are written from q directly."""
    import dataclasses
    wl = gen.make_custom([50, 200, 300], n_heads_q=2, n_heads_kv=2, head_dim=64, mask="none",
                         causal=True, seed=2, theta=1.0e4)
    T = wl.total_tokens
    sri = np.zeros((1, 4, T), dtype=np.int32)
    sri[0, 1] = T
    sri[0, 3] = T
    sri[0, 0, 250:] = 550  # the last sample keeps its causal lower triangle
    sri[0, 1, 250:] = 550
    wl = dataclasses.replace(wl, startend_row_indices=sri)
    b = assert_bitwise(fm, wl, 128, 128, True)
    assert float(b["out"][:250].abs().max()) == 0.0


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_fused_equals_unfused_workloads(fm, cfg):
    wl = gen.make_workload(cfg, seed=0)
    assert_bitwise(fm, wl, wl.block_m, wl.block_n, wl.causal, force_int64=wl.force_int64)


def test_fused_int64_path_bit_identical(fm):
    import torch
    wl = gen.make_workload(2, seed=1)
    a = run_fused(fm, wl, 128, 128, True, force_int64=False)
    b = run_fused(fm, wl, 128, 128, True, force_int64=True)
    for key in ("out", "k", "q_rot"):
        assert torch.equal(_bits(a[key]), _bits(b[key])), key
    assert torch.equal(a["lse"], b["lse"])


# --------------------------------------------------------------------------
# against the oracle
# --------------------------------------------------------------------------

def _rope_bf16(bits, cu, theta):
    """Oracle RoPE of generator inputs, stored as bfloat16 (test-side format
    conversion of the oracle's float64 result)."""
    y = orope.rope_apply(gen.bf16_bits_to_f64(bits), cu, theta)
    return gen.bf16_bits_to_f64(gen.f32_to_bf16_bits(y.astype(np.float32)))


def oracle_fused(wl, rows=None, heads=None):
    q = _rope_bf16(wl.q_bits, wl.cu_seqlens, wl.theta)
    k = _rope_bf16(wl.k_bits, wl.cu_seqlens, wl.theta)
    v = gen.bf16_bits_to_f64(wl.v_bits)
    if heads is None:
        return oat.attention_forward(q, k, v, wl.cu_seqlens, wl.startend_row_indices, wl.causal,
                                     rows=rows)
    group = wl.n_heads_q // wl.n_heads_kv
    kvh = [h // group for h in heads]
    o, l_ = oat.attention_forward(q[:, heads], k[:, kvh], v[:, kvh], wl.cu_seqlens,
                                  wl.startend_row_indices, wl.causal, rows=rows)
    T = wl.total_tokens
    out = np.full((T, wl.n_heads_q, wl.head_dim), np.nan)
    lse = np.full((wl.n_heads_q, T), np.nan)
    out[:, heads] = o
    lse[heads] = l_
    return out, lse


def _compare(b, ref, rows=None, heads=None, what="", wl=None):
    mag = None
    if wl is not None:
        mag = abs_v_magnitude(workload_inputs(wl, rope=True), wl.cu_seqlens,
                              wl.startend_row_indices, wl.causal, rows, heads)
    o = bf16_tensor_to_f64(b["out"])
    l_ = b["lse"].cpu().numpy().astype(np.float64)
    ro, rl = ref
    if rows is not None:
        o, ro, l_, rl = o[rows], ro[rows], l_[:, rows], rl[:, rows]
    if heads is not None:
        o, ro, l_, rl = o[:, heads], ro[:, heads], l_[heads], rl[heads]
    check_close_bf16(o, ro, ATTN_MAX_ABS, ATTN_MEAN_ABS, what=what + " out", magnitude=mag)
    check_lse(l_, rl, what=what + " lse")


def test_fused_tiny_against_oracle(fm):
    wl = gen.make_workload(1, seed=0)
    b = run_fused(fm, wl, wl.block_m, wl.block_n, wl.causal)
    _compare(b, oracle_fused(wl), what="cfg1 fused", wl=wl)
    assert b["counts"].tolist() == [2, 5, 2]


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("mask,causal", [("causal_document", True), ("bidir_prefix", False)])
def test_fused_small_against_oracle(fm, head_dim, mask, causal):
    wl = gen.make_custom(LENS, n_heads_q=4, n_heads_kv=2, head_dim=head_dim, mask=mask,
                         causal=causal, seed=23, theta=1.0e4)
    b = run_fused(fm, wl, 128, 128, causal)
    _compare(b, oracle_fused(wl), what=f"{mask} D{head_dim} fused", wl=wl)


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_fused_full_size_against_oracle(fm, cfg):
    """Workloads 2-4 in full (every row, every q head): the fused call
    against the oracle on RoPE(q), RoPE(k) stored as bfloat16."""
    wl = gen.make_workload(cfg, seed=0)
    b = run_fused(fm, wl, 128, 128, wl.causal)
    _compare(b, oracle_runs.forward_full(cfg, 0, rope=True), what=f"cfg{cfg} fused", wl=wl)


@pytest.mark.parametrize("seed", range(2))
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("per_head", [False, True])
@pytest.mark.parametrize("block_n", [128, 64])
def test_fused_equals_unfused_random_intervals(fm, seed, causal, per_head, block_n):
    """Arbitrary column intervals (many partially masked blocks, rows with no
    visible key), one mask shared by all heads or one mask per q head."""
    wl = gen.make_custom([3, 200, 129, 0, 64, 400], n_heads_q=4, n_heads_kv=1, head_dim=128,
                         mask="random", causal=causal, seed=seed, theta=1.0e4,
                         n_mask_heads=4 if per_head else 1)
    assert_bitwise(fm, wl, 128, block_n, causal)
