"""GPU parity: fm_attn_bwd_varlen (after fm_attn_fwd_varlen) against the
float64 gradient oracle.

Tolerance (derived from the arithmetic, not fitted): every gradient element
is a sum of products in which one factor was rounded once to bfloat16 (P for
dv, dS for dq and dk; unit roundoff u = 2^-8), dS also carries the error of
delta = dout . out through the bf16 forward output (at most about 3u times
e_i = sum_d |dout_id| sum_j p_ij |v_jd|), and the result is rounded once to
bf16.  So |gpu - oracle| <= 4u * m + u * |oracle|, where m is the magnitude
sum the oracle returns alongside the gradients (the sum of the absolute
values of the terms, with the delta error folded in; a factor 2 of slack
over the 2u the roundings give).  Inputs with sharp scores (q and k scaled
so that a few keys dominate every row) make single terms matter, so a wrong
mask element or a dropped block cannot hide under that bound.
"""

import numpy as np
import pytest

from helpers import bf16_tensor_to_f64, ensure_library, to_device_bf16
import oracle_runs
from oracle import attention_bwd as ob
from workloads import gen

pytestmark = pytest.mark.gpu

U = 2.0 ** -8


@pytest.fixture(scope="module")
def fm():
    return ensure_library()


def _dout_bits(wl, seed):
    return oracle_runs.dout_bits(wl, seed)


def run_grad(fm, wl, do_bits, causal=None, force_int64=False, sri="default"):
    """Forward then backward on the GPU; returns (dq, dk, dv, out, lse) tensors."""
    import torch
    q, k, v, do = (to_device_bf16(b) for b in (wl.q_bits, wl.k_bits, wl.v_bits, do_bits))
    c = wl.causal if causal is None else causal
    sri_np = wl.startend_row_indices if isinstance(sri, str) else sri
    cu_t = torch.from_numpy(np.ascontiguousarray(wl.cu_seqlens)).cuda()
    sri_t = mm = None
    if sri_np is not None:
        sri_t = torch.from_numpy(np.ascontiguousarray(sri_np)).cuda()
        mm = fm.mask_block_minmax(sri_t, cu_t, 128)
    out, lse = fm.attn_fwd_varlen(q, k, v, cu_t, sri_t, mm, causal=c, force_int64=force_int64)
    ws = torch.empty(fm.attn_bwd_workspace_size(wl.total_tokens, wl.n_seqs, wl.n_heads_q),
                     dtype=torch.uint8, device="cuda")
    dq, dk, dv = fm.attn_bwd_varlen(q, k, v, out, do, lse, cu_t, sri_t, mm, causal=c,
                                    workspace=ws, force_int64=force_int64)
    torch.cuda.synchronize()
    err = fm.get_device_error(ws)
    assert err == 0, f"device error {err}, first expired wait {fm.get_device_timeout_info(ws)}"
    return dq, dk, dv, out, lse


def oracle_grad(wl, do_bits, causal=None, kv_heads=None, sri="default"):
    """Oracle gradients and magnitude sums at full head positions; with
    ``kv_heads`` only those key/value heads and their q heads are evaluated
    (the rest stays NaN)."""
    f64 = gen.bf16_bits_to_f64
    c = wl.causal if causal is None else causal
    sri_np = wl.startend_row_indices if isinstance(sri, str) else sri
    grp = wl.n_heads_q // wl.n_heads_kv
    if kv_heads is None:
        kv_heads = list(range(wl.n_heads_kv))
    T, D = wl.total_tokens, wl.head_dim
    full = [np.full((T, h, D), np.nan) for h in (wl.n_heads_q, wl.n_heads_kv, wl.n_heads_kv)]
    mags = [np.full((T, h, D), np.nan) for h in (wl.n_heads_q, wl.n_heads_kv, wl.n_heads_kv)]
    for g in kv_heads:
        hs = list(range(g * grp, (g + 1) * grp))
        s = sri_np
        if s is not None and s.shape[0] > 1:
            s = s[hs]
        dq, dk, dv, mq, mk, mv = ob.attention_backward(
            f64(wl.q_bits[:, hs]), f64(wl.k_bits[:, [g]]), f64(wl.v_bits[:, [g]]),
            f64(do_bits[:, hs]), wl.cu_seqlens, s, c, magnitudes=True)
        full[0][:, hs], full[1][:, [g]], full[2][:, [g]] = dq, dk, dv
        mags[0][:, hs], mags[1][:, [g]], mags[2][:, [g]] = mq, mk, mv
    return full, mags


def check_grad(got, ref, mag, what, rows=None, heads=None):
    g = bf16_tensor_to_f64(got)
    if rows is not None:
        g, ref, mag = g[rows], ref[rows], mag[rows]
    if heads is not None:
        g, ref, mag = g[:, heads], ref[:, heads], mag[:, heads]
    assert np.all(np.isfinite(g)), f"{what}: non-finite gradient"
    err = np.abs(g - ref)
    bound = 4 * U * mag + U * np.abs(ref) + 1e-30
    ratio = err / bound
    if (ratio > 1).any():
        i = np.unravel_index(np.argmax(ratio), ratio.shape)
        raise AssertionError(f"{what}: {int((ratio > 1).sum())} elements over bound; worst at {i}: "
                             f"got {g[i]} ref {ref[i]} err {err[i]:.3e} bound {bound[i]:.3e}")
    return float(ratio.max())


def check_all(fm_out, ref, mags, what, rows=None, heads_q=None, heads_kv=None):
    dq, dk, dv = fm_out[:3]
    r = [check_grad(dq, ref[0], mags[0], what + " dq", rows, heads_q),
         check_grad(dk, ref[1], mags[1], what + " dk", rows, heads_kv),
         check_grad(dv, ref[2], mags[2], what + " dv", rows, heads_kv)]
    print(f"{what}: max err / bound (dq, dk, dv) = {r[0]:.3f} {r[1]:.3f} {r[2]:.3f}")
    return r


LENS = [1, 77, 128, 300, 5, 513, 0, 260, 64]


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("mask,causal", [("none", True), ("none", False),
                                         ("causal_document", True), ("window", True),
                                         ("bidir_prefix", False)])
def test_small_mask_shapes(fm, head_dim, mask, causal):
    wl = gen.make_custom(LENS, n_heads_q=4, n_heads_kv=2, head_dim=head_dim, mask=mask,
                         causal=causal, window=100, seed=7)
    do = _dout_bits(wl, 0)
    ref, mags = oracle_grad(wl, do)
    check_all(run_grad(fm, wl, do), ref, mags, f"{mask} D{head_dim}")


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("per_head", [False, True])
def test_random_intervals(fm, seed, causal, per_head):
    """Arbitrary column intervals: many partial blocks, fully masked rows."""
    wl = gen.make_custom([3, 200, 129, 0, 64, 400], n_heads_q=4, n_heads_kv=1, head_dim=128,
                         mask="random", causal=causal, seed=seed,
                         n_mask_heads=4 if per_head else 1)
    do = _dout_bits(wl, seed)
    ref, mags = oracle_grad(wl, do)
    check_all(run_grad(fm, wl, do), ref, mags, "random")


def _sharpen(wl, factor):
    """q and k scaled (rounded back to bf16): each row's softmax is dominated
    by a few keys, so every masked or unmasked element matters."""
    f = gen.bf16_bits_to_f32
    wl.q_bits = gen.f32_to_bf16_bits(f(wl.q_bits) * factor)
    wl.k_bits = gen.f32_to_bf16_bits(f(wl.k_bits) * factor)
    return wl


@pytest.mark.parametrize("mask,causal,per_head", [("causal_document", True, False),
                                                  ("window", True, False),
                                                  ("bidir_prefix", False, False),
                                                  ("random", True, True),
                                                  ("random", False, False)])
def test_sharp_scores(fm, mask, causal, per_head):
    wl = gen.make_custom([150, 257, 64, 333], n_heads_q=4, n_heads_kv=2, head_dim=128, mask=mask,
                         causal=causal, window=70, seed=11, n_mask_heads=4 if per_head else 1)
    wl = _sharpen(wl, 3.0)
    do = _dout_bits(wl, 5)
    ref, mags = oracle_grad(wl, do)
    check_all(run_grad(fm, wl, do), ref, mags, f"sharp {mask}")


def test_every_row_masked(fm):
    """Every element masked: lse = -inf everywhere and all gradients are 0."""
    import torch
    wl = gen.make_custom([300, 200], n_heads_q=2, n_heads_kv=1, head_dim=128, mask="none",
                         causal=True, seed=3)
    T = wl.total_tokens
    sri = np.zeros((1, 4, T), dtype=np.int32)
    sri[0, 1, :] = T   # lower triangle (with the diagonal) masked for every row
    do = _dout_bits(wl, 1)
    dq, dk, dv, _, lse = run_grad(fm, wl, do, sri=sri)
    assert torch.isneginf(lse).all()
    for t in (dq, dk, dv):
        assert not t.float().abs().sum().item()


def test_bitwise_reproducible(fm):
    import torch
    wl = gen.make_custom([700, 129, 1000], n_heads_q=8, n_heads_kv=2, head_dim=128,
                         mask="causal_document", causal=True, seed=2)
    do = _dout_bits(wl, 2)
    a = run_grad(fm, wl, do)
    b = run_grad(fm, wl, do)
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_int64_path_bit_identical(fm):
    import torch
    wl = gen.make_custom([333, 64, 517], n_heads_q=4, n_heads_kv=2, head_dim=128,
                         mask="window", causal=True, window=90, seed=4)
    do = _dout_bits(wl, 3)
    a = run_grad(fm, wl, do)
    b = run_grad(fm, wl, do, force_int64=True)
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_full_size_configs(fm, cfg):
    """The full-size workloads in the launch configuration the benchmark
    times: every row of every q and key/value head against the oracle."""
    wl = gen.make_workload(cfg, seed=0)
    do = _dout_bits(wl, cfg)
    got = run_grad(fm, wl, do)
    ref, mags = oracle_runs.backward_full(cfg, 0, cfg)
    check_all(got, ref, mags, f"cfg{cfg}")


def test_unsupported_arguments_raise(fm):
    import torch
    q = torch.zeros((10, 2, 96), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((10, 1, 96), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((2, 10), dtype=torch.float32, device="cuda")
    cu = torch.tensor([0, 10], dtype=torch.int32, device="cuda")
    with pytest.raises(fm.FMError):
        fm.attn_bwd_varlen(q, k, k, q, q, lse, cu)
