"""GPU parity: fm_attn_fwd_varlen against the float64 oracle.

Outputs are compared element by element (|gpu - oracle| <= max(1e-2, one
bf16 ulp of the oracle value), mean <= 1e-3; lse <= 1e-3 with identical -inf
rows); block-class counts must be identical.
"""

import numpy as np
import pytest

from helpers import (ATTN_MAX_ABS, ATTN_MEAN_ABS, bf16_tensor_to_f64, check_close_bf16, check_lse,
                     ensure_library, to_device_bf16)
from oracle import attention as oat
from oracle import mask as om
from workloads import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    return ensure_library()


def run_attn(fm, wl, block_m=None, block_n=None, causal=None, force_int64=None, cu=None,
             sri="default"):
    import torch
    q, k, v = (to_device_bf16(b) for b in (wl.q_bits, wl.k_bits, wl.v_bits))
    cu_np = wl.cu_seqlens if cu is None else cu
    sri_np = wl.startend_row_indices if isinstance(sri, str) else sri
    bm = wl.block_m if block_m is None else block_m
    bn = wl.block_n if block_n is None else block_n
    c = wl.causal if causal is None else causal
    f64 = wl.force_int64 if force_int64 is None else force_int64
    cu_t = torch.from_numpy(np.ascontiguousarray(cu_np)).cuda()
    sri_t = mm = None
    if sri_np is not None:
        sri_t = torch.from_numpy(np.ascontiguousarray(sri_np)).cuda()
        mm = fm.mask_block_minmax(sri_t, cu_t, bn)
    counts = torch.zeros(3, dtype=torch.int64, device="cuda")
    T, hq = wl.total_tokens, wl.n_heads_q
    ws = torch.empty(fm.attn_fwd_workspace_size(T, len(cu_np) - 1, hq, bm), dtype=torch.uint8,
                     device="cuda")
    out, lse = fm.attn_fwd_varlen(q, k, v, cu_t, sri_t, mm, causal=c, block_m=bm, block_n=bn,
                                  class_counts=counts, workspace=ws, force_int64=f64)
    torch.cuda.synchronize()
    assert fm.get_device_error(ws) == 0
    return out, lse, counts.cpu().tolist(), ws


def oracle(wl, rows=None, heads=None, causal=None, cu=None, sri="default"):
    """Oracle outputs; with ``heads`` only those q heads are evaluated (their
    key/value heads gathered next to them), returned at full head positions."""
    cu_np = wl.cu_seqlens if cu is None else cu
    sri_np = wl.startend_row_indices if isinstance(sri, str) else sri
    c = wl.causal if causal is None else causal
    if heads is None:
        return oat.attention_forward(gen.bf16_bits_to_f64(wl.q_bits),
                                     gen.bf16_bits_to_f64(wl.k_bits),
                                     gen.bf16_bits_to_f64(wl.v_bits), cu_np, sri_np, c, rows=rows)
    group = wl.n_heads_q // wl.n_heads_kv
    kvh = [h // group for h in heads]
    assert sri_np is None or sri_np.shape[0] == 1
    o, l_ = oat.attention_forward(gen.bf16_bits_to_f64(wl.q_bits[:, heads]),
                                  gen.bf16_bits_to_f64(wl.k_bits[:, kvh]),
                                  gen.bf16_bits_to_f64(wl.v_bits[:, kvh]), cu_np, sri_np, c,
                                  rows=rows)
    T = wl.total_tokens
    out = np.full((T, wl.n_heads_q, wl.head_dim), np.nan)
    lse = np.full((wl.n_heads_q, T), np.nan)
    out[:, heads] = o
    lse[heads] = l_
    return out, lse


def compare(out, lse, ref, rows=None, heads=None, what=""):
    o = bf16_tensor_to_f64(out)
    l_ = lse.cpu().numpy().astype(np.float64)
    ro, rl = ref
    if rows is not None:
        o, ro = o[rows], ro[rows]
        l_, rl = l_[:, rows], rl[:, rows]
    if heads is not None:
        o, ro = o[:, heads], ro[:, heads]
        l_, rl = l_[heads], rl[heads]
    check_close_bf16(o, ro, ATTN_MAX_ABS, ATTN_MEAN_ABS, what=what + " out")
    check_lse(l_, rl, what=what + " lse")


def expected_counts(wl, block_m, block_n, causal=None, cu=None, sri="default"):
    cu_np = wl.cu_seqlens if cu is None else cu
    sri_np = wl.startend_row_indices if isinstance(sri, str) else sri
    c = wl.causal if causal is None else causal
    return list(om.block_class_counts(cu_np, sri_np, wl.n_heads_q, block_m, block_n, c))


def test_tiny_causal_document(fm):
    wl = gen.make_workload(1, seed=0)
    out, lse, counts, _ = run_attn(fm, wl)
    compare(out, lse, oracle(wl), what="cfg1")
    assert counts == [2, 5, 2]


LENS = [1, 77, 128, 300, 5, 513, 0, 260, 64]


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("blocks", [(128, 128), (64, 64), (128, 64), (64, 128)])
@pytest.mark.parametrize("mask,causal", [("none", True), ("none", False),
                                         ("causal_document", True), ("window", True),
                                         ("bidir_prefix", False)])
def test_small_mask_shapes(fm, head_dim, blocks, mask, causal):
    wl = gen.make_custom(LENS, n_heads_q=4, n_heads_kv=2, head_dim=head_dim, mask=mask,
                         causal=causal, window=100, seed=7)
    bm, bn = blocks
    out, lse, counts, _ = run_attn(fm, wl, block_m=bm, block_n=bn)
    compare(out, lse, oracle(wl), what=f"{mask} D{head_dim} {bm}x{bn}")
    assert counts == expected_counts(wl, bm, bn)


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("per_head", [False, True])
@pytest.mark.parametrize("block_n", [128, 64])
def test_random_intervals(fm, seed, causal, per_head, block_n):
    """Arbitrary column intervals: many partial blocks, fully masked rows."""
    wl = gen.make_custom([3, 200, 129, 0, 64, 400], n_heads_q=4, n_heads_kv=1, head_dim=128,
                         mask="random", causal=causal, seed=seed,
                         n_mask_heads=4 if per_head else 1)
    out, lse, counts, _ = run_attn(fm, wl, block_n=block_n)
    ref = oracle(wl)
    compare(out, lse, ref, what="random")
    assert counts == expected_counts(wl, 128, block_n)


@pytest.mark.parametrize("blocks", [(128, 128), (128, 64), (64, 64)])
def test_growing_scores_rescale_o(fm, blocks):
    """A score bias that grows along every sample (q[..., 0] = 1, k[..., 0] =
    0.3 * position) raises the running row max by more than 2^8 every few
    KV tiles, so O is rescaled in TMEM many times within an item (with two S
    buffers: after waiting for the previous PV).  The bias is gentle enough
    that each row still spreads its weight over tens of keys."""
    import dataclasses
    lens = [700, 300, 1500]
    wl = gen.make_custom(lens, n_heads_q=4, n_heads_kv=2, head_dim=128,
                         mask="causal_document", seed=11)
    q = gen.bf16_bits_to_f32(wl.q_bits)
    k = gen.bf16_bits_to_f32(wl.k_bits)
    pos = np.concatenate([np.arange(n) for n in lens]).astype(np.float32)
    q[:, :, 0] = 1.0
    k[:, :, 0] = 0.3 * pos[:, None]
    wl = dataclasses.replace(wl, q_bits=gen.f32_to_bf16_bits(q), k_bits=gen.f32_to_bf16_bits(k))
    bm, bn = blocks
    out, lse, counts, _ = run_attn(fm, wl, block_m=bm, block_n=bn)
    compare(out, lse, oracle(wl), what=f"growing scores {bm}x{bn}")
    assert counts == expected_counts(wl, bm, bn)


def test_every_row_masked(fm):
    wl = gen.make_custom([50, 200], n_heads_q=2, n_heads_kv=2, head_dim=64, mask="none",
                         causal=True, seed=2)
    T = wl.total_tokens
    sri = np.zeros((1, 4, T), dtype=np.int32)
    sri[0, 1] = T
    sri[0, 3] = T
    out, lse, counts, _ = run_attn(fm, wl, sri=sri)
    assert float(out.abs().max()) == 0.0
    assert bool(np.all(np.isneginf(lse.cpu().numpy())))
    assert counts == expected_counts(wl, 128, 128, sri=sri)
    assert counts[1] == 0 and counts[2] == 0


def test_short_packs(fm):
    for lens in ([1], [3], [127], [128], [129], [0, 5, 0]):
        wl = gen.make_custom(lens, n_heads_q=2, n_heads_kv=1, head_dim=128, seed=len(lens))
        out, lse, counts, _ = run_attn(fm, wl)
        compare(out, lse, oracle(wl), what=f"lens {lens}")


def test_causal_document_encodings_agree(fm):
    """cu = [0, T] + LTS = doc end intervals == per-sample cu + causal, no intervals."""
    import torch
    wl = gen.make_custom([100, 37, 260, 1, 90], n_heads_q=4, n_heads_kv=4, head_dim=128, seed=4)
    T = wl.total_tokens
    a = run_attn(fm, wl, sri=None)
    b = run_attn(fm, wl, cu=np.array([0, T], dtype=np.int32))
    ref = oracle(wl, sri=None)
    compare(a[0], a[1], ref, what="per-sample")
    compare(b[0], b[1], ref, what="single sample + intervals")
    assert torch.equal(a[0].view(torch.int16), run_attn(fm, wl, sri=None)[0].view(torch.int16))


def test_work_items_are_real_q_tiles(fm):
    """Varlen-Packing document example: lengths [128, 128, 4096], 2 heads,
    Br = 128 -> 68 work items instead of the fixed grid's 192."""
    wl = gen.make_custom([128, 128, 4096], n_heads_q=2, n_heads_kv=2, head_dim=128, seed=0)
    _, _, _, ws = run_attn(fm, wl)
    assert fm.attn_fwd_num_work_items(ws) == 68


def _sample_rows(wl, block_m, rng, extra=2000):
    cu = wl.cu_seqlens.astype(np.int64)
    rows = [rng.integers(0, wl.total_tokens, extra)]
    for s in range(wl.n_seqs):
        a, b = int(cu[s]), int(cu[s + 1])
        if b > a:
            rows.append(np.arange(a, min(a + block_m, b)))
            rows.append(np.arange(max(a, b - block_m), b))
    return np.unique(np.concatenate(rows))


@pytest.mark.parametrize("cfg", [2, 3, 4])
@pytest.mark.parametrize("block_n", [128, 64])
def test_full_size_configs_sampled(fm, cfg, block_n):
    wl = gen.make_workload(cfg, seed=0)
    out, lse, counts, _ = run_attn(fm, wl, block_n=block_n)
    rng = np.random.default_rng(cfg)
    rows = _sample_rows(wl, 128, rng)
    heads = sorted(set([0, wl.n_heads_q - 1] + list(rng.integers(0, wl.n_heads_q, 2))))
    ref = oracle(wl, rows=rows, heads=heads)
    compare(out, lse, ref, rows=rows, heads=heads, what=f"cfg{cfg}")
    assert counts == expected_counts(wl, 128, block_n)


@pytest.mark.parametrize("block_n", [128, 64])
def test_long_context_sampled(fm, block_n):
    wl = gen.make_workload(5, seed=0)
    out, lse, counts, _ = run_attn(fm, wl, block_n=block_n)
    rng = np.random.default_rng(5)
    rows = _sample_rows(wl, 128, rng, extra=300)
    rows = np.unique(np.concatenate([rows, np.arange(65536 - 256, 65536),
                                     np.arange(40000, 40128)]))
    heads = [0, 13, 31]
    ref = oracle(wl, rows=rows, heads=heads)
    compare(out, lse, ref, rows=rows, heads=heads, what="cfg5")
    assert counts == expected_counts(wl, 128, block_n)


def test_int64_path_bit_identical(fm):
    import torch
    wl = gen.make_workload(2, seed=1)
    a = run_attn(fm, wl, force_int64=False)
    b = run_attn(fm, wl, force_int64=True)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1])
    assert a[2] == b[2]


def test_bounded_wait_reports_timeout(fm):
    assert fm.debug_bounded_wait(2_000_000) == 6   # FM_ERR_TIMEOUT, context still usable
    import torch
    assert torch.ones(4, device="cuda").sum().item() == 4.0


def test_unsupported_arguments_raise(fm):
    import torch
    q = torch.zeros((16, 1, 96), dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 16], dtype=torch.int32, device="cuda")
    with pytest.raises(fm.FMError):
        fm.attn_fwd_varlen(q, q, q, cu)
    with pytest.raises(fm.FMError):
        fm.rope_qk_varlen(q, q, cu, 1e4)
