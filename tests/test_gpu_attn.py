"""GPU parity: fm_attn_fwd_varlen against the float64 oracle.

Outputs are compared element by element (|gpu - oracle| <= 1e-2, or half a
bf16 ulp of the oracle value plus fp32 slack where that is larger, i.e. for
|value| >= 4; mean <= 1e-3; lse <= 1e-3 with identical -inf rows); block-class
counts must be identical.  The measured workloads 2-4 are compared in full
(every row, every q head), workload 2 at five seeds; the 131072-token
workload on sampled rows.
"""

import numpy as np
import pytest

from helpers import (ATTN_MAX_ABS, ATTN_MEAN_ABS, abs_v_magnitude, bf16_tensor_to_f64,
                     check_close_bf16, check_lse, ensure_library, to_device_bf16, workload_inputs)
import oracle_runs
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


def compare(out, lse, ref, rows=None, heads=None, what="", wl=None, cu=None, sri="default",
            causal=None):
    """out / lse against the oracle result ``ref``; ``wl`` (with the same
    cu / sri / causal overrides as the oracle call) lets over-bound elements
    be held to the P-rounding bound."""
    mag = None
    if wl is not None:
        mag = abs_v_magnitude(workload_inputs(wl), wl.cu_seqlens if cu is None else cu,
                              wl.startend_row_indices if isinstance(sri, str) else sri,
                              wl.causal if causal is None else causal, rows, heads)
    o = bf16_tensor_to_f64(out)
    l_ = lse.cpu().numpy().astype(np.float64)
    ro, rl = ref
    if rows is not None:
        o, ro = o[rows], ro[rows]
        l_, rl = l_[:, rows], rl[:, rows]
    if heads is not None:
        o, ro = o[:, heads], ro[:, heads]
        l_, rl = l_[heads], rl[heads]
    check_close_bf16(o, ro, ATTN_MAX_ABS, ATTN_MEAN_ABS, what=what + " out", magnitude=mag)
    check_lse(l_, rl, what=what + " lse")


def expected_counts(wl, block_m, block_n, causal=None, cu=None, sri="default"):
    cu_np = wl.cu_seqlens if cu is None else cu
    sri_np = wl.startend_row_indices if isinstance(sri, str) else sri
    c = wl.causal if causal is None else causal
    return list(om.block_class_counts(cu_np, sri_np, wl.n_heads_q, block_m, block_n, c))


def test_tiny_causal_document(fm):
    wl = gen.make_workload(1, seed=0)
    out, lse, counts, _ = run_attn(fm, wl)
    compare(out, lse, oracle(wl), what="cfg1", wl=wl)
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
    compare(out, lse, oracle(wl), what=f"{mask} D{head_dim} {bm}x{bn}", wl=wl)
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
    compare(out, lse, ref, what="random", wl=wl)
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
    compare(out, lse, oracle(wl), what=f"growing scores {bm}x{bn}", wl=wl)
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
        compare(out, lse, oracle(wl), what=f"lens {lens}", wl=wl)


def test_causal_document_encodings_agree(fm):
    """cu = [0, T] + LTS = doc end intervals == per-sample cu + causal, no intervals."""
    import torch
    wl = gen.make_custom([100, 37, 260, 1, 90], n_heads_q=4, n_heads_kv=4, head_dim=128, seed=4)
    T = wl.total_tokens
    a = run_attn(fm, wl, sri=None)
    b = run_attn(fm, wl, cu=np.array([0, T], dtype=np.int32))
    ref = oracle(wl, sri=None)
    compare(a[0], a[1], ref, what="per-sample", wl=wl, sri=None)
    compare(b[0], b[1], ref, what="single sample + intervals", wl=wl, sri=None)
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
def test_full_size_configs(fm, cfg):
    """Every row and every q head of workloads 2-4 against the float64 oracle,
    with 128- and 64-column key tiles."""
    wl = gen.make_workload(cfg, seed=0)
    ref = oracle_runs.forward_full(cfg, 0)
    for block_n in (128, 64):
        out, lse, counts, _ = run_attn(fm, wl, block_n=block_n)
        compare(out, lse, ref, what=f"cfg{cfg} block_n {block_n}", wl=wl)
        assert counts == expected_counts(wl, 128, block_n)


@pytest.mark.parametrize("seed", [1, 2, 3, 4])
def test_headline_other_seeds(fm, seed):
    """The headline workload at the other four seeds of the parity sweep, in
    full."""
    wl = gen.make_workload(2, seed=seed)
    out, lse, counts, _ = run_attn(fm, wl)
    compare(out, lse, oracle_runs.forward_full(2, seed), what=f"cfg2 seed {seed}", wl=wl)
    assert counts == expected_counts(wl, 128, 128)


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
    compare(out, lse, ref, rows=rows, heads=heads, what="cfg5", wl=wl)
    assert counts == expected_counts(wl, 128, block_n)


@pytest.mark.parametrize("cfg", [2, 5])
def test_int64_path_bit_identical(fm, cfg):
    """The 32-bit and 64-bit index specialisations give the same bits, on the
    headline workload and on the 131072-token one (whose offsets fit in 32
    bits, so both instantiations can run it)."""
    import torch
    wl = gen.make_workload(cfg, seed=1 if cfg == 2 else 0)
    a = run_attn(fm, wl, force_int64=False)
    b = run_attn(fm, wl, force_int64=True)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))
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


@pytest.mark.parametrize("cu_list", [[0, 600, 300, 1000], [0, 400, 900], [0, 1000, 1000, 700]])
def test_malformed_cu_seqlens_sets_data_error(fm, cu_list):
    """cu_seqlens whose entries all lie in [0, T] but are not non-decreasing or
    do not end at T.  The kernels clamp every index, so all accesses stay in
    bounds by construction; the call must report FM_DEVERR_DATA in the
    workspace error word and leave finite outputs.  A clean call on the same
    workspace then reads 0."""
    import torch
    wl = gen.make_custom([300, 500, 200], n_heads_q=4, n_heads_kv=2, head_dim=128,
                         mask="none", causal=True, seed=13)
    q, k, v = (to_device_bf16(b) for b in (wl.q_bits, wl.k_bits, wl.v_bits))
    ws = torch.empty(fm.attn_fwd_workspace_size(1000, 3, 4, 128), dtype=torch.uint8,
                     device="cuda")
    out = torch.zeros_like(q)
    lse = torch.zeros((4, 1000), dtype=torch.float32, device="cuda")
    bad = torch.tensor(cu_list, dtype=torch.int32, device="cuda")
    fm.attn_fwd_varlen(q, k, v, bad, causal=True, out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    assert fm.get_device_error(ws) & fm.FM_DEVERR_DATA
    assert bool(torch.isfinite(out.float()).all())
    assert not bool(torch.isnan(lse).any())
    good = torch.from_numpy(wl.cu_seqlens).cuda()
    fm.attn_fwd_varlen(q, k, v, good, causal=True, out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    assert fm.get_device_error(ws) == 0
    compare(out, lse, oracle(wl, sri=None), what="clean call after malformed", wl=wl,
            sri=None)


@pytest.mark.parametrize("block_n", [128, 64])
def test_per_head_masks_with_unequal_cost(fm, block_n):
    """One mask per q head with very different sparsity (head 0 keeps only a
    short window, head 1 is causal, head 2 sees every key of its sample,
    head 3 sees almost nothing): the planner orders work by the costliest
    head of each Q tile, and every head's result matches the oracle."""
    import dataclasses
    wl = gen.make_custom([1500, 700, 2100, 90], n_heads_q=4, n_heads_kv=2, head_dim=128,
                         mask="none", causal=False, seed=21)
    T = wl.total_tokens
    cu = wl.cu_seqlens.astype(np.int64)
    ends = np.repeat(cu[1:], np.diff(cu))
    starts = np.repeat(cu[:-1], np.diff(cu))
    j = np.arange(T)
    sri = np.zeros((4, 4, T), dtype=np.int32)
    sri[:, 1] = T
    sri[:, 3] = T
    sri[0, 0] = np.minimum(ends, j + 64)     # short causal window
    sri[0, 2], sri[0, 3] = 0, j              # upper triangle masked
    sri[1, 0] = ends                         # causal document
    sri[1, 2], sri[1, 3] = 0, j
    sri[2, 0] = ends                         # bidirectional document
    sri[2, 2], sri[2, 3] = 0, starts
    sri[3, 0] = np.minimum(ends, j + 1)      # only the diagonal
    sri[3, 2], sri[3, 3] = 0, j
    wl = dataclasses.replace(wl, startend_row_indices=sri)
    out, lse, counts, _ = run_attn(fm, wl, block_n=block_n)
    compare(out, lse, oracle(wl), what=f"per-head masks block_n {block_n}", wl=wl)
    assert counts == expected_counts(wl, 128, block_n)
