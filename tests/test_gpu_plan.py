"""GPU: the forward scheduler run once and reused (fm_attn_fwd_plan and
FM_FLAG_REUSE_PLAN).

The work list depends only on cu_seqlens and the sizes, so the layers of one
packed batch can share one plan.  Every call that reuses it must give the
bits of a call that plans for itself, call after call and under CUDA-graph
replay (the kernel resets the item counter it claims from), and the first
such layer must match the float64 oracle.  A plan that does not fit the call
(other sizes, overwritten by the backward, or made from malformed
cu_seqlens) must compute nothing and set FM_DEVERR_DATA.  Every buffer is
sized for the call that uses it, so all cases stay in bounds by
construction.
"""

import numpy as np
import pytest

from helpers import ensure_library, to_device_bf16
import oracle_runs
from test_gpu_attn import compare
from test_gpu_graph import _capture, _same
from workloads import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    return ensure_library()


class Batch:
    """One packed batch (samples and mask of a workload) and the inputs of
    several layers over it: layer 0 holds the workload's own q, k, v, the
    others seeded normals of the same shapes."""

    def __init__(self, fm, wl, n_layers):
        import torch
        self.wl = wl
        self.cu = torch.from_numpy(np.ascontiguousarray(wl.cu_seqlens)).cuda()
        self.sri = self.mm = None
        if wl.startend_row_indices is not None:
            self.sri = torch.from_numpy(np.ascontiguousarray(wl.startend_row_indices)).cuda()
            self.mm = fm.mask_block_minmax(self.sri, self.cu, wl.block_n)
        self.layers = [tuple(to_device_bf16(b) for b in (wl.q_bits, wl.k_bits, wl.v_bits))]
        rng = np.random.default_rng(1234)
        for _ in range(n_layers - 1):
            self.layers.append(tuple(
                to_device_bf16(gen.f32_to_bf16_bits(rng.standard_normal(b.shape, dtype=np.float32)))
                for b in (wl.q_bits, wl.k_bits, wl.v_bits)))

    def plan(self, fm, workspace=None):
        wl = self.wl
        return fm.attn_fwd_plan(self.cu, wl.total_tokens, wl.n_heads_q, wl.n_heads_kv,
                                self.sri, self.mm,
                                causal=wl.causal, block_m=wl.block_m, block_n=wl.block_n,
                                workspace=workspace)

    def attn(self, fm, layer, ws, reuse, out=None, lse=None, counts=None):
        wl = self.wl
        q, k, v = self.layers[layer]
        return fm.attn_fwd_varlen(q, k, v, self.cu, self.sri, self.mm, causal=wl.causal,
                                  block_m=wl.block_m, block_n=wl.block_n, out=out, lse=lse,
                                  class_counts=counts, workspace=ws, force_int64=wl.force_int64,
                                  reuse_plan=reuse)


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_reused_plan_gives_the_bits_of_a_fresh_call(fm, cfg):
    import torch
    wl = gen.make_workload(cfg, seed=0)
    b = Batch(fm, wl, n_layers=3)
    ws = b.plan(fm)
    for layer in range(3):
        cr = torch.zeros(3, dtype=torch.int64, device="cuda")
        cf = torch.zeros(3, dtype=torch.int64, device="cuda")
        out_r, lse_r = b.attn(fm, layer, ws, True, counts=cr)
        out_f, lse_f = b.attn(fm, layer, None, False, counts=cf)
        torch.cuda.synchronize()
        assert fm.get_device_error(ws) == 0
        assert _same(out_r, out_f) and _same(lse_r, lse_f), f"layer {layer}"
        assert cr.tolist() == cf.tolist()
        if layer == 0 and cfg == 2:
            compare(out_r, lse_r, oracle_runs.forward_full(cfg, 0), what=f"cfg{cfg} reused plan",
                    wl=wl)


@pytest.mark.parametrize("head_dim,block", [(64, 64), (128, 64), (64, 128)])
def test_reused_plan_other_tile_shapes(fm, head_dim, block):
    """The 64-row / 64-column tile kernels and head_dim 64 on one plan, two
    layers: the bits of calls that plan for themselves, and the oracle."""
    import torch
    from test_gpu_attn import oracle
    wl = gen.make_custom([300, 77, 1000, 129, 64], n_heads_q=4, n_heads_kv=2,
                         head_dim=head_dim, block_m=block, block_n=block,
                         mask="causal_document", seed=17)
    b = Batch(fm, wl, n_layers=2)
    ws = b.plan(fm)
    for layer in range(2):
        out_r, lse_r = b.attn(fm, layer, ws, True)
        out_f, lse_f = b.attn(fm, layer, None, False)
        torch.cuda.synchronize()
        assert fm.get_device_error(ws) == 0
        assert _same(out_r, out_f) and _same(lse_r, lse_f), f"layer {layer}"
        if layer == 0:
            compare(out_r, lse_r, oracle(wl), what=f"D={head_dim} block {block} reused plan",
                    wl=wl)


def test_reused_plan_with_fused_rope(fm):
    import torch
    wl = gen.make_workload(2, seed=1)
    b = Batch(fm, wl, n_layers=2)
    ws = b.plan(fm)
    for layer in range(2):
        q, k, v = b.layers[layer]
        res = []
        for reuse in (True, False):
            kk = k.clone()
            q_rot = torch.empty_like(q)
            out, lse = fm.attn_fwd_varlen_rope(
                q, kk, v, b.cu, wl.theta, b.sri, b.mm, causal=wl.causal, block_m=wl.block_m,
                block_n=wl.block_n, q_rot=q_rot, workspace=ws if reuse else None,
                force_int64=wl.force_int64, reuse_plan=reuse)
            res.append((out, lse, q_rot, kk))
        torch.cuda.synchronize()
        assert fm.get_device_error(ws) == 0
        for x, y in zip(*res):
            assert _same(x, y), f"layer {layer}"


def test_plan_for_other_sizes_computes_nothing(fm):
    """A plan made for the 8192-token batch, reused by a call on a smaller
    batch (its workspace is large enough for both): nothing is written, the
    error word says FM_DEVERR_DATA, and a call that plans for itself on the
    same workspace then computes the right result again."""
    import torch
    big = Batch(fm, gen.make_workload(2, seed=0), n_layers=1)
    ws = big.plan(fm)
    wl = gen.make_custom([300, 500, 200], n_heads_q=4, n_heads_kv=2, head_dim=128,
                         mask="none", causal=True, seed=13)
    small = Batch(fm, wl, n_layers=1)
    assert ws.numel() >= fm.attn_fwd_workspace_size(wl.total_tokens, wl.n_seqs, 4, wl.block_m)
    q = small.layers[0][0]
    out = torch.full_like(q, 7.0)
    lse = torch.full((4, wl.total_tokens), 7.0, dtype=torch.float32, device="cuda")
    small.attn(fm, 0, ws, True, out=out, lse=lse)
    torch.cuda.synchronize()
    assert fm.get_device_error(ws) & fm.FM_DEVERR_DATA
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())
    ref_out, ref_lse = small.attn(fm, 0, None, False)
    small.attn(fm, 0, ws, False, out=out, lse=lse)  # plans for itself
    torch.cuda.synchronize()
    assert fm.get_device_error(ws) == 0
    assert _same(out, ref_out) and _same(lse, ref_lse)
    out2, lse2 = small.attn(fm, 0, ws, True)  # that plan is reusable
    torch.cuda.synchronize()
    assert fm.get_device_error(ws) == 0
    assert _same(out2, ref_out) and _same(lse2, ref_lse)


def test_backward_on_the_workspace_retires_the_plan(fm):
    import torch
    wl = gen.make_custom([700, 1100, 250], n_heads_q=4, n_heads_kv=2, head_dim=128,
                         mask="causal_document", seed=5)
    b = Batch(fm, wl, n_layers=1)
    T, n = wl.total_tokens, wl.n_seqs
    nbytes = max(fm.attn_fwd_workspace_size(T, n, 4, wl.block_m),
                 fm.attn_bwd_workspace_size(T, n, 4))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    b.plan(fm, workspace=ws)
    out, lse = b.attn(fm, 0, ws, True)
    torch.cuda.synchronize()
    assert fm.get_device_error(ws) == 0
    q, k, v = b.layers[0]
    mm128 = fm.mask_block_minmax(b.sri, b.cu, 128)
    fm.attn_bwd_varlen(q, k, v, out, torch.ones_like(out), lse, b.cu, b.sri, mm128,
                       causal=wl.causal, workspace=ws)
    torch.cuda.synchronize()
    assert fm.get_device_error(ws) == 0
    out2 = torch.full_like(out, 7.0)
    b.attn(fm, 0, ws, True, out=out2)
    torch.cuda.synchronize()
    assert fm.get_device_error(ws) & fm.FM_DEVERR_DATA
    assert bool((out2 == 7.0).all())


def test_plan_from_malformed_cu_seqlens_is_not_reused(fm):
    """cu_seqlens inside [0, T] but decreasing: the planner flags
    FM_DEVERR_DATA, and a call that reuses that plan computes nothing (the
    error stays set until the next plan)."""
    import torch
    wl = gen.make_custom([300, 500, 200], n_heads_q=4, n_heads_kv=2, head_dim=128,
                         mask="none", causal=True, seed=13)
    b = Batch(fm, wl, n_layers=1)
    bad = torch.tensor([0, 600, 300, 1000], dtype=torch.int32, device="cuda")
    ws = fm.attn_fwd_plan(bad, wl.total_tokens, 4, 2, causal=True)
    q, k, v = b.layers[0]
    out = torch.full_like(q, 7.0)
    fm.attn_fwd_varlen(q, k, v, bad, causal=True, out=out, workspace=ws, reuse_plan=True)
    torch.cuda.synchronize()
    assert fm.get_device_error(ws) & fm.FM_DEVERR_DATA
    assert bool((out == 7.0).all())


def test_reused_plan_under_graph_replay(fm):
    """Two layers on one plan captured in a CUDA graph and replayed three
    times: every replay gives the bits of the eager calls that plan for
    themselves."""
    import torch
    wl = gen.make_workload(2, seed=2)
    b = Batch(fm, wl, n_layers=2)
    ws = b.plan(fm)
    outs = [torch.empty_like(b.layers[i][0]) for i in range(2)]
    lses = [torch.empty((wl.n_heads_q, wl.total_tokens), dtype=torch.float32, device="cuda")
            for _ in range(2)]
    refs = [b.attn(fm, i, None, False) for i in range(2)]

    def layers():
        for i in range(2):
            b.attn(fm, i, ws, True, out=outs[i], lse=lses[i])

    g = _capture(layers)
    for _ in range(3):
        for t in outs + lses:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for i in range(2):
            assert _same(outs[i], refs[i][0]) and _same(lses[i], refs[i][1]), f"layer {i}"
    assert fm.get_device_error(ws) == 0
