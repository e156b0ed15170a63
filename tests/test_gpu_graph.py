"""GPU: the hot path captured in a CUDA graph.

Every call is stream-ordered, allocates nothing and never synchronises, and
its kernels are programmatic dependent launches; so a training or serving
loop can capture RoPE -> tile statistics -> attention (forward, fused-RoPE
forward, backward) once and replay it.  Each test captures the calls on
preallocated buffers, replays the graph twice and requires the bits of the
eager calls on the same inputs.
"""

import numpy as np
import pytest

from helpers import ensure_library, to_device_bf16
from workloads import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fm():
    return ensure_library()


class Buffers:
    def __init__(self, fm, wl):
        import torch
        self.wl = wl
        self.q0, self.k0, self.v = (to_device_bf16(b) for b in (wl.q_bits, wl.k_bits, wl.v_bits))
        self.q = self.q0.clone()
        self.k = self.k0.clone()
        self.cu = torch.from_numpy(np.ascontiguousarray(wl.cu_seqlens)).cuda()
        self.sri = torch.from_numpy(np.ascontiguousarray(wl.startend_row_indices)).cuda()
        T, n = wl.total_tokens, wl.n_seqs
        self.mm = torch.empty((self.sri.shape[0], 8, fm.num_kv_tiles_bound(T, n, wl.block_n)),
                              dtype=torch.int32, device="cuda")
        self.mm128 = torch.empty((self.sri.shape[0], 8, fm.num_kv_tiles_bound(T, n, 128)),
                                 dtype=torch.int32, device="cuda")
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((wl.n_heads_q, T), dtype=torch.float32, device="cuda")
        self.q_rot = torch.empty_like(self.q)
        self.ws = torch.empty(fm.attn_fwd_workspace_size(T, n, wl.n_heads_q, wl.block_m),
                              dtype=torch.uint8, device="cuda")
        rng = np.random.default_rng(99)
        self.dout = to_device_bf16(gen.f32_to_bf16_bits(
            rng.standard_normal(wl.q_bits.shape, dtype=np.float32)))
        self.dq = torch.empty_like(self.q)
        self.dk = torch.empty_like(self.k)
        self.dv = torch.empty_like(self.v)
        self.bws = torch.empty(fm.attn_bwd_workspace_size(T, n, wl.n_heads_q), dtype=torch.uint8,
                               device="cuda")

    def forward(self, fm):
        wl = self.wl
        self.q.copy_(self.q0)
        self.k.copy_(self.k0)
        fm.rope_qk_varlen(self.q, self.k, self.cu, wl.theta, force_int64=wl.force_int64)
        fm.mask_block_minmax(self.sri, self.cu, wl.block_n, out=self.mm)
        fm.attn_fwd_varlen(self.q, self.k, self.v, self.cu, self.sri, self.mm, causal=wl.causal,
                           block_m=wl.block_m, block_n=wl.block_n, out=self.out, lse=self.lse,
                           workspace=self.ws, force_int64=wl.force_int64)

    def fused(self, fm):
        wl = self.wl
        self.k.copy_(self.k0)
        fm.mask_block_minmax(self.sri, self.cu, wl.block_n, out=self.mm)
        fm.attn_fwd_varlen_rope(self.q0, self.k, self.v, self.cu, wl.theta, self.sri, self.mm,
                                causal=wl.causal, block_m=wl.block_m, block_n=wl.block_n,
                                out=self.out, lse=self.lse, q_rot=self.q_rot, workspace=self.ws,
                                force_int64=wl.force_int64)

    def backward(self, fm):
        wl = self.wl
        self.forward(fm)
        fm.mask_block_minmax(self.sri, self.cu, 128, out=self.mm128)
        fm.attn_bwd_varlen(self.q, self.k, self.v, self.out, self.dout, self.lse, self.cu,
                           self.sri, self.mm128, causal=wl.causal, dq=self.dq, dk=self.dk,
                           dv=self.dv, workspace=self.bws, force_int64=wl.force_int64)

    def snapshot(self, names):
        return [getattr(self, n).clone() for n in names]


def _capture(fn):
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()  # first calls (device attributes, kernel attributes) outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _same(a, b):
    import torch
    if a.dtype == torch.bfloat16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    if a.dtype == torch.float32:
        return torch.equal(a.view(torch.int32), b.view(torch.int32))
    return torch.equal(a, b)


@pytest.mark.parametrize("cfg", [1, 2, 3])
@pytest.mark.parametrize("path,names", [
    ("forward", ["q", "k", "out", "lse"]),
    ("fused", ["k", "q_rot", "out", "lse"]),
    ("backward", ["out", "lse", "dq", "dk", "dv"]),
])
def test_graph_replay_matches_eager(fm, cfg, path, names):
    import torch
    wl = gen.make_workload(cfg, seed=3)
    b = Buffers(fm, wl)
    fn = lambda: getattr(b, path)(fm)  # noqa: E731
    fn()
    torch.cuda.synchronize()
    ref = b.snapshot(names)
    g = _capture(fn)
    for _ in range(2):
        for n in names:
            getattr(b, n).zero_()
        g.replay()
        torch.cuda.synchronize()
        for n, r in zip(names, ref):
            assert _same(getattr(b, n), r), f"{path} {n} differs after graph replay"
    assert fm.get_device_error(b.ws) == 0
    if path == "backward":
        assert fm.get_device_error(b.bws) == 0
