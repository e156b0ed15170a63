"""GPU: the host collator's packs give the same results as each sample alone.

Tiles, block classes and work items are all local to a sample, so the RoPE +
tile statistics + attention step on a pack built by
``packing.collate`` must reproduce, bit for bit, the same step run on every
sample as a batch of its own (Unsloth packing blog: packing must not let
attention leak across samples and must restart positions per sample;
FlashMask article, section 6.7: the row-index offset of concatenated
samples).  The pack is also checked against the float64 oracle.
"""

import numpy as np
import pytest

from helpers import (ATTN_MAX_ABS, ATTN_MEAN_ABS, abs_v_magnitude, bf16_tensor_to_f64,
                     check_close_bf16, check_lse, ensure_library)
from oracle import attention as oat
from oracle import rope as orope
from packed_varlen_attention_gb300 import packing as pk
from workloads import gen

pytestmark = pytest.mark.gpu

HQ, HKV, D = 4, 2, 128
THETA = 1.0e4


@pytest.fixture(scope="module")
def fm():
    return ensure_library()


def _samples(seed, causal):
    rng = np.random.default_rng(seed)
    specs = []
    if causal:
        specs = [("causal", 300), ("shared", (200, [150, 90, 64])), ("window", (513, 100)),
                 ("none", 77), ("causal", 1), ("shared", (64, [129]))]
    else:
        specs = [("prefix", (700, 200)), ("bidir", 129), ("causal", 256), ("prefix", (65, 64)),
                 ("bidir", 3)]
    lens, ivs = [], []
    for kind, a in specs:
        if kind == "causal":
            n, iv = a, pk.intervals_causal(a)
        elif kind == "none":
            n, iv = a, None
        elif kind == "shared":
            n, iv = a[0] + sum(a[1]), pk.intervals_shared_question(a[0], a[1])
        elif kind == "window":
            n, iv = a[0], pk.intervals_sliding_window(a[0], a[1])
        elif kind == "prefix":
            n, iv = a[0], pk.intervals_prefix_lm(a[0], a[1])
        else:
            n, iv = a, pk.intervals_bidirectional(a)
        lens.append(n)
        ivs.append(iv)
    qs = [gen.f32_to_bf16_bits(rng.standard_normal((n, HQ, D)).astype(np.float32)) for n in lens]
    ks = [gen.f32_to_bf16_bits(rng.standard_normal((n, HKV, D)).astype(np.float32)) for n in lens]
    vs = [gen.f32_to_bf16_bits(rng.standard_normal((n, HKV, D)).astype(np.float32)) for n in lens]
    return lens, ivs, qs, ks, vs


def _step(fm, q_bits, k_bits, v_bits, cu, sri, causal, block_n):
    import torch
    dt = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    q, k, v = dt(q_bits), dt(k_bits), dt(v_bits)
    cu_t = torch.from_numpy(np.ascontiguousarray(cu, dtype=np.int32)).cuda()
    fm.rope_qk_varlen(q, k, cu_t, THETA)
    sri_t = torch.from_numpy(np.ascontiguousarray(sri, dtype=np.int32)).cuda()
    mm = fm.mask_block_minmax(sri_t, cu_t, block_n)
    out, lse = fm.attn_fwd_varlen(q, k, v, cu_t, sri_t, mm, causal=causal, block_m=128,
                                  block_n=block_n)
    torch.cuda.synchronize()
    return q, k, out, lse


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("block_n", [128, 64])
def test_pack_equals_samples_alone(fm, causal, block_n):
    import torch
    lens, ivs, qs, ks, vs = _samples(5 if causal else 6, causal)
    p = pk.collate(qs, ivs)
    kp = pk.collate(ks).tokens
    vp = pk.collate(vs).tokens
    cu = p.cu_seqlens
    qr, kr, out, lse = _step(fm, p.tokens, kp, vp, cu, p.startend_row_indices, causal, block_n)
    for s, n in enumerate(lens):
        if n == 0:
            continue
        a = int(cu[s])
        local = pk.collate([qs[s]], [ivs[s]]).startend_row_indices
        q1, k1, o1, l1 = _step(fm, qs[s], ks[s], vs[s], np.array([0, n]), local, causal, block_n)
        assert torch.equal(qr[a:a + n].view(torch.int16), q1.view(torch.int16)), f"rope q, sample {s}"
        assert torch.equal(kr[a:a + n].view(torch.int16), k1.view(torch.int16)), f"rope k, sample {s}"
        assert torch.equal(out[a:a + n].view(torch.int16), o1.view(torch.int16)), f"out, sample {s}"
        assert torch.equal(lse[:, a:a + n], l1), f"lse, sample {s}"
    # and the pack against the float64 oracle: RoPE on the inputs, then
    # attention on the oracle's rotated values stored as bf16 (the in-place
    # rotation keeps q and k in bf16; nothing here comes from the GPU)
    f64 = gen.bf16_bits_to_f64
    q_rot = orope.rope_apply(f64(p.tokens), cu, THETA)
    k_rot = orope.rope_apply(f64(kp), cu, THETA)
    check_close_bf16(bf16_tensor_to_f64(qr), q_rot, 8e-3, what="pack rope q")
    check_close_bf16(bf16_tensor_to_f64(kr), k_rot, 8e-3, what="pack rope k")
    as_bf16 = lambda x: f64(gen.f32_to_bf16_bits(x.astype(np.float32)))
    ref_o, ref_l = oat.attention_forward(as_bf16(q_rot), as_bf16(k_rot), f64(vp), cu,
                                         p.startend_row_indices, causal)
    mag = abs_v_magnitude(lambda: (as_bf16(q_rot), as_bf16(k_rot), f64(vp)), cu,
                          p.startend_row_indices, causal)
    check_close_bf16(bf16_tensor_to_f64(out), ref_o, ATTN_MAX_ABS, ATTN_MEAN_ABS, what="pack out",
                     magnitude=mag)
    check_lse(lse.cpu().numpy().astype(np.float64), ref_l, what="pack lse")
