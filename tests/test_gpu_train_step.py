"""GPU: the attention block of one packed training step, forward and backward.

q, k are rotated in place (positions restarting per sample), attention runs
forward and backward, and the gradients of the rotated q, k are rotated back
(RoPE backward: the same rotation with sin -> -sin; Unsloth packing blog,
section "Fused QK RoPE Triton kernel with packing").  The float64 oracle
takes the generator's inputs only: RoPE, rotated values stored as bf16 (the
in-place rotation keeps them in bf16), the attention gradients, the inverse
rotation.

Tolerance: the gradient bound of the backward tests, 4u m + u |oracle| with
u = 2^-8 and m the oracle's magnitude sums, carried through the rotation
(each output pairs channel i with i + D/2, so a pair's bounds combine as
sqrt(b_i^2 + b_j^2)), plus one more bf16 rounding for the rotated-back
result.
"""

import numpy as np
import pytest

from helpers import bf16_tensor_to_f64, ensure_library, to_device_bf16
from oracle import attention_bwd as ob
from oracle import rope as orope
from workloads import gen

pytestmark = pytest.mark.gpu

U = 2.0 ** -8


@pytest.fixture(scope="module")
def fm():
    return ensure_library()


def _pair_bound(mag):
    """sqrt(m_i^2 + m_j^2) for channel pairs (i, i + D/2)."""
    half = mag.shape[-1] // 2
    a, b = mag[..., :half], mag[..., half:]
    r = np.sqrt(a * a + b * b)
    return np.concatenate([r, r], axis=-1)


@pytest.mark.parametrize("mask,causal,lens", [
    ("causal_document", True, [300, 129, 700, 64, 1]),
    ("window", True, [513, 250, 90]),
    ("bidir_prefix", False, [400, 333, 128]),
])
def test_rope_attention_forward_backward(fm, mask, causal, lens):
    import torch
    wl = gen.make_custom(lens, n_heads_q=8, n_heads_kv=2, head_dim=128, mask=mask, causal=causal,
                         window=120, seed=21, theta=5.0e5)
    rng = np.random.default_rng(77)
    do_bits = gen.f32_to_bf16_bits(
        rng.standard_normal((wl.total_tokens, 8, 128)).astype(np.float32))
    q, k, v, do = (to_device_bf16(b) for b in (wl.q_bits, wl.k_bits, wl.v_bits, do_bits))
    cu = torch.from_numpy(wl.cu_seqlens).cuda()
    sri = torch.from_numpy(wl.startend_row_indices).cuda()
    mm = fm.mask_block_minmax(sri, cu, 128)
    fm.rope_qk_varlen(q, k, cu, wl.theta)
    out, lse = fm.attn_fwd_varlen(q, k, v, cu, sri, mm, causal=causal)
    dq, dk, dv = fm.attn_bwd_varlen(q, k, v, out, do, lse, cu, sri, mm, causal=causal)
    fm.rope_qk_varlen(dq, dk, cu, wl.theta, backward=True)
    torch.cuda.synchronize()

    f64 = gen.bf16_bits_to_f64
    as_bf16 = lambda x: f64(gen.f32_to_bf16_bits(x.astype(np.float32)))
    q_rot = as_bf16(orope.rope_apply(f64(wl.q_bits), wl.cu_seqlens, wl.theta))
    k_rot = as_bf16(orope.rope_apply(f64(wl.k_bits), wl.cu_seqlens, wl.theta))
    gq, gk, gv, mq, mk, mv = ob.attention_backward(q_rot, k_rot, f64(wl.v_bits), f64(do_bits),
                                                   wl.cu_seqlens, wl.startend_row_indices,
                                                   causal, magnitudes=True)
    ref_q = orope.rope_apply(gq, wl.cu_seqlens, wl.theta, backward=True)
    ref_k = orope.rope_apply(gk, wl.cu_seqlens, wl.theta, backward=True)
    for got, ref, mag, what in ((dq, ref_q, _pair_bound(mq), "dq"),
                                (dk, ref_k, _pair_bound(mk), "dk"),
                                (dv, gv, mv, "dv")):
        g = bf16_tensor_to_f64(got)
        extra = U * np.abs(ref) if what != "dv" else 0.0
        bound = 4 * U * mag + U * np.abs(ref) + extra + 1e-30
        ratio = np.abs(g - ref) / bound
        assert np.all(np.isfinite(g)), what
        assert ratio.max() <= 1.0, (f"{mask} {what}: worst ratio {ratio.max():.3f} at "
                                    f"{np.unravel_index(np.argmax(ratio), ratio.shape)}")
