"""Full-size oracle evaluations for the parity tests, spread over the host cores.

Test infrastructure only.  The float64 oracle is evaluated head by head (the
forward pass) or key/value head group by group (the backward pass) in a pool
of worker processes started with ``spawn`` (a forked child of a process that
has touched CUDA can hang), one BLAS thread each.  Every worker rebuilds the
seeded workload from ``(cfg, seed)`` itself, so only results cross process
boundaries.  Results are cached for the session: the forward tests of the
plain, fused-RoPE and allocation-free entry points share one evaluation.

Nothing here adds arithmetic: each task calls ``oracle.attention`` /
``oracle.attention_bwd`` / ``oracle.rope`` on a subset of heads, and the
subsets are put back at their head positions.
"""

from __future__ import annotations

import concurrent.futures as cf
import functools
import multiprocessing as mp
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                "BLIS_NUM_THREADS", "VECLIB_MAXIMUM_THREADS")
_POOL = None


def _init_worker(root):
    if root not in sys.path:
        sys.path.insert(0, root)


def pool() -> cf.ProcessPoolExecutor:
    global _POOL
    if _POOL is None:
        # Workers are spawned lazily and inherit the environment at that
        # moment; this process's own BLAS was configured when it imported
        # numpy and is not affected.
        for k in _THREAD_VARS:
            os.environ[k] = "1"
        n = max(1, min(os.cpu_count() or 1, 32))
        _POOL = cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"),
                                       initializer=_init_worker, initargs=(ROOT,))
    return _POOL


# ---------------------------------------------------------------------------
# worker side
# ---------------------------------------------------------------------------

_WL = {}
_DOUT = {}


def _workload(cfg, seed):
    key = (cfg, seed)
    if key not in _WL:
        from workloads import gen
        _WL.clear()
        _DOUT.clear()
        _WL[key] = gen.make_workload(cfg, seed=seed)
    return _WL[key]


def dout_bits(wl, dout_seed):
    """Seeded output gradient of a workload (bf16 bits), as the backward tests
    draw it."""
    import numpy as np
    from workloads import gen
    rng = np.random.default_rng(1000 + dout_seed)
    return gen.f32_to_bf16_bits(
        rng.standard_normal((wl.total_tokens, wl.n_heads_q, wl.head_dim)).astype(np.float32))


def _rope_bf16(x64, cu, theta):
    """Oracle RoPE of float64 inputs, stored as bfloat16 like the rotated
    tensors the attention consumes (a format conversion of the oracle's
    result)."""
    import numpy as np
    from oracle import rope as orope
    from workloads import gen
    y = orope.rope_apply(x64, cu, theta)
    return gen.bf16_bits_to_f64(gen.f32_to_bf16_bits(y.astype(np.float32)))


def _fwd_task(cfg, seed, heads, rope):
    from oracle import attention as oat
    from workloads import gen
    wl = _workload(cfg, seed)
    group = wl.n_heads_q // wl.n_heads_kv
    kvh = [h // group for h in heads]
    q = gen.bf16_bits_to_f64(wl.q_bits[:, heads])
    k = gen.bf16_bits_to_f64(wl.k_bits[:, kvh])
    v = gen.bf16_bits_to_f64(wl.v_bits[:, kvh])
    if rope:
        q = _rope_bf16(q, wl.cu_seqlens, wl.theta)
        k = _rope_bf16(k, wl.cu_seqlens, wl.theta)
    sri = wl.startend_row_indices
    if sri is not None and sri.shape[0] > 1:
        sri = sri[heads]
    o, lse = oat.attention_forward(q, k, v, wl.cu_seqlens, sri, wl.causal)
    return heads, o, lse


def _bwd_task(cfg, seed, dout_seed, g):
    from oracle import attention_bwd as ob
    from workloads import gen
    wl = _workload(cfg, seed)
    key = (cfg, seed, dout_seed)
    if key not in _DOUT:
        _DOUT[key] = dout_bits(wl, dout_seed)
    do = _DOUT[key]
    grp = wl.n_heads_q // wl.n_heads_kv
    hs = list(range(g * grp, (g + 1) * grp))
    sri = wl.startend_row_indices
    if sri is not None and sri.shape[0] > 1:
        sri = sri[hs]
    f64 = gen.bf16_bits_to_f64
    r = ob.attention_backward(f64(wl.q_bits[:, hs]), f64(wl.k_bits[:, [g]]),
                              f64(wl.v_bits[:, [g]]), f64(do[:, hs]), wl.cu_seqlens, sri,
                              wl.causal, magnitudes=True)
    return g, hs, r


# ---------------------------------------------------------------------------
# caller side
# ---------------------------------------------------------------------------

@functools.lru_cache(maxsize=2)
def forward_full(cfg: int, seed: int = 0, rope: bool = False):
    """Oracle (out [T, Hq, D], lse [Hq, T]) of workload ``cfg`` at ``seed``,
    every row and every q head.  ``rope``: on RoPE(q), RoPE(k) stored as
    bf16."""
    import numpy as np
    from workloads import gen
    wl = gen.make_workload(cfg, seed=seed, tensors=False)
    T, Hq, D = wl.total_tokens, wl.n_heads_q, wl.head_dim
    out = np.empty((T, Hq, D))
    lse = np.empty((Hq, T))
    futs = [pool().submit(_fwd_task, cfg, seed, [h], rope) for h in range(Hq)]
    for f in futs:
        heads, o, l_ = f.result()
        out[:, heads] = o
        lse[heads] = l_
    return out, lse


@functools.lru_cache(maxsize=1)
def backward_full(cfg: int, seed: int, dout_seed: int):
    """Oracle gradients ([dq, dk, dv]) and magnitude sums ([mq, mk, mv]) of
    workload ``cfg`` at ``seed`` with the output gradient drawn by
    ``dout_bits(wl, dout_seed)``, every row and head."""
    import numpy as np
    from workloads import gen
    wl = gen.make_workload(cfg, seed=seed, tensors=False)
    T, D = wl.total_tokens, wl.head_dim
    shapes = (wl.n_heads_q, wl.n_heads_kv, wl.n_heads_kv)
    grads = [np.empty((T, h, D)) for h in shapes]
    mags = [np.empty((T, h, D)) for h in shapes]
    futs = [pool().submit(_bwd_task, cfg, seed, dout_seed, g) for g in range(wl.n_heads_kv)]
    for f in futs:
        g, hs, (dq, dk, dv, mq, mk, mv) = f.result()
        grads[0][:, hs], grads[1][:, [g]], grads[2][:, [g]] = dq, dk, dv
        mags[0][:, hs], mags[1][:, [g]], mags[2][:, [g]] = mq, mk, mv
    return grads, mags
