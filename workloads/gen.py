"""Seeded generator for the five packed-document workloads.

Every workload is a 1-D packed token tensor: documents are concatenated with
no padding and described by ``cu_seqlens`` (int32, ``cu[0] = 0``,
``cu[n] = T``), following the padding-free packing of the Unsloth packing
blog ("Why padding is needed" and "Uncontaminated packing" sections) and the
varlen layout of the Varlen-Packing document (section 1.1, ``cu_seqlens``
kept in HBM).

Masks are written in FlashMask's column-wise form (PaddleNLP FlashMask
article, sections 2.1-2.2): for every key column ``j`` four row indices
LTS/LTE (rows masked below the diagonal are ``[LTS_j, LTE_j)``) and UTS/UTE
(rows masked above the diagonal are ``[UTS_j, UTE_j)``).  Indices are global
row coordinates of the packed tensor, i.e. every sample's indices carry the
running ``sequence_sum`` offset that the article's ZeroPadding section adds
when samples are concatenated.  The array layout is ``int32[Hm][4][T]`` with
the four vectors in the order LTS, LTE, UTS, UTE.  Vectors a recipe leaves
unused hold the article's defaults (start 0, end = query length ``T``).

Random numbers: ``numpy.random.default_rng(seed)``; integer lengths are
inclusive-uniform; "until full" truncates the last document to the tokens
left.  q/k/v are N(0, 1) float32 draws rounded to bfloat16 (round to nearest
even); they are returned as raw bfloat16 bit patterns (uint16).

Nothing here computes RoPE, masks, block statistics or attention.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

CONFIG_NAMES = {
    1: "tiny_causal_document_h1_d64_t256",
    2: "llama3_8b_sft_packing_gqa32x8_d128_t8192",
    3: "dpo_rm_shared_question_h32_d128_t16k",
    4: "bidirectional_prefix_lm_mix_h16_d128_t16384",
    5: "long_context_causal_doc_window4096_gqa32x8_d128_t131072",
}


# ----------------------------------------------------------------------------
# bfloat16 bit helpers (storage format conversion only)
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(b).astype(np.float64)


# ----------------------------------------------------------------------------
# workload description
# ----------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    total_tokens: int
    n_heads_q: int
    n_heads_kv: int
    head_dim: int
    theta: float
    causal: bool
    block_m: int
    block_n: int
    force_int64: bool
    cu_seqlens: np.ndarray                     # int32 [n_seqs + 1]
    startend_row_indices: Optional[np.ndarray]  # int32 [Hm][4][T] or None
    doc_kinds: List[str] = field(default_factory=list)
    # shared-question workloads: (group start, question length, [answer lengths])
    groups: List[tuple] = field(default_factory=list)
    q_bits: Optional[np.ndarray] = None        # uint16 [T, Hq, D]
    k_bits: Optional[np.ndarray] = None        # uint16 [T, Hkv, D]
    v_bits: Optional[np.ndarray] = None        # uint16 [T, Hkv, D]
    seed: int = 0

    @property
    def n_seqs(self) -> int:
        return int(len(self.cu_seqlens) - 1)

    @property
    def seq_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens.astype(np.int64))

    @property
    def max_seqlen(self) -> int:
        return int(self.seq_lens.max()) if self.n_seqs else 0

    @property
    def n_mask_heads(self) -> int:
        return 0 if self.startend_row_indices is None else int(self.startend_row_indices.shape[0])


# ----------------------------------------------------------------------------
# document structure
# ----------------------------------------------------------------------------

def _fill_until_full(rng, total, draw):
    lens = []
    used = 0
    while used < total:
        n = int(draw())
        n = min(n, total - used)
        lens.append(n)
        used += n
    return lens


def _cu_from_lens(lens) -> np.ndarray:
    cu = np.zeros(len(lens) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(lens, dtype=np.int64))
    return cu.astype(np.int32)


def _doc_end_per_token(cu: np.ndarray, total: int) -> np.ndarray:
    lens = np.diff(cu.astype(np.int64))
    return np.repeat(cu[1:].astype(np.int64), lens)


def _doc_start_per_token(cu: np.ndarray, total: int) -> np.ndarray:
    lens = np.diff(cu.astype(np.int64))
    return np.repeat(cu[:-1].astype(np.int64), lens)


def _default_intervals(total: int, n_mask_heads: int = 1) -> np.ndarray:
    sri = np.zeros((n_mask_heads, 4, total), dtype=np.int32)
    sri[:, 1, :] = total  # LTE default: query length
    sri[:, 3, :] = total  # UTE default: query length
    return sri


# ----------------------------------------------------------------------------
# mask recipes (PaddleNLP FlashMask article, sections 1, 5.1-5.2)
# ----------------------------------------------------------------------------

def causal_document_intervals(cu: np.ndarray, total: int) -> np.ndarray:
    """Causal document mask: key column j hides rows from its doc end onward."""
    sri = _default_intervals(total)
    sri[0, 0, :] = _doc_end_per_token(cu, total)
    return sri


def sliding_window_intervals(cu: np.ndarray, total: int, window: int) -> np.ndarray:
    """Causal document mask intersected with a window of ``window`` keys.

    Key j is visible to row i iff 0 <= i - j < window and both are in the same
    document, so rows from ``min(doc_end, j + window)`` onward are hidden.
    """
    sri = _default_intervals(total)
    j = np.arange(total, dtype=np.int64)
    sri[0, 0, :] = np.minimum(_doc_end_per_token(cu, total), j + window)
    return sri


def shared_question_intervals(groups, total: int) -> np.ndarray:
    """DPO/RM shared-question mask (one question followed by its answers).

    ``groups`` is a list of (group_start, question_len, [answer_lens]).  The
    question's columns stay visible to the whole group; an answer's columns
    are hidden from rows after the answer up to the group end, so sibling
    answers never see each other.  The upper triangle is causal.
    """
    sri = _default_intervals(total)
    for g0, qlen, alens in groups:
        gend = g0 + qlen + sum(alens)
        sri[0, 0, g0:g0 + qlen] = gend
        a0 = g0 + qlen
        for alen in alens:
            sri[0, 0, a0:a0 + alen] = a0 + alen
            sri[0, 1, a0:a0 + alen] = gend
            a0 += alen
    return sri


def bidir_prefix_intervals(cu: np.ndarray, kinds, total: int, alt: bool = False) -> np.ndarray:
    """Mix of bidirectional documents and prefix-LM documents (non-causal mode).

    Bidirectional document: no row of the document is hidden from any of its
    key columns.  Prefix-LM document with prefix P: prefix columns are visible
    to the whole document, a later column j is visible only to rows >= j.

    ``alt=False`` writes UTS = 0 with UTE = doc start (bidirectional and prefix
    columns) or UTE = j (causal columns).  ``alt=True`` writes an equivalent
    encoding: empty upper intervals UTS = UTE = j for visible columns and
    UTS = doc start, UTE = j for causal columns.
    """
    sri = _default_intervals(total)
    sri[0, 0, :] = _doc_end_per_token(cu, total)
    sri[0, 2, :] = 0
    for s, kind in enumerate(kinds):
        a, b = int(cu[s]), int(cu[s + 1])
        n = b - a
        j = np.arange(a, b, dtype=np.int64)
        if kind == "bidir":
            plen = n
        else:
            plen = n // 4
        if not alt:
            ute = np.where(j < a + plen, a, j)
            sri[0, 3, a:b] = ute
        else:
            vis = j < a + plen
            sri[0, 2, a:b] = np.where(vis, j, a)
            sri[0, 3, a:b] = j
    return sri


# ----------------------------------------------------------------------------
# sparsity sweep (PaddleNLP FlashMask article, section 4.3): one segment of T
# tokens, the structure expressed only through the column intervals, so every
# block of the T x T grid is classified and the fully masked ones skipped
# ----------------------------------------------------------------------------

def single_segment_causal_documents(doc_lens) -> np.ndarray:
    """Causal document mask over one segment: column j of a document ending at
    e is hidden from rows [e, T); the upper triangle is causal."""
    T = int(sum(doc_lens))
    sri = _default_intervals(T)
    ends = np.repeat(np.cumsum(doc_lens), doc_lens)
    sri[0, 0, :] = ends
    return sri


def single_segment_documents(doc_lens) -> np.ndarray:
    """Bidirectional document mask over one segment (non-causal): column j of
    a document [a, e) is hidden from rows [e, T) and [0, a)."""
    T = int(sum(doc_lens))
    sri = _default_intervals(T)
    cum = np.cumsum(doc_lens)
    sri[0, 0, :] = np.repeat(cum, doc_lens)
    sri[0, 2, :] = 0
    sri[0, 3, :] = np.repeat(cum - np.asarray(doc_lens), doc_lens)
    return sri


def single_segment_shared_question(groups) -> np.ndarray:
    """Shared-question mask over one segment (causal): ``groups`` is a list of
    (question_len, [answer_lens]).  Question columns are hidden from rows after
    their group; answer columns from rows after the answer (sibling answers and
    later groups)."""
    T = int(sum(q + sum(a) for q, a in groups))
    sri = _default_intervals(T)
    g0 = 0
    for q, alens in groups:
        gend = g0 + q + sum(alens)
        sri[0, 0, g0:g0 + q] = gend
        a0 = g0 + q
        for a in alens:
            sri[0, 0, a0:a0 + a] = a0 + a
            a0 += a
        g0 = gend
    return sri


def sparsity_sweep(T: int = 16384):
    """The sweep's mask points: (family, parameter, causal, intervals).

    causal_document / document: the segment split into n equal documents,
    n = 1, 2, 4, ..., 64; shared_question: T / 4096 groups of one 1024-token
    question (T / 16 in general) followed by k equal answers, k = 1, 2, 3, 4,
    6, 8, 12.  Sparsity grows with n and with k.
    """
    pts = []
    for n in (1, 2, 4, 8, 16, 32, 64):
        if T % n:
            continue
        lens = [T // n] * n
        pts.append(("causal_document", n, True, single_segment_causal_documents(lens)))
        pts.append(("document", n, False, single_segment_documents(lens)))
    g = T // 4
    q = g // 4
    for k in (1, 2, 3, 4, 6, 8, 12):
        rest = g - q
        alens = [rest // k] * k
        alens[-1] += rest - sum(alens)
        pts.append(("shared_question", k, True, single_segment_shared_question([(q, alens)] * 4)))
    return pts


# ----------------------------------------------------------------------------
# tensors
# ----------------------------------------------------------------------------

def _normal_bf16(rng, shape) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    chunk = 1 << 24
    for i in range(0, n, chunk):
        m = min(chunk, n - i)
        out[i:i + m] = f32_to_bf16_bits(rng.standard_normal(m, dtype=np.float32))
    return out.reshape(shape)


def _attach_tensors(wl: Workload, rng) -> Workload:
    T = wl.total_tokens
    wl.q_bits = _normal_bf16(rng, (T, wl.n_heads_q, wl.head_dim))
    wl.k_bits = _normal_bf16(rng, (T, wl.n_heads_kv, wl.head_dim))
    wl.v_bits = _normal_bf16(rng, (T, wl.n_heads_kv, wl.head_dim))
    return wl


# ----------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------

def make_workload(cfg: int, seed: int = 0, tensors: bool = True,
                  alt_mask: bool = False) -> Workload:
    """Build workload ``cfg`` (1..5) deterministically from ``seed``."""
    rng = np.random.default_rng(seed)
    if cfg == 1:
        lens = [32, 96, 128]
        T = 256
        cu = _cu_from_lens(lens)
        wl = Workload(CONFIG_NAMES[1], T, 1, 1, 64, 1.0e4, True, 64, 64, False,
                      cu, causal_document_intervals(cu, T), ["causal"] * 3)
    elif cfg == 2:
        T = 8192

        def draw():
            if rng.random() < 0.8:
                return rng.integers(64, 512, endpoint=True)
            return rng.integers(2048, 4096, endpoint=True)
        lens = _fill_until_full(rng, T, draw)
        cu = _cu_from_lens(lens)
        wl = Workload(CONFIG_NAMES[2], T, 32, 8, 128, 5.0e5, True, 128, 128, False,
                      cu, causal_document_intervals(cu, T), ["causal"] * len(lens))
    elif cfg == 3:
        while True:
            spec = []
            for _ in range(4):
                ql = int(rng.integers(512, 1536, endpoint=True))
                al = [int(rng.integers(256, 768, endpoint=True)) for _ in range(4)]
                spec.append((ql, al))
            total = sum(ql + sum(al) for ql, al in spec)
            if total <= 16384:
                break
        T = total
        groups = []
        g0 = 0
        glens = []
        for ql, al in spec:
            groups.append((g0, ql, al))
            glens.append(ql + sum(al))
            g0 += ql + sum(al)
        cu = _cu_from_lens(glens)
        wl = Workload(CONFIG_NAMES[3], T, 32, 32, 128, 1.0e4, True, 128, 128, False,
                      cu, shared_question_intervals(groups, T), ["shared_question"] * 4,
                      groups=groups)
    elif cfg == 4:
        T = 16384
        lens = _fill_until_full(rng, T, lambda: rng.integers(256, 4096, endpoint=True))
        cu = _cu_from_lens(lens)
        kinds = ["bidir" if i % 2 == 0 else "prefix_lm" for i in range(len(lens))]
        wl = Workload(CONFIG_NAMES[4], T, 16, 16, 128, 1.0e4, False, 128, 128, False,
                      cu, bidir_prefix_intervals(cu, kinds, T, alt=alt_mask), kinds)
    elif cfg == 5:
        T = 131072
        lens = [65536] + _fill_until_full(rng, T - 65536,
                                          lambda: rng.integers(512, 8192, endpoint=True))
        cu = _cu_from_lens(lens)
        wl = Workload(CONFIG_NAMES[5], T, 32, 8, 128, 1.0e6, True, 128, 128, True,
                      cu, sliding_window_intervals(cu, T, 4096), ["causal_window"] * len(lens))
    else:
        raise ValueError(f"unknown workload {cfg}")
    wl.seed = seed
    if tensors:
        _attach_tensors(wl, rng)
    return wl


def make_custom(lens, n_heads_q=1, n_heads_kv=1, head_dim=64, theta=1.0e4,
                mask="causal_document", causal=True, block_m=128, block_n=128,
                seed=0, window=None, n_mask_heads=1, tensors=True,
                force_int64=False) -> Workload:
    """Small workload with explicit document lengths (tests and edge cases).

    ``mask`` is one of ``none``, ``causal_document``, ``window``,
    ``bidir_prefix`` or ``random``.  ``random`` draws, per mask head and key
    column, arbitrary intervals ``0 <= LTS <= LTE <= T`` and
    ``0 <= UTS <= UTE <= T`` (any column-wise pattern the representation
    allows).
    """
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in lens]
    T = int(sum(lens))
    cu = _cu_from_lens(lens)
    kinds = []
    if mask == "none":
        sri = None
    elif mask == "causal_document":
        sri = causal_document_intervals(cu, T)
    elif mask == "window":
        sri = sliding_window_intervals(cu, T, int(window))
    elif mask == "bidir_prefix":
        kinds = ["bidir" if i % 2 == 0 else "prefix_lm" for i in range(len(lens))]
        sri = bidir_prefix_intervals(cu, kinds, T)
    elif mask == "random":
        sri = np.zeros((n_mask_heads, 4, T), dtype=np.int32)
        for h in range(n_mask_heads):
            for v in (0, 2):
                a = rng.integers(0, T, size=T, endpoint=True)
                b = rng.integers(0, T, size=T, endpoint=True)
                sri[h, v] = np.minimum(a, b)
                sri[h, v + 1] = np.maximum(a, b)
    else:
        raise ValueError(mask)
    wl = Workload(f"custom_{mask}", T, n_heads_q, n_heads_kv, head_dim, theta, causal,
                  block_m, block_n, force_int64, cu, sri, kinds)
    wl.seed = seed
    if tensors:
        _attach_tensors(wl, rng)
    return wl
