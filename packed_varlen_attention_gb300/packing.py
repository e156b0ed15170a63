"""Host-side packing and collation for the packed variable-length path.

What the pages describe:

* Unsloth packing blog ("padding-free packing"): variable-length samples are
  concatenated into one 1-D token tensor and their lengths kept as metadata,
  so attention never crosses a sample boundary and positions restart at every
  sample (the RoPE kernel derives the positions from ``cu_seqlens``).
* PaddleNLP FlashMask article, section 6.4: with ``zero_padding`` /
  ``greedy_zero_padding`` the data side builds the column intervals
  ``startend_row_indices`` (O(N) per sample) instead of a dense mask, and
  section 6.7: when a batch is concatenated, every sample's row indices are
  shifted by the running token offset (``sequence_sum``), turning the
  per-sample intervals into global row coordinates of the pack.
* FlashMask article, section 2.2: four vectors LTS, LTE, UTS, UTE per key
  column; an omitted LTS/UTS defaults to 0 and an omitted LTE/UTE to the
  query length.

Everything here is plain NumPy on the host; the packed arrays it returns are
what ``rope_qk_varlen``, ``mask_block_minmax`` and ``attn_fwd_varlen`` take
(after moving them to the device).
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np

__all__ = [
    "Packed",
    "greedy_pack",
    "collate",
    "intervals_causal",
    "intervals_bidirectional",
    "intervals_prefix_lm",
    "intervals_shared_question",
    "intervals_sliding_window",
]


# ---------------------------------------------------------------------------
# packing
# ---------------------------------------------------------------------------

def greedy_pack(lengths: Sequence[int], max_tokens: int,
                longest_first: bool = False) -> List[List[int]]:
    """Assigns samples to packs of at most ``max_tokens`` tokens.

    First fit: each sample (in input order, or longest first when
    ``longest_first``) goes into the first pack that still has room for it;
    a new pack is opened when none has.  Returns the sample indices of every
    pack in the order they were placed.  A sample longer than ``max_tokens``
    or a negative length raises ``ValueError``.
    """
    if max_tokens <= 0:
        raise ValueError("max_tokens must be positive")
    lens = [int(n) for n in lengths]
    for i, n in enumerate(lens):
        if n < 0:
            raise ValueError(f"sample {i} has negative length {n}")
        if n > max_tokens:
            raise ValueError(f"sample {i} ({n} tokens) does not fit in a pack of {max_tokens}")
    order = sorted(range(len(lens)), key=lambda i: (-lens[i], i)) if longest_first \
        else list(range(len(lens)))
    packs: List[List[int]] = []
    room: List[int] = []
    for i in order:
        for p, r in enumerate(room):
            if lens[i] <= r:
                packs[p].append(i)
                room[p] -= lens[i]
                break
        else:
            packs.append([i])
            room.append(max_tokens - lens[i])
    return packs


# ---------------------------------------------------------------------------
# per-sample column intervals (local row coordinates 0 .. n)
# ---------------------------------------------------------------------------

def _full(n: int, lts, lte, uts, ute) -> np.ndarray:
    out = np.empty((1, 4, n), dtype=np.int32)
    out[0, 0], out[0, 1], out[0, 2], out[0, 3] = lts, lte, uts, ute
    return out


def intervals_causal(n: int) -> np.ndarray:
    """Causal attention within the sample (use with ``causal=True``): nothing
    is masked below the diagonal, the upper triangle is masked."""
    return _full(n, n, n, 0, np.arange(n))


def intervals_bidirectional(n: int) -> np.ndarray:
    """Full (bidirectional) attention within the sample (``causal=False``)."""
    return _full(n, n, n, 0, 0)


def intervals_prefix_lm(n: int, prefix: int) -> np.ndarray:
    """Prefix-LM (``causal=False``): the first ``prefix`` tokens see each
    other in both directions, the rest attend causally."""
    if not 0 <= prefix <= n:
        raise ValueError("prefix must lie in [0, n]")
    j = np.arange(n)
    ute = np.where(j < prefix, 0, j)  # upper rows [0, j) masked outside the prefix
    return _full(n, n, n, 0, ute)


def intervals_shared_question(prompt: int, answers: Sequence[int]) -> np.ndarray:
    """DPO / reward-model sample: one prompt followed by several answers
    (``causal=True``).  Every answer attends causally to the prompt and to
    itself, never to another answer: below the diagonal, an answer's columns
    are masked for every row after the end of that answer."""
    ans = [int(a) for a in answers]
    if prompt < 0 or any(a < 0 for a in ans):
        raise ValueError("lengths must be non-negative")
    n = prompt + sum(ans)
    lts = np.full(n, n, dtype=np.int64)
    end = prompt
    for a in ans:
        lts[end:end + a] = end + a
        end += a
    return _full(n, lts, n, 0, np.arange(n))


def intervals_sliding_window(n: int, window: int) -> np.ndarray:
    """Causal attention limited to the last ``window`` keys (``causal=True``):
    row i sees column j iff j <= i < j + window."""
    if window <= 0:
        raise ValueError("window must be positive")
    j = np.arange(n)
    return _full(n, np.minimum(j + window, n), n, 0, j)


# ---------------------------------------------------------------------------
# collation
# ---------------------------------------------------------------------------

@dataclass
class Packed:
    """One packed batch.

    tokens                 the samples concatenated along axis 0
    cu_seqlens             int32 [n_samples + 1], cu_seqlens[0] = 0
    startend_row_indices   int32 [n_mask_heads, 4, T] in global row
                           coordinates, or None when no sample gave any
    """
    tokens: np.ndarray
    cu_seqlens: np.ndarray
    startend_row_indices: Optional[np.ndarray]

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def n_seqs(self) -> int:
        return len(self.cu_seqlens) - 1


def _expand_local(sri: Optional[np.ndarray], n: int, n_mask_heads: int) -> np.ndarray:
    """A sample's intervals as [n_mask_heads, 4, n] local coordinates.

    ``sri`` may be None (no interval mask: nothing masked below the diagonal,
    the whole upper triangle masked), or have shape [k, n] or [h, k, n] with
    k = 1 (LTS), 2 (LTS, LTE) or 4 (LTS, LTE, UTS, UTE) and h = 1 or
    ``n_mask_heads``; omitted vectors take the defaults LTE = UTE = n,
    UTS = 0.
    """
    out = np.empty((n_mask_heads, 4, n), dtype=np.int64)
    out[:, 0] = 0
    out[:, 1] = n
    out[:, 2] = 0
    out[:, 3] = n
    if sri is None:
        out[:, 0] = n
        return out
    a = np.asarray(sri)
    if a.ndim == 2:
        a = a[None]
    if a.ndim != 3 or a.shape[2] != n or a.shape[1] not in (1, 2, 4):
        raise ValueError(f"intervals of shape {np.shape(sri)} do not match a sample of {n} tokens")
    if a.shape[0] not in (1, n_mask_heads):
        raise ValueError("intervals must have 1 or n_mask_heads heads")
    k = a.shape[1]
    out[:, :k] = a
    if np.any(out < 0) or np.any(out > n):
        raise ValueError("interval bounds must lie in [0, sample length]")
    return out


def collate(samples: Sequence[np.ndarray],
            intervals: Optional[Sequence[Optional[np.ndarray]]] = None,
            n_mask_heads: int = 1) -> Packed:
    """Concatenates samples into one pack.

    ``samples[i]`` is any array whose axis 0 runs over the sample's tokens
    (token ids, or [n, heads, head_dim] activations).  ``intervals[i]`` are
    the sample's column intervals in its own row coordinates (see
    ``_expand_local``); each is shifted by the sample's token offset, so the
    result is in global row coordinates of the pack.  With ``intervals``
    None the pack carries no interval mask (attention is still restricted to
    each sample by ``cu_seqlens``).
    """
    if n_mask_heads < 1:
        raise ValueError("n_mask_heads must be >= 1")
    lens = [int(np.shape(x)[0]) for x in samples]
    cu = np.zeros(len(lens) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lens)
    if cu[-1] >= 2 ** 31:
        raise ValueError("a pack is limited to 2^31 - 1 tokens")
    tokens = np.concatenate([np.asarray(x) for x in samples], axis=0) if samples \
        else np.zeros((0,), dtype=np.int64)
    sri = None
    if intervals is not None:
        if len(intervals) != len(samples):
            raise ValueError("one interval entry per sample")
        T = int(cu[-1])
        sri = np.empty((n_mask_heads, 4, T), dtype=np.int32)
        for s, (n, iv) in enumerate(zip(lens, intervals)):
            local = _expand_local(iv, n, n_mask_heads)
            sri[:, :, cu[s]:cu[s + 1]] = local + cu[s]  # the sequence_sum shift
    return Packed(tokens=tokens, cu_seqlens=cu.astype(np.int32), startend_row_indices=sri)
