"""FlashMask column intervals, block statistics and block classes, float64/int.

TEST INFRASTRUCTURE ONLY (see the package docstring).

PaddleNLP FlashMask article:

* section 2.1: the masked rows of key column j form one contiguous interval
  ``[start_j, end_j)``;
* section 2.2: two intervals per column split by the diagonal, lower
  triangle ``[LTS_j, LTE_j)`` and upper triangle ``[UTS_j, UTE_j)``;
  defaults LTS = UTS = 0 and LTE = UTE = query length;
* section 3.1: per key tile (the FlashAttention column tile), the minimum and
  maximum of each vector, eight vectors in all;
* section 3.2: a (row tile, column tile) block is fully masked, partially
  masked or unmasked, decided from those eight numbers.

Readings:

1. The intervals apply only inside their own triangle: element (i, j) with
   i >= j (diagonal included) is masked iff ``LTS_j <= i < LTE_j``; with
   i < j it is masked iff ``UTS_j <= i < UTE_j``.  Causal mode masks the whole
   upper triangle regardless of UTS/UTE.  With the defaults this makes
   UTS = 0, UTE = N the full upper triangle, as the article implies.
2. Attention is also restricted to the packed sample (block-diagonal by
   ``cu_seqlens``); cross-sample pairs are masked.  Indices are global row
   coordinates of the packed tensor.
3. Tiles are sample-local: the row tile ``qt`` of sample s covers rows
   ``[cu[s] + qt*Br, min(cu[s] + (qt+1)*Br, cu[s+1]))``, the same for columns.
4. The comparison signs of section 3.2 are garbled in the page.  With rows
   ``[r0, r1)`` (r1 exclusive) the classes are: lower part fully masked iff
   ``r0 >= LTS_max and r1 <= LTE_min``; lower part touched iff
   ``r0 < LTE_max and r1 > LTS_min``; likewise for the upper part (always
   full and touched in causal mode).  A block entirely below the diagonal
   (``r0 >= c1 - 1``) takes the lower part's class, one entirely above
   (``r1 - 1 < c0``) the upper part's; a block the diagonal crosses is fully
   masked only if both parts are, partially masked if causal or either part
   is touched, unmasked otherwise.  This reproduces all three examples the
   article prints.  "Partially masked" is conservative (it may hold no
   masked element); "fully masked" and "unmasked" are always exact.
"""

from __future__ import annotations

from typing import Optional

import numpy as np

FULL, PARTIAL, UNMASKED = "F", "P", "U"


def dense_mask(sri_h: Optional[np.ndarray], rows: np.ndarray, cols: np.ndarray,
               causal: bool) -> np.ndarray:
    """Boolean [len(rows), len(cols)], True where (row, col) is masked.

    ``sri_h`` is the int array [4][T] (LTS, LTE, UTS, UTE) of one mask head,
    or None for no interval mask.  ``rows`` / ``cols`` are global indices of
    one packed sample (the caller applies the sample restriction).
    """
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.asarray(cols, dtype=np.int64)[None, :]
    lower = i >= j
    if sri_h is None:
        lt = np.zeros(lower.shape, dtype=bool)
        ut = np.zeros(lower.shape, dtype=bool)
    else:
        lts = sri_h[0].astype(np.int64)[j]
        lte = sri_h[1].astype(np.int64)[j]
        uts = sri_h[2].astype(np.int64)[j]
        ute = sri_h[3].astype(np.int64)[j]
        lt = (lts <= i) & (i < lte)
        ut = (uts <= i) & (i < ute)
    if causal:
        ut = np.ones(lower.shape, dtype=bool)
    return np.where(lower, lt, ut)


def tiles(cu_seqlens: np.ndarray, block: int):
    """Sample-local tiles: list of (sample, tile index, start, end)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    out = []
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        t = 0
        for c0 in range(a, b, block):
            out.append((s, t, c0, min(c0 + block, b)))
            t += 1
    return out


def block_minmax(sri: np.ndarray, cu_seqlens: np.ndarray, block_n: int) -> dict:
    """Eight per-tile statistics for every mask head and sample-local tile.

    Returns {(head, sample, tile): (LTS_min, LTS_max, LTE_min, LTE_max,
    UTS_min, UTS_max, UTE_min, UTE_max)}.
    """
    out = {}
    for h in range(sri.shape[0]):
        for s, t, c0, c1 in tiles(cu_seqlens, block_n):
            v = []
            for k in range(4):
                seg = sri[h, k, c0:c1]
                v.append(int(seg.min()))
                v.append(int(seg.max()))
            out[(h, s, t)] = tuple(v)
    return out


def classify_block(r0: int, r1: int, c0: int, c1: int, stats, causal: bool) -> str:
    """Class of the block rows [r0, r1) x cols [c0, c1) (reading 4 above).

    ``stats`` is the eight-number tuple of ``block_minmax`` or None when
    there is no interval mask.
    """
    if stats is None:
        lt_full = lt_touch = False
        ut_full = ut_touch = False
    else:
        lts_min, lts_max, lte_min, lte_max, uts_min, uts_max, ute_min, ute_max = stats
        lt_full = r0 >= lts_max and r1 <= lte_min
        lt_touch = r0 < lte_max and r1 > lts_min
        ut_full = r0 >= uts_max and r1 <= ute_min
        ut_touch = r0 < ute_max and r1 > uts_min
    if causal:
        ut_full = ut_touch = True
    if r1 - 1 < c0:          # entirely above the diagonal
        return FULL if ut_full else (PARTIAL if ut_touch else UNMASKED)
    if r0 >= c1 - 1:         # entirely below (diagonal counts as lower)
        return FULL if lt_full else (PARTIAL if lt_touch else UNMASKED)
    if lt_full and ut_full:
        return FULL
    if causal or lt_touch or ut_touch:
        return PARTIAL
    return UNMASKED


def block_class_counts(cu_seqlens: np.ndarray, sri: Optional[np.ndarray], n_heads_q: int,
                       block_m: int, block_n: int, causal: bool):
    """Counts (F, P, U) over every (sample, q tile, kv tile, q head) block.

    Mask head of q head h is h when there is one mask head per q head,
    else 0.
    """
    stats = None if sri is None else block_minmax(sri, cu_seqlens, block_n)
    n_mask_heads = 0 if sri is None else sri.shape[0]
    rtiles = tiles(cu_seqlens, block_m)
    ctiles = tiles(cu_seqlens, block_n)
    by_sample = {}
    for s, t, c0, c1 in ctiles:
        by_sample.setdefault(s, []).append((t, c0, c1))
    counts = {FULL: 0, PARTIAL: 0, UNMASKED: 0}
    heads = [0] if n_mask_heads <= 1 else list(range(n_heads_q))
    mult = n_heads_q if n_mask_heads <= 1 else 1
    for h in heads:
        for s, _, r0, r1 in rtiles:
            for t, c0, c1 in by_sample.get(s, []):
                st = None if stats is None else stats[(h, s, t)]
                counts[classify_block(r0, r1, c0, c1, st, causal)] += mult
    return counts[FULL], counts[PARTIAL], counts[UNMASKED]
