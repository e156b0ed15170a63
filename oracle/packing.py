"""Token and launch counts of padded versus packed batches (test infrastructure).

Unsloth packing blog, section "Why padding is needed and the maths of the
speedup": a padded batch stores ``batch * max_len`` tokens, a packed one
only the real tokens; with half long (L) and half short (S) samples the
ratio is ``2 L / (L + S)``.

Varlen-Packing technical document, section 2: a varlen FlashAttention
launch uses the grid ``(seq_count, n_head, ceil(max_seq_len / Br))``;
section 3.1: padding every sample to the longest one.  A launch over only
the real Q tiles of each sample needs ``n_head * sum_s ceil(len_s / Br)``
thread blocks.
"""

from __future__ import annotations

import math
from typing import Sequence


def padded_tokens(lengths: Sequence[int]) -> int:
    return len(lengths) * max(lengths)


def packed_tokens(lengths: Sequence[int]) -> int:
    return int(sum(lengths))


def padding_speedup(lengths: Sequence[int]) -> float:
    """Tokens processed padded divided by tokens processed packed."""
    return padded_tokens(lengths) / packed_tokens(lengths)


def varlen_grid_blocks(lengths: Sequence[int], n_head: int, block_m: int) -> int:
    """Thread blocks of the fixed 3-D varlen grid."""
    return len(lengths) * n_head * math.ceil(max(lengths) / block_m)


def real_q_tiles(lengths: Sequence[int], n_head: int, block_m: int) -> int:
    """Work items when only every sample's real Q tiles are launched."""
    return n_head * sum(math.ceil(n / block_m) for n in lengths if n > 0)
