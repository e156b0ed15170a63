"""Float64 CPU oracle for packed variable-length FlashMask attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import,
call or execute anything in this package.  The product (the CUDA library and
its Python binding) never imports it and has no CPU fallback.

The oracle computes each step from its plain definition, slowly and in
float64, and shares no code with the CUDA path (no kernels, headers,
helpers, constants or pre/post-processing).  Its only common dependency is
the seeded input generator in ``workloads`` (random numbers and document /
mask layouts, no method arithmetic).

Sources, cited by page title and section:

* Unsloth, "3x faster LLM training with Unsloth kernels + packing" (Chinese
  edition): section "Fused QK RoPE Triton kernel with packing" (RoPE as
  ``Q*cos + rotate_half(Q)*sin`` with ``rotate_half(Q) = Q @ R``,
  ``R = [[0, I], [-I, 0]]``, and the backward rule ``sin -> -sin``);
  section "Uncontaminated packing" (positions reset for every packed
  sample); section "Why padding is needed and the maths of the speedup".
* "PaddleNLP FlashMask in practice" article: section 3.4 (the backward
  operator's inputs and outputs); section 2.1 (column-wise
  intervals ``[start_j, end_j)``), section 2.2 (the LTS/LTE/UTS/UTE vectors,
  their defaults and the 16x16 causal example), section 3.1 (the eight
  per-tile min/max vectors), section 3.2 (the three block classes), section
  3.3 (exact equivalence with dense-mask attention), section 4.3 (block
  sparsity).
* "Varlen-Packing technical document": section 1.3 (Q-tile / KV-tile
  tiling), section 2 (the varlen 3-D grid and its [128, 128, 4096] example),
  section 3.1 (padded token counts).

Readings where the pages are silent or garbled are stated in each function's
docstring.

Parity status per function (what pins it, besides itself):

* ``rope.rope_apply`` / ``rope.rope_backward``: pinned (identity at position
  0, complex-rotation restatement, round trip, finite differences).
* ``mask.dense_mask``: pinned (16x16 worked table, brute-force enumeration).
* ``mask.block_minmax``: pinned (the worked example's first tile).
* ``mask.classify_block`` / ``mask.block_class_counts``: pinned (the three
  printed examples, soundness against the dense mask).
* ``attention.attention_forward``: pinned (single key, textbook softmax via
  scipy, brute-force loop on tiny inputs, encoding invariants).
* ``packing``: pinned (the printed closed forms and token / CTA counts).
* ``attention_bwd.attention_backward``: pinned (central finite differences of
  ``attention_forward`` for six mask styles with GQA, fully masked rows, a
  closed form); ``attention_bwd.row_delta``: pinned (sum of p times dp).
"""

from . import attention, attention_bwd, mask, packing, rope  # noqa: F401
