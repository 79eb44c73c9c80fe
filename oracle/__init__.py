"""fp64 CPU oracle for packed variable-length (THD) attention and its padding mask.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously-correct
statement of what the CUDA library computes.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference arm of ``bench.py``
may import it.  The product path (``variable_length_packed_gb300``) never
imports, calls or links anything here, and this package imports nothing from
the product: the two share only the seeded input generators in ``workloads``.

Sources followed (web pages; titles and sections):

* "How to pad sequences that cannot be evenly split in context parallelism (CP)?"
  (Megatron-LM issue): the THD layout, ``cu_seqlens``, the ``padding`` mask type
  and the printed full-attention output of the 7-token constant example.
* "Add per-sequence causal policy to packed THD attention" (TransformerEngine
  PR): ``thd_sequence_is_causal`` (Changes), the ``[111aaa222bb3344cccc]``
  example and the two-call ``cu_seqlens`` / ``cu_seqlens_padded`` arrays of the
  ``pad_between_seqs`` review comment.
* "[PyTorch] Build the attention padding mask without host syncs"
  (TransformerEngine PR): the old per-sequence loop and the vectorised
  ``positions >= seqlens`` form (Description), the ``[1 : batch_size + 1]``
  slice (Changes) and the invalid-input rule (Equivalence).

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(closed forms, the pages' printed values, a library routine, brute force and
case counts).  Nothing is "parity unpinned".
"""
from .attention import (thd_attention_fwd, thd_attention_rows, sequence_spans, thd_attention_fwd_general,
                        merge_partials, visible_keys, visible_range, thd_attention_bwd,
                        thd_attention_bwd_dq_rows, MASK_PADDING,
                        MASK_PADDING_CAUSAL, MASK_PADDING_CAUSAL_BOTTOM_RIGHT)
from .mask import (padding_mask_loop, padding_mask_formula, padding_mask_cross_loop,
                   padding_mask_cross_formula)

__all__ = [
    "thd_attention_fwd",
    "thd_attention_rows",
    "thd_attention_bwd_dq_rows",
    "sequence_spans",
    "thd_attention_fwd_general",
    "merge_partials",
    "thd_attention_bwd",
    "visible_keys",
    "visible_range",
    "MASK_PADDING",
    "MASK_PADDING_CAUSAL",
    "MASK_PADDING_CAUSAL_BOTTOM_RIGHT",
    "padding_mask_loop",
    "padding_mask_formula",
    "padding_mask_cross_loop",
    "padding_mask_cross_formula",
]
