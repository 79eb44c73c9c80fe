"""fp64-free oracle for the attention padding mask (integer work).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: "[PyTorch] Build the attention padding mask without host syncs"
(TransformerEngine PR).  The mask is boolean ``[batch, 1, 1, max_seqlen]``;
True marks a padded position.  Two forms are kept, both written here from the
page's description:

* ``padding_mask_loop``: the old construction (Description): per sequence,
  ``seqlen`` False entries followed by ``max_seqlen - seqlen`` True entries,
  the rows stacked over ``range(batch_size)``.  Like the old code it cannot
  build a row longer than ``max_seqlen`` (Equivalence: it raised), so it
  raises ``ValueError`` there.
* ``padding_mask_formula``: the vectorised definition (Description):
  ``seqlens = cu[1:B+1] - cu[:B]`` and ``mask[b, p] = p >= seqlens[b]``.  The
  slice reads exactly ``batch_size + 1`` entries, so a longer buffer's tail is
  ignored (Changes).  A sequence longer than ``max_seqlen`` gives an all-False
  row (Equivalence).
"""
from __future__ import annotations

import numpy as np


def padding_mask_loop(cu_seqlens, batch_size, max_seqlen):
    cu = [int(x) for x in np.asarray(cu_seqlens).tolist()]
    rows = []
    for b in range(batch_size):
        n = cu[b + 1] - cu[b]
        row = [False] * n + [True] * (max_seqlen - n)
        if len(row) != max_seqlen:
            raise ValueError(f"sequence {b} has length {n} outside [0, {max_seqlen}]")
        rows.append(row)
    return np.array(rows, dtype=bool).reshape(batch_size, 1, 1, max_seqlen)


def padding_mask_formula(cu_seqlens, batch_size, max_seqlen):
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    seqlens = cu[1:batch_size + 1] - cu[:batch_size]
    positions = np.arange(max_seqlen, dtype=np.int64)
    mask = positions[None, :] >= seqlens[:, None]
    return mask.reshape(batch_size, 1, 1, max_seqlen)


def padding_mask_cross_loop(cu_seqlens_q, cu_seqlens_kv, batch_size, max_seqlen_q, max_seqlen_kv):
    """Cross-attention form (Equivalence section: q and kv lengths): the pair of masks
    (query positions, key positions), each built by the old loop."""
    return (padding_mask_loop(cu_seqlens_q, batch_size, max_seqlen_q),
            padding_mask_loop(cu_seqlens_kv, batch_size, max_seqlen_kv))


def padding_mask_cross_formula(cu_seqlens_q, cu_seqlens_kv, batch_size, max_seqlen_q, max_seqlen_kv):
    return (padding_mask_formula(cu_seqlens_q, batch_size, max_seqlen_q),
            padding_mask_formula(cu_seqlens_kv, batch_size, max_seqlen_kv))
