"""fp64 oracle: scaled dot-product self-attention over a packed THD batch.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What is computed (written from the pages' definitions, not from any kernel):

* Layout ("How to pad sequences ... context parallelism", repro script): Q, K, V
  are ``[t, h, d]`` tensors; all sequences of the batch are concatenated along
  the token axis.
* Boundaries ("Add per-sequence causal policy ...", ``pad_between_seqs``
  review comment): sequence ``b`` has ``cu_seqlens[b+1] - cu_seqlens[b]``
  valid tokens.  With ``cu_seqlens_padded`` its tokens start at row
  ``cu_seqlens_padded[b]`` of the packed buffer; the rows up to the next start
  are padding.  Without it, sequence ``b`` starts at ``cu_seqlens[b]``.
  Only the first ``batch_size + 1`` entries are read (the slice rule of
  "[PyTorch] Build the attention padding mask ...", Changes).
* Policy ("Add per-sequence causal policy ...", Changes): one boolean per
  sequence.  True selects ``padding_causal`` (key ``j`` visible to query ``i``
  iff ``j <= i``, positions counted from the sequence's first token); False
  selects ``padding`` (every valid key visible).
* Output: for each valid query row ``softmax(scale * q k^T) v`` over the
  visible keys; every row that belongs to no sequence is 0 (the example's
  "0s on pad positions").  The log-sum-exp ``lse = log(sum_j exp(scale*q.k_j))``
  (natural log, scale included) is returned per (head, row), ``-inf`` on pad
  rows and on rows with no visible key.
* Grouped-query heads: query head ``h`` reads key/value head
  ``h // (Hq // Hkv)``.

Arithmetic is fp64 throughout; the inputs are the exact bf16/fp16 values,
upcast.  Query rows are processed in blocks of ``row_block`` with a plain
matrix product (numpy ``@``): no online softmax, no reordering of the
definition beyond the standard max-shift used to evaluate ``exp`` safely.
"""
from __future__ import annotations

import numpy as np


def _as64(x):
    if hasattr(x, "detach"):  # torch tensor -> numpy without importing torch here
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def sequence_spans(cu_seqlens, cu_seqlens_padded, batch_size):
    """(start_row, length) of every sequence; reads only entries 0..batch_size."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)[: batch_size + 1]
    lengths = cu[1:] - cu[:-1]
    if cu_seqlens_padded is None:
        starts = cu[:-1].copy()
    else:
        starts = np.asarray(cu_seqlens_padded, dtype=np.int64)[:batch_size].copy()
    return starts, lengths


def _one_sequence(q, k, v, causal, scale, row_ids=None):
    """softmax(scale q k^T [+ causal]) v for one (sequence, head).

    q: [L, d], k/v: [L, d] fp64.  ``row_ids`` selects query rows (default all).
    Returns (out [n, d], lse [n]).
    """
    L = k.shape[0]
    rows = np.arange(q.shape[0]) if row_ids is None else np.asarray(row_ids)
    z = scale * (q[rows] @ k.T)                     # [n, L] logits
    if causal:
        visible = np.arange(L)[None, :] <= rows[:, None]
        z = np.where(visible, z, -np.inf)
    zmax = z.max(axis=1, keepdims=True)
    e = np.exp(z - zmax)
    s = e.sum(axis=1, keepdims=True)
    lse = (zmax + np.log(s))[:, 0]
    out = (e / s) @ v
    return out, lse


def thd_attention_fwd(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                      cu_seqlens_kv_padded, seq_is_causal, batch_size, softmax_scale,
                      row_block=1024):
    """Whole-batch oracle.  Returns (out [T, Hq, d] fp64, lse [Hq, T] fp64).

    ``seq_is_causal`` may be None (every sequence full-context).  Self-attention
    is assumed: ``cu_seqlens_q`` and ``cu_seqlens_kv`` describe the same
    sequences (the lengths must agree).
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    group = Hq // Hkv
    qs, ql = sequence_spans(cu_seqlens_q, cu_seqlens_q_padded, batch_size)
    ks, kl = sequence_spans(cu_seqlens_kv, cu_seqlens_kv_padded, batch_size)
    if not np.array_equal(ql, kl):
        raise ValueError("oracle covers self-attention: q and kv lengths must agree")
    flags = (np.zeros(batch_size, dtype=bool) if seq_is_causal is None
             else np.asarray(seq_is_causal)[:batch_size].astype(bool))
    out = np.zeros((T, Hq, d), dtype=np.float64)
    lse = np.full((Hq, T), -np.inf, dtype=np.float64)
    for b in range(batch_size):
        L = int(ql[b])
        if L <= 0:
            continue
        s0, k0 = int(qs[b]), int(ks[b])
        for h in range(Hq):
            g = h // group
            kk = k[k0:k0 + L, g, :]
            vv = v[k0:k0 + L, g, :]
            qq = q[s0:s0 + L, h, :]
            for r0 in range(0, L, row_block):
                rows = np.arange(r0, min(L, r0 + row_block))
                o, m = _one_sequence(qq, kk, vv, bool(flags[b]), softmax_scale, rows)
                out[s0 + rows, h, :] = o
                lse[h, s0 + rows] = m
    return out, lse


def thd_attention_rows(q, k, v, start_q, start_kv, length, causal, head, group,
                       softmax_scale, row_ids, window=(-1, -1)):
    """Oracle values for selected query rows of one (sequence, head).

    Used to check full-size batches on sampled rows.  ``row_ids`` are positions
    inside the sequence (0-based).  ``q``/``k``/``v`` are the full packed
    tensors (torch or numpy).  ``window``: (left, right) as in ``visible_range``
    (top-left causal or full, equal query and key lengths).  Returns
    (out [n, d], lse [n]) in fp64.
    """
    g = head // group
    rows = np.asarray(row_ids, dtype=np.int64)
    qq = _as64(q[start_q + rows, head, :])
    kk = _as64(k[start_kv:start_kv + length, g, :])
    vv = _as64(v[start_kv:start_kv + length, g, :])
    z = softmax_scale * (qq @ kk.T)
    if tuple(window) != (-1, -1):
        code = MASK_PADDING_CAUSAL if causal else MASK_PADDING
        band = np.array([visible_range(int(i), length, length, code, window) for i in rows])
        keys = np.arange(length)[None, :]
        z = np.where((keys >= band[:, :1]) & (keys < band[:, 1:]), z, -np.inf)
    elif causal:
        z = np.where(np.arange(length)[None, :] <= rows[:, None], z, -np.inf)
    zmax = z.max(axis=1, keepdims=True)
    e = np.exp(z - zmax)
    s = e.sum(axis=1, keepdims=True)
    return (e / s) @ vv, (zmax + np.log(s))[:, 0]


# ---------------------------------------------------------------------------------------------
# General form: separate query / key-value sequences and a per-sequence mask type.
# ---------------------------------------------------------------------------------------------

MASK_PADDING = 0                  # every valid key visible
MASK_PADDING_CAUSAL = 1           # top-left: key j visible to query i iff j <= i
MASK_PADDING_CAUSAL_BOTTOM_RIGHT = 2   # key j visible iff j <= i + (Lkv - Lq)


def visible_keys(i, Lq, Lkv, mask_type):
    """Number of visible keys (a prefix of the key sequence) for query position i.

    The mask types are the ones the per-sequence policy review comment of "Add
    per-sequence causal policy to packed THD attention" lists (padding,
    padding_causal, padding_causal_bottom_right).  Any code other than 0 and 2 means
    top-left causal, so a boolean flag keeps its meaning.
    """
    if mask_type == MASK_PADDING:
        return Lkv
    shift = (Lkv - Lq) if mask_type == MASK_PADDING_CAUSAL_BOTTOM_RIGHT else 0
    return int(min(Lkv, max(0, i + shift + 1)))


def visible_range(i, Lq, Lkv, mask_type, window=(-1, -1)):
    """Keys [lo, hi) of a sequence visible to query position i, with a sliding window.

    The pages name sliding windows only as an option the per-sequence policy PR rejects
    ("Add per-sequence causal policy to packed THD attention", Changes); the window is read
    here as a band around the diagonal the sequence's mask type uses: with
    shift = Lkv - Lq for bottom-right alignment and 0 otherwise, key j is visible iff it is
    visible under the mask type (visible_keys) and
        i + shift - left <= j <= i + shift + right,
    a negative ``left`` / ``right`` leaving that side unbounded.  (-1, -1) is no window.
    Returns (lo, hi) with lo == hi when no key is visible.
    """
    left, right = int(window[0]), int(window[1])
    hi = visible_keys(i, Lq, Lkv, mask_type)
    shift = (Lkv - Lq) if mask_type == MASK_PADDING_CAUSAL_BOTTOM_RIGHT else 0
    if right >= 0:
        hi = min(hi, max(0, i + shift + right + 1))
    lo = max(0, i + shift - left) if left >= 0 else 0
    return lo, max(lo, hi)


def thd_attention_fwd_general(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                              cu_seqlens_kv_padded, mask_type, batch_size, softmax_scale,
                              window=(-1, -1)):
    """Packed attention with separate query and key/value sequences.

    Query sequence b is rows [sq_b, sq_b + Lq_b) of q, its key/value sequence rows
    [sk_b, sk_b + Lkv_b) of k and v (same packing rules as thd_attention_fwd).  Query i
    sees the keys visible_range(i, ...) of its sequence (a prefix, visible_keys, without
    a window).  Rows that see no key, and rows of no sequence, get out = 0 and lse = -inf.
    mask_type: per-sequence codes (None = all MASK_PADDING).  window: (left, right), see
    visible_range.  Returns (out [Tq, Hq, d], lse [Hq, Tq]) in fp64.
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    Tq, Hq, d = q.shape
    group = Hq // k.shape[1]
    qs, ql = sequence_spans(cu_seqlens_q, cu_seqlens_q_padded, batch_size)
    ks, kl = sequence_spans(cu_seqlens_kv, cu_seqlens_kv_padded, batch_size)
    codes = (np.zeros(batch_size, dtype=np.int64) if mask_type is None
             else np.asarray(mask_type)[:batch_size].astype(np.int64))
    out = np.zeros((Tq, Hq, d), dtype=np.float64)
    lse = np.full((Hq, Tq), -np.inf, dtype=np.float64)
    for b in range(batch_size):
        Lq, Lkv = int(ql[b]), int(kl[b])
        if Lq <= 0:
            continue
        ranges = [visible_range(i, Lq, max(Lkv, 0), int(codes[b]), window) for i in range(Lq)]
        for h in range(Hq):
            g = h // group
            qq = q[qs[b]:qs[b] + Lq, h, :]
            kk = k[ks[b]:ks[b] + max(Lkv, 0), g, :]
            vv = v[ks[b]:ks[b] + max(Lkv, 0), g, :]
            for i in range(Lq):
                lo, hi = ranges[i]
                if hi == lo:
                    continue
                z = softmax_scale * (kk[lo:hi] @ qq[i])
                zmax = z.max()
                e = np.exp(z - zmax)
                s = e.sum()
                out[qs[b] + i, h, :] = (e / s) @ vv[lo:hi]
                lse[h, qs[b] + i] = zmax + np.log(s)
    return out, lse


def merge_partials(out_a, lse_a, out_b, lse_b):
    """Attention over the union of two disjoint key sets, from the attention over each.

    With S = exp(lse_a) + exp(lse_b):  lse = log S and
    out = exp(lse_a - lse) out_a + exp(lse_b - lse) out_b.  A partial with lse = -inf saw no
    key and has weight 0; when both are -inf the row is out = 0, lse = -inf.  Layouts:
    out [T, H, d], lse [H, T].  This is the combination the two-call pad_between_seqs
    example relies on (each call's rows have -inf where the other call has values).
    """
    out_a, out_b = _as64(out_a), _as64(out_b)
    lse_a = np.asarray(lse_a, dtype=np.float64)
    lse_b = np.asarray(lse_b, dtype=np.float64)
    lse = np.logaddexp(lse_a, lse_b)
    both = np.isneginf(lse)
    safe = np.where(both, 0.0, lse)
    wa = np.where(np.isneginf(lse_a), 0.0, np.exp(lse_a - safe))
    wb = np.where(np.isneginf(lse_b), 0.0, np.exp(lse_b - safe))
    out = wa.T[:, :, None] * out_a + wb.T[:, :, None] * out_b
    return out, lse


# ---------------------------------------------------------------------------------------------
# Backward: gradients of the packed attention with respect to Q, K and V.
# ---------------------------------------------------------------------------------------------

def thd_attention_bwd(q, k, v, dout, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                      cu_seqlens_kv_padded, mask_type, batch_size, softmax_scale, window=(-1, -1)):
    """dQ, dK, dV of out = softmax(scale q k^T [masked]) v for every sequence and head.

    "Add per-sequence causal policy to packed THD attention" (Changes, Validation) checks
    Q/K/V gradient parity against scalar-policy attention; this is the gradient of the
    forward defined above, written out from the chain rule (fp64):

        P = softmax(Z) row-wise, Z = scale q k^T with invisible keys at -inf
        dV = P^T dO,  dP = dO V^T,  dZ = P * (dP - rowsum(P * dP)),
        dQ = scale dZ K,  dK = scale dZ^T Q.

    Grouped-query heads: dK / dV of a key/value head sum the contributions of every query
    head that reads it.  Rows of no sequence, rows that see no key and keys no query sees
    get zero gradient.  window: (left, right) as in visible_range.  Returns
    (dq [Tq,Hq,d], dk [Tkv,Hkv,d], dv [Tkv,Hkv,d]) in fp64.
    """
    q, k, v, dout = _as64(q), _as64(k), _as64(v), _as64(dout)
    Tq, Hq, d = q.shape
    Hkv = k.shape[1]
    group = Hq // Hkv
    qs, ql = sequence_spans(cu_seqlens_q, cu_seqlens_q_padded, batch_size)
    ks, kl = sequence_spans(cu_seqlens_kv, cu_seqlens_kv_padded, batch_size)
    codes = (np.zeros(batch_size, dtype=np.int64) if mask_type is None
             else np.asarray(mask_type)[:batch_size].astype(np.int64))
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(batch_size):
        Lq, Lkv = int(ql[b]), int(kl[b])
        if Lq <= 0 or Lkv <= 0:
            continue
        ranges = np.array([visible_range(i, Lq, Lkv, int(codes[b]), window) for i in range(Lq)])
        keys = np.arange(Lkv)[None, :]
        visible = (keys >= ranges[:, :1]) & (keys < ranges[:, 1:])
        rows = ranges[:, 1] > ranges[:, 0]
        sq, sk = slice(qs[b], qs[b] + Lq), slice(ks[b], ks[b] + Lkv)
        for h in range(Hq):
            g = h // group
            Q, K, V, dO = q[sq, h, :], k[sk, g, :], v[sk, g, :], dout[sq, h, :]
            Z = np.where(visible, softmax_scale * (Q @ K.T), -np.inf)
            P = np.zeros_like(Z)
            Zr = Z[rows]
            E = np.exp(Zr - Zr.max(axis=1, keepdims=True))
            P[rows] = E / E.sum(axis=1, keepdims=True)
            dP = dO @ V.T
            dZ = P * (dP - (P * dP).sum(axis=1, keepdims=True))
            dq[sq, h, :] = softmax_scale * (dZ @ K)
            dk[sk, g, :] += softmax_scale * (dZ.T @ Q)
            dv[sk, g, :] += P.T @ dO
    return dq, dk, dv


def thd_attention_bwd_dq_rows(q, k, v, dout, start_q, start_kv, length, causal, head, group,
                              softmax_scale, row_ids):
    """dQ of selected query rows of one (sequence, head), for full-size batches checked on
    sampled rows: the gradient of ``thd_attention_rows``'s output, written out row by row from
    the same chain rule as ``thd_attention_bwd`` (a query row's dQ depends on that row and on
    the sequence's keys and values only):

        z_j = scale q_i . k_j (visible j),  p = softmax(z),  dp_j = dO_i . v_j,
        dz_j = p_j (dp_j - sum_l p_l dp_l),  dQ_i = scale sum_j dz_j k_j.

    ``row_ids`` are positions inside the sequence; returns dq [n, d] in fp64.
    """
    g = head // group
    rows = np.asarray(row_ids, dtype=np.int64)
    qq = _as64(q[start_q + rows, head, :])
    oo = _as64(dout[start_q + rows, head, :])
    kk = _as64(k[start_kv:start_kv + length, g, :])
    vv = _as64(v[start_kv:start_kv + length, g, :])
    z = softmax_scale * (qq @ kk.T)
    if causal:
        z = np.where(np.arange(length)[None, :] <= rows[:, None], z, -np.inf)
    e = np.exp(z - z.max(axis=1, keepdims=True))
    p = e / e.sum(axis=1, keepdims=True)
    dp = oo @ vv.T
    dz = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    return softmax_scale * (dz @ kk)
