"""Plant plausible mistakes in the oracle (on the CPU) and check that some pin catches each.

Each mutant replaces one helper of ``oracle.attention`` for the duration of a test;
the pins of ``test_oracle_pins`` are then run and at least one must fail.
"""
import numpy as np
import pytest

import oracle.attention as oa
import test_oracle_pins as pins

PINS = [
    pins.test_page1_printed_values,
    pins.test_page1_closed_form_full,
    pins.test_page1_closed_form_causal,
    pins.test_page1_pad_row_is_zero_and_ignored,
    pins.test_mixed_policy_equals_per_sequence_scalar_policy,
    pins.test_two_call_pad_between_seqs_sum,
    pins.test_brute_force_scalar_loops,
    pins.test_gqa_against_torch_sdpa_fp64,
    pins.test_causal_first_row_is_first_value_and_rows_are_convex,
]


def _softmax_rows(z, v):
    zmax = z.max(axis=1, keepdims=True)
    e = np.exp(z - zmax)
    s = e.sum(axis=1, keepdims=True)
    return (e / s) @ v, (zmax + np.log(s))[:, 0]


def strict_causal(q, k, v, causal, scale, row_ids=None):
    rows = np.arange(q.shape[0]) if row_ids is None else np.asarray(row_ids)
    z = scale * (q[rows] @ k.T)
    if causal:  # mistake: the diagonal is hidden (j < i), row 0 sees nothing
        z = np.where(np.arange(k.shape[0])[None, :] < rows[:, None], z, -1e300)
    return _softmax_rows(z, v)


def no_scale(q, k, v, causal, scale, row_ids=None):
    rows = np.arange(q.shape[0]) if row_ids is None else np.asarray(row_ids)
    z = q[rows] @ k.T   # mistake: scale dropped
    if causal:
        z = np.where(np.arange(k.shape[0])[None, :] <= rows[:, None], z, -np.inf)
    return _softmax_rows(z, v)


def bottom_right(q, k, v, causal, scale, row_ids=None):
    rows = np.arange(q.shape[0]) if row_ids is None else np.asarray(row_ids)
    z = scale * (q[rows] @ k.T)
    if causal:  # mistake: causal mask anchored at the other corner of a rectangular block
        off = k.shape[0] - q.shape[0] + 1
        z = np.where(np.arange(k.shape[0])[None, :] <= rows[:, None] + off, z, -np.inf)
    return _softmax_rows(z, v)


def lse_without_max(q, k, v, causal, scale, row_ids=None):
    out, lse = pins_free_reference(q, k, v, causal, scale, row_ids)
    z = scale * (q @ k.T)
    return out, lse - z.max()  # mistake: the max shift is dropped from the LSE


def pins_free_reference(q, k, v, causal, scale, row_ids=None):
    rows = np.arange(q.shape[0]) if row_ids is None else np.asarray(row_ids)
    z = scale * (q[rows] @ k.T)
    if causal:
        z = np.where(np.arange(k.shape[0])[None, :] <= rows[:, None], z, -np.inf)
    return _softmax_rows(z, v)


def transposed_values(q, k, v, causal, scale, row_ids=None):
    rows = np.arange(q.shape[0]) if row_ids is None else np.asarray(row_ids)
    z = scale * (q[rows] @ k.T)
    if causal:
        z = np.where(np.arange(k.shape[0])[None, :] <= rows[:, None], z, -np.inf)
    o, l = _softmax_rows(z, k)   # mistake: weights applied to K instead of V
    return o, l


def starts_from_cu(cu_seqlens, cu_seqlens_padded, batch_size):
    cu = np.asarray(cu_seqlens, dtype=np.int64)[: batch_size + 1]
    return cu[:-1].copy(), cu[1:] - cu[:-1]   # mistake: padded offsets ignored


@pytest.mark.parametrize("target,mutant", [
    ("_one_sequence", strict_causal),
    ("_one_sequence", no_scale),
    ("_one_sequence", bottom_right),
    ("_one_sequence", lse_without_max),
    ("_one_sequence", transposed_values),
    ("sequence_spans", starts_from_cu),
])
def test_pins_catch_mutant(monkeypatch, target, mutant):
    monkeypatch.setattr(oa, target, mutant)
    failed = 0
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed += 1
    assert failed >= 1, f"no pin caught mutant {mutant.__name__}"


import test_oracle_general as gen

GENERAL_PINS = [
    gen.test_page1_context_parallel_merge_gives_printed_output,
    gen.test_two_call_merge_equals_mixed_call,
    lambda: [gen.test_general_against_torch_sdpa_with_mask(lq, lkv, 2) for lq, lkv in ((5, 9), (9, 5))],
    gen.test_single_query_bottom_right_sees_every_key,
    lambda: gen.test_merge_of_key_split_equals_full(13),
]


def bottom_right_sign_flipped(i, Lq, Lkv, mask_type):
    if mask_type == 0:
        return Lkv
    shift = (Lq - Lkv) if mask_type == 2 else 0   # mistake: offset of the wrong sign
    return int(min(Lkv, max(0, i + shift + 1)))


def merge_unweighted(out_a, lse_a, out_b, lse_b):
    return out_a + out_b, np.logaddexp(lse_a, lse_b)   # mistake: partials not reweighted


@pytest.mark.parametrize("target,mutant", [
    ("visible_keys", bottom_right_sign_flipped),
    ("merge_partials", merge_unweighted),
])
def test_general_pins_catch_mutant(monkeypatch, target, mutant):
    import oracle as pkg
    monkeypatch.setattr(oa, target, mutant)
    monkeypatch.setattr(pkg, target, mutant)
    failed = 0
    for pin in GENERAL_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed += 1
    assert failed >= 1, f"no pin caught mutant {mutant.__name__}"


import test_oracle_window as win

WINDOW_PINS = [
    lambda: [win.test_band_against_torch_tril_triu(lq, lkv, code, w) for lq, lkv in ((11, 11), (6, 13))
             for code in (0, 1, 2) for w in ((3, -1), (-1, 2), (2, 4))],
    lambda: [win.test_zero_width_window_copies_one_value_row(*c) for c in ((9, 9, 0), (5, 12, 2))],
    lambda: win.test_causal_window_is_full_attention_over_the_last_keys(4),
]


def window_lower_off_by_one(i, Lq, Lkv, mask_type, window=(-1, -1)):
    left, right = window
    hi = oa.visible_keys(i, Lq, Lkv, mask_type)
    shift = (Lkv - Lq) if mask_type == 2 else 0
    if right >= 0:
        hi = min(hi, max(0, i + shift + right + 1))
    lo = max(0, i + shift - left + 1) if left >= 0 else 0   # mistake: one key too few on the left
    return lo, max(lo, hi)


def window_upper_exclusive(i, Lq, Lkv, mask_type, window=(-1, -1)):
    left, right = window
    hi = oa.visible_keys(i, Lq, Lkv, mask_type)
    shift = (Lkv - Lq) if mask_type == 2 else 0
    if right >= 0:
        hi = min(hi, max(0, i + shift + right))             # mistake: right edge excluded
    lo = max(0, i + shift - left) if left >= 0 else 0
    return lo, max(lo, hi)


def window_ignores_alignment(i, Lq, Lkv, mask_type, window=(-1, -1)):
    left, right = window
    hi = oa.visible_keys(i, Lq, Lkv, mask_type)
    if right >= 0:
        hi = min(hi, max(0, i + right + 1))                 # mistake: band not moved to the
    lo = max(0, i - left) if left >= 0 else 0               # bottom-right diagonal
    return lo, max(lo, hi)


@pytest.mark.parametrize("mutant", [window_lower_off_by_one, window_upper_exclusive, window_ignores_alignment])
def test_window_pins_catch_mutant(monkeypatch, mutant):
    import oracle as pkg
    monkeypatch.setattr(oa, "visible_range", mutant)
    monkeypatch.setattr(pkg, "visible_range", mutant)
    failed = 0
    for pin in WINDOW_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed += 1
    assert failed >= 1, f"no pin caught mutant {mutant.__name__}"


# ---- the sampled-rows oracles used on full-size batches ----

import test_oracle_bwd as bwd_pins


def _dq_rows_mutant(kind):
    def dq_rows(q, k, v, dout, start_q, start_kv, length, causal, head, group, softmax_scale, row_ids):
        g = head // group
        rows = np.asarray(row_ids, dtype=np.int64)
        qq = oa._as64(q[start_q + rows, head, :])
        oo = oa._as64(dout[start_q + rows, head, :])
        kk = oa._as64(k[start_kv:start_kv + length, g, :])
        vv = oa._as64(v[start_kv:start_kv + length, g, :])
        z = softmax_scale * (qq @ kk.T)
        if causal:
            z = np.where(np.arange(length)[None, :] <= rows[:, None], z, -np.inf)
        e = np.exp(z - z.max(axis=1, keepdims=True))
        p = e / e.sum(axis=1, keepdims=True)
        dp = oo @ vv.T
        if kind == "no_centering":     # mistake: the softmax Jacobian's rowsum term dropped
            dz = p * dp
        else:
            dz = p * (dp - (p * dp).sum(axis=1, keepdims=True))
        if kind == "value_operand":    # mistake: dQ contracted with V instead of K
            return softmax_scale * (dz @ vv)
        if kind == "no_scale":         # mistake: the outer scale of dQ = scale dZ K dropped
            return dz @ kk
        return softmax_scale * (dz @ kk)
    dq_rows.__name__ = f"dq_rows_{kind}"
    return dq_rows


@pytest.mark.parametrize("kind", ["no_centering", "value_operand", "no_scale"])
def test_dq_rows_pin_catches_mutant(monkeypatch, kind):
    import oracle as pkg
    mutant = _dq_rows_mutant(kind)
    monkeypatch.setattr(oa, "thd_attention_bwd_dq_rows", mutant)
    monkeypatch.setattr(pkg, "thd_attention_bwd_dq_rows", mutant)
    failed = 0
    for causal in (False, True):
        try:
            bwd_pins.test_dq_rows_against_torch_autograd(causal)
        except AssertionError:
            failed += 1
    assert failed >= 1, f"no pin caught mutant {mutant.__name__}"


@pytest.mark.parametrize("mutant", [window_lower_off_by_one, window_upper_exclusive])
def test_windowed_rows_pin_catches_mutant(monkeypatch, mutant):
    import oracle as pkg
    monkeypatch.setattr(oa, "visible_range", mutant)
    monkeypatch.setattr(pkg, "visible_range", mutant)
    failed = 0
    for code in (0, 1):
        for w in ((3, -1), (2, 4), (5, 0)):
            try:
                with np.errstate(invalid="ignore"):   # a mutant may leave a row without keys
                    win.test_sampled_rows_with_window_against_tril_triu(code, w)
            except AssertionError:
                failed += 1
    assert failed >= 1, f"no pin caught mutant {mutant.__name__}"
