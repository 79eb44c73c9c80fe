"""Pins for the padding-mask oracle.

Source: "[PyTorch] Build the attention padding mask without host syncs"
(TransformerEngine PR).  The Equivalence section reports an exhaustive check:
every combination of lengths in [0, max_seqlen] for max_seqlen 1..8 and batch
1..4, with and without a cu_seqlens buffer longer than batch + 1, 35368 cases
(tests/golden/mask_case_counts.txt).  Here both oracle forms (the old loop and
the vectorised formula) are run over exactly that space, the case count must
equal the printed one, and the two forms must agree on every case.
"""
import itertools

import numpy as np
import pytest

import oracle
from conftest import read_golden


def enumerate_self_cases():
    """Yield (cu_buffer, batch, max_seqlen) over the page's exhaustive space."""
    rng = np.random.default_rng(123)
    for S in range(1, 9):
        for B in range(1, 5):
            for lens in itertools.product(range(S + 1), repeat=B):
                cu = np.zeros(B + 1, dtype=np.int32)
                cu[1:] = np.cumsum(lens)
                yield cu, B, S
                tail = rng.integers(-2**31, 2**31 - 1, size=3).astype(np.int32)
                yield np.concatenate([cu, tail]), B, S


def test_self_mask_exhaustive_case_count_and_forms_agree():
    expected = int(read_golden("mask_case_counts.txt")["self_attention_cases"])
    n = 0
    for cu, B, S in enumerate_self_cases():
        a = oracle.padding_mask_loop(cu, B, S)
        b = oracle.padding_mask_formula(cu, B, S)
        assert a.shape == (B, 1, 1, S) and a.dtype == np.bool_
        assert np.array_equal(a, b)
        n += 1
    assert n == expected


def test_cross_case_count_reading():
    """The cross-attention count: lengths (q, kv) per sequence, S_q, S_kv in 1..5, B in 1..3."""
    expected = int(read_golden("mask_case_counts.txt")["cross_attention_cases"])
    n = sum(((sq + 1) * (skv + 1)) ** b for sq in range(1, 6) for skv in range(1, 6)
            for b in range(1, 4))
    assert n == expected


def test_invalid_lengths():
    # longer than max_seqlen: the loop cannot build the row, the formula gives all-False
    cu = np.array([0, 9, 10], dtype=np.int32)
    with pytest.raises(ValueError):
        oracle.padding_mask_loop(cu, 2, 8)
    m = oracle.padding_mask_formula(cu, 2, 8)
    assert not m[0].any() and m[1, 0, 0].tolist() == [False] + [True] * 7
    # negative length (non-monotone buffer): formula gives all-True
    m = oracle.padding_mask_formula(np.array([5, 2], dtype=np.int32), 1, 4)
    assert m.all()


def test_empty_batch_and_zero_width():
    assert oracle.padding_mask_formula(np.array([0], np.int32), 0, 8).shape == (0, 1, 1, 8)
    assert oracle.padding_mask_formula(np.array([0, 3], np.int32), 1, 0).shape == (1, 1, 1, 0)
