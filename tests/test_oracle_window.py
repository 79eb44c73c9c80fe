"""Pins for the sliding-window form of the oracle (visible_range, the ``window`` argument of
thd_attention_fwd_general and thd_attention_bwd).

The pages only name sliding windows (an option the per-sequence policy PR rejects); the
window is read as a band [i + shift - left, i + shift + right] around the diagonal of the
sequence's mask type, intersected with that mask type.  Pins that do not reuse the oracle's
index arithmetic:

* the band built with torch's tril / triu (library routines) and an fp64 softmax, for every
  mask type, one- and two-sided windows, square and rectangular sequences;
* a window of width zero copies one value row: out_i = v_(i+shift), lse_i = scale q_i.k_(i+shift);
* a causal window of w keys equals full attention of the query over the w + 1 keys ending at
  it (torch's scaled_dot_product_attention on that key slice);
* (-1, -1), and any window wider than the sequence, changes nothing;
* gradients: torch autograd through the tril / triu band.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

BIG = 1 << 20


def _rect(lq, lkv, h=2, d=8, seed=0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(lq, h, d, generator=g, dtype=torch.float64)
    k = torch.randn(lkv, h, d, generator=g, dtype=torch.float64)
    v = torch.randn(lkv, h, d, generator=g, dtype=torch.float64)
    return q, k, v


def _band(lq, lkv, code, left, right):
    """Boolean [lq, lkv] mask from torch.tril / torch.triu diagonals."""
    shift = lkv - lq if code == 2 else 0
    upper = BIG if right < 0 else shift + right
    if code != 0:
        upper = min(upper, shift)
    lower = -BIG if left < 0 else shift - left
    ones = torch.ones(lq, lkv, dtype=torch.bool)
    return ones.tril(diagonal=upper) & ones.triu(diagonal=lower)


def _torch_attention(q, k, v, mask, scale):
    """fp64 softmax(scale q k^T) v with a boolean mask; rows without a key give 0 / -inf."""
    z = torch.einsum("ihd,jhd->hij", q, k) * scale
    z = z.masked_fill(~mask[None], float("-inf"))
    rows = mask.any(dim=1)
    p = torch.zeros_like(z)
    p[:, rows] = torch.softmax(z[:, rows], dim=-1)
    out = torch.einsum("hij,jhd->ihd", p, v)
    lse = torch.full((q.shape[1], q.shape[0]), float("-inf"), dtype=torch.float64)
    lse[:, rows] = torch.logsumexp(z[:, rows], dim=-1)
    return out, lse


@pytest.mark.parametrize("lq,lkv", [(11, 11), (6, 13), (13, 6)])
@pytest.mark.parametrize("code", [0, 1, 2])
@pytest.mark.parametrize("window", [(3, -1), (-1, 2), (2, 4), (0, 0), (5, 0), (0, 7)])
def test_band_against_torch_tril_triu(lq, lkv, code, window):
    q, k, v = _rect(lq, lkv, seed=lq * 31 + lkv + code)
    scale = 0.37
    out, lse = oracle.thd_attention_fwd_general(q, k, v, [0, lq], [0, lkv], None, None, [code], 1, scale,
                                                window=window)
    ref, ref_lse = _torch_attention(q, k, v, _band(lq, lkv, code, *window), scale)
    np.testing.assert_allclose(out, ref.numpy(), atol=1e-12)
    fin = np.isfinite(ref_lse.numpy())
    np.testing.assert_allclose(lse[fin], ref_lse.numpy()[fin], atol=1e-12)
    assert np.all(np.isneginf(lse[~fin]))


@pytest.mark.parametrize("lq,lkv,code", [(9, 9, 0), (9, 9, 1), (5, 12, 2), (12, 5, 2)])
def test_zero_width_window_copies_one_value_row(lq, lkv, code):
    q, k, v = _rect(lq, lkv, seed=3)
    scale = 0.5
    out, lse = oracle.thd_attention_fwd_general(q, k, v, [0, lq], [0, lkv], None, None, [code], 1, scale,
                                                window=(0, 0))
    shift = lkv - lq if code == 2 else 0
    for i in range(lq):
        j = i + shift
        if 0 <= j < lkv:
            assert np.array_equal(out[i], v[j].numpy())
            np.testing.assert_allclose(lse[:, i], scale * (q[i] * k[j]).sum(-1).numpy(), atol=1e-14)
        else:
            assert np.all(out[i] == 0) and np.all(np.isneginf(lse[:, i]))


@pytest.mark.parametrize("w", [0, 1, 4, 9])
def test_causal_window_is_full_attention_over_the_last_keys(w):
    L = 14
    q, k, v = _rect(L, L, h=1, d=16, seed=w)
    scale = 0.25
    out, lse = oracle.thd_attention_fwd_general(q, k, v, [0, L], [0, L], None, None, [1], 1, scale,
                                                window=(w, -1))
    for i in range(L):
        lo = max(0, i - w)
        o = torch.nn.functional.scaled_dot_product_attention(q[i:i + 1].transpose(0, 1), k[lo:i + 1].transpose(0, 1),
                                                             v[lo:i + 1].transpose(0, 1), scale=scale)
        np.testing.assert_allclose(out[i], o.transpose(0, 1)[0].numpy(), atol=1e-13)


def test_unbounded_and_wide_windows_change_nothing():
    w = workloads.from_lengths("wide", [7, 19, 3, 12], [1, 0, 1, 0], gaps_before=[2, 1, 0, 4], heads_q=4, heads_kv=2,
                               head_dim=16, seed=6)
    codes = np.array([1, 0, 2, 1], np.uint8)
    args = (w.q, w.k, w.v, w.cu_seqlens, w.cu_seqlens, w.cu_seqlens_padded, w.cu_seqlens_padded, codes,
            w.batch_size, w.softmax_scale)
    base_o, base_l = oracle.thd_attention_fwd_general(*args)
    for window in ((-1, -1), (19, -1), (-1, 19), (40, 40)):
        o, l = oracle.thd_attention_fwd_general(*args, window=window)
        assert np.array_equal(o, base_o) and np.array_equal(l, base_l), window


@pytest.mark.parametrize("code,window", [(0, (2, 3)), (1, (4, -1)), (2, (1, 1))])
def test_window_gradients_against_autograd(code, window):
    lq, lkv = (10, 10) if code != 2 else (7, 11)
    q, k, v = _rect(lq, lkv, seed=11 + code)
    g = torch.Generator().manual_seed(5)
    do = torch.randn(lq, 2, 8, generator=g, dtype=torch.float64)
    scale = 0.45
    dq, dk, dv = oracle.thd_attention_bwd(q, k, v, do, [0, lq], [0, lkv], None, None, [code], 1, scale,
                                          window=window)
    mask = _band(lq, lkv, code, *window)
    qq, kk, vv = (t.clone().requires_grad_() for t in (q, k, v))
    out, _ = _torch_attention(qq, kk, vv, mask, scale)
    out.backward(do)
    np.testing.assert_allclose(dq, qq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, kk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, vv.grad.numpy(), atol=1e-12)


@pytest.mark.parametrize("code", [0, 1])
@pytest.mark.parametrize("window", [(3, -1), (2, 4), (0, 0), (5, 0), (-1, -1)])
def test_sampled_rows_with_window_against_tril_triu(code, window):
    """The sampled-rows oracle (used on full-size batches) with a window equals the torch
    tril / triu band on those rows, for a sequence inside a packed buffer with grouped heads."""
    L, off = 23, 4
    q, k, v = _rect(L + off + 3, L + off + 3, h=2, d=8, seed=code * 7 + window[0] + 3)
    scale = 0.41
    rows = np.array([0, 1, 9, L - 2, L - 1])
    band = _band(L, L, code, *window)
    kk, vv = k[:, :1].repeat(1, 2, 1), v[:, :1].repeat(1, 2, 1)   # key/value head 0 serves both query heads
    ref, ref_lse = _torch_attention(q[off:off + L], kk[off:off + L], vv[off:off + L], band, scale)
    for h in range(2):
        out, lse = oracle.thd_attention_rows(q, k, v, off, off, L, code == 1, h, 2, scale, rows, window=window)
        np.testing.assert_allclose(out, ref[rows, h].numpy(), atol=1e-12)
        np.testing.assert_allclose(lse, ref_lse[h, rows].numpy(), atol=1e-12)
