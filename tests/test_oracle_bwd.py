"""Pins for the backward oracle (dQ, dK, dV).

* torch fp64 autograd through scaled_dot_product_attention, per sequence, with GQA and each
  mask type (a library routine);
* central finite differences of the forward oracle on a tiny case (brute force);
* the policy identity of "Add per-sequence causal policy to packed THD attention"
  (Validation: Q/K/V gradient parity against scalar-policy attention): the mixed batch's
  gradients equal those of each sequence run alone with its own policy;
* zero gradient on pad rows, on rows that see no key and on keys no query sees.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads


def _grads(w, dout, codes=None):
    return oracle.thd_attention_bwd(w.q, w.k, w.v, dout, w.cu_seqlens, w.cu_seqlens, w.cu_seqlens_padded,
                                    w.cu_seqlens_padded, w.seq_is_causal if codes is None else codes,
                                    w.batch_size, w.softmax_scale)


def _dout(w, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(w.q.shape, generator=g).to(w.dtype)


@pytest.mark.parametrize("code", [0, 1, 2])
def test_against_torch_autograd(code):
    w = workloads.from_lengths("bw", [7, 19, 3], [1, 1, 1], gaps_before=[2, 1, 3], trailing=2, heads_q=4,
                               heads_kv=2, head_dim=16, seed=31)
    dout = _dout(w, 32)
    codes = np.full(3, code, np.uint8)
    dq, dk, dv = _grads(w, dout, codes)
    for b in range(3):
        s, L = int(w.starts[b]), int(w.lengths[b])
        q = w.q[s:s + L].double().transpose(0, 1).clone().requires_grad_()
        k = w.k[s:s + L].double().transpose(0, 1).clone().requires_grad_()
        v = w.v[s:s + L].double().transpose(0, 1).clone().requires_grad_()
        kk, vv = k.repeat_interleave(2, dim=0), v.repeat_interleave(2, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, is_causal=code != 0, scale=w.softmax_scale)
        o.backward(dout[s:s + L].double().transpose(0, 1))
        np.testing.assert_allclose(dq[s:s + L], q.grad.transpose(0, 1).numpy(), atol=1e-12)
        np.testing.assert_allclose(dk[s:s + L], k.grad.transpose(0, 1).numpy(), atol=1e-12)
        np.testing.assert_allclose(dv[s:s + L], v.grad.transpose(0, 1).numpy(), atol=1e-12)
    pad = np.ones(w.total_tokens, bool)
    for s, L in zip(w.starts, w.lengths):
        pad[s:s + L] = False
    assert np.all(dq[pad] == 0) and np.all(dk[pad] == 0) and np.all(dv[pad] == 0)


def test_rectangular_bottom_right_against_autograd():
    g = torch.Generator().manual_seed(5)
    Lq, Lkv = 9, 4
    q = torch.randn(Lq, 2, 8, generator=g, dtype=torch.float64)
    k = torch.randn(Lkv, 2, 8, generator=g, dtype=torch.float64)
    v = torch.randn(Lkv, 2, 8, generator=g, dtype=torch.float64)
    do = torch.randn(Lq, 2, 8, generator=g, dtype=torch.float64)
    dq, dk, dv = oracle.thd_attention_bwd(q, k, v, do, [0, Lq], [0, Lkv], None, None, [2], 1, 0.4)
    allowed = torch.arange(Lkv)[None, :] <= torch.arange(Lq)[:, None] + (Lkv - Lq)
    rows = allowed.any(1)
    qq = q.transpose(0, 1).clone().requires_grad_()
    kk = k.transpose(0, 1).clone().requires_grad_()
    vv = v.transpose(0, 1).clone().requires_grad_()
    # torch's fp64 softmax / matmul with autograd (its fused SDPA on fp64 inputs with a boolean
    # mask agrees only to ~1e-7)
    z = (qq[:, rows] @ kk.transpose(-1, -2) * 0.4).masked_fill(~allowed[rows], float("-inf"))
    o = torch.softmax(z, dim=-1) @ vv
    o.backward(do.transpose(0, 1)[:, rows])
    np.testing.assert_allclose(dq, qq.grad.transpose(0, 1).numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, kk.grad.transpose(0, 1).numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, vv.grad.transpose(0, 1).numpy(), atol=1e-12)
    assert np.all(dq[~rows.numpy()] == 0)


def test_finite_differences_tiny():
    w = workloads.from_lengths("fd", [4, 3], [1, 0], gaps_before=[0, 1], heads_q=2, heads_kv=1, head_dim=4,
                               seed=8)
    q, k, v = (t.double().numpy().copy() for t in (w.q, w.k, w.v))
    dout = np.random.default_rng(3).standard_normal(q.shape)
    dq, dk, dv = oracle.thd_attention_bwd(q, k, v, dout, w.cu_seqlens, w.cu_seqlens, w.cu_seqlens_padded,
                                          w.cu_seqlens_padded, w.seq_is_causal, 2, w.softmax_scale)

    def loss(q_, k_, v_):
        o, _ = oracle.thd_attention_fwd(q_, k_, v_, w.cu_seqlens, w.cu_seqlens, w.cu_seqlens_padded,
                                        w.cu_seqlens_padded, w.seq_is_causal, 2, w.softmax_scale)
        return float((o * dout).sum())

    eps = 1e-6
    for arr, grad in ((q, dq), (k, dk), (v, dv)):
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            up = loss(q, k, v)
            arr[idx] = old - eps
            down = loss(q, k, v)
            arr[idx] = old
            assert abs((up - down) / (2 * eps) - grad[idx]) < 1e-7, idx


def test_mixed_policy_gradients_equal_per_sequence():
    w = workloads.make("tiny_mixed")
    dout = _dout(w, 9)
    dq, dk, dv = _grads(w, dout)
    for b in range(w.batch_size):
        s, L = int(w.starts[b]), int(w.lengths[b])
        sub = slice(s, s + L)
        g1 = oracle.thd_attention_bwd(w.q[sub], w.k[sub], w.v[sub], dout[sub], [0, L], [0, L], None, None,
                                      [int(w.causal[b])], 1, w.softmax_scale)
        np.testing.assert_allclose(dq[sub], g1[0], atol=1e-14)
        np.testing.assert_allclose(dk[sub], g1[1], atol=1e-14)
        np.testing.assert_allclose(dv[sub], g1[2], atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_dq_rows_against_torch_autograd(causal):
    """The row-wise dQ used to check full-size batches on sampled rows equals torch fp64
    autograd through scaled_dot_product_attention on those rows (grouped heads, a sequence
    inside a packed buffer)."""
    w = workloads.from_lengths("bwr", [5, 37], [causal, causal], gaps_before=[1, 4], trailing=3, heads_q=4,
                               heads_kv=2, head_dim=16, seed=61)
    dout = _dout(w, 62)
    s, L = int(w.starts[1]), int(w.lengths[1])
    rows = np.array([0, 1, 17, L - 2, L - 1])
    q = w.q[s:s + L].double().transpose(0, 1).clone().requires_grad_()
    kk = w.k[s:s + L].double().transpose(0, 1).repeat_interleave(2, dim=0)
    vv = w.v[s:s + L].double().transpose(0, 1).repeat_interleave(2, dim=0)
    o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, is_causal=causal, scale=w.softmax_scale)
    o.backward(dout[s:s + L].double().transpose(0, 1))
    for h in range(4):
        got = oracle.thd_attention_bwd_dq_rows(w.q, w.k, w.v, dout, s, s, L, causal, h, 2, w.softmax_scale, rows)
        np.testing.assert_allclose(got, q.grad[h, rows].numpy(), atol=1e-12)
