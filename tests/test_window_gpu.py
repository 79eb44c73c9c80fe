"""Sliding-window attention (thd_attn_fwd_window / thd_attn_bwd_window) on the GPU against the
fp64 oracle with the same window.  The band is the oracle's reading (visible_range): keys
[i + shift - left, i + shift + right] around the diagonal of each sequence's mask type.

Batches mix long sequences (256-row blocks whose two query tiles start at different KV
tiles), short ones (paired tiles) and head dims on the serial kernel; windows cover one- and
two-sided bands, width zero, and bands wider than the sequences.  Forward tolerances as for
thd_attn_fwd; gradients as in test_bwd_gpu (relative to the tensor's largest magnitude)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from test_bwd_gpu import REL
from thd_testutil import LSE_ATOL, OutErrors, assert_out_close, to_device

pytestmark = pytest.mark.gpu
vlp = pytest.importorskip("variable_length_packed_gb300")

WINDOWS = [(64, -1), (100, 50), (0, 0), (300, 0), (-1, 37), (129, 129), (1000, 1000)]


def _batch(d, dtype, seed):
    lens = [700, 1, 129, 90, 300, 0, 257, 41, 128, 513]
    codes = np.array([1, 0, 2, 1, 0, 1, 2, 0, 1, 0], np.uint8)
    w = workloads.from_lengths("win", lens, codes != 0, gaps_before=[3, 0, 5, 1, 0, 2, 7, 0, 1, 4], trailing=6,
                               heads_q=4, heads_kv=2, head_dim=d, dtype=dtype, seed=seed, with_padded=True)
    return w, codes


def _fwd(w, codes, window, dev=None):
    dev = dev or to_device(w)
    c = torch.from_numpy(codes).cuda()
    ws = torch.zeros(vlp.thd_attn_workspace_size(), dtype=torch.uint8, device="cuda")
    out, lse = vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], dev["padded"], dev["padded"], c,
                                w.batch_size, w.max_seqlen, w.softmax_scale, workspace=ws, window=window)
    torch.cuda.synchronize()
    assert int(ws[8:12].cpu().numpy().view(np.uint32)[0]) == 0
    return out, lse


@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float16), (40, torch.bfloat16)])
def test_window_forward_matches_oracle(d, dtype):
    w, codes = _batch(d, dtype, seed=d)
    dev = to_device(w)
    for window in WINDOWS:
        out, lse = _fwd(w, codes, window, dev)
        ref, ref_lse = oracle.thd_attention_fwd_general(w.q, w.k, w.v, w.cu_seqlens, w.cu_seqlens,
                                                        w.cu_seqlens_padded, w.cu_seqlens_padded, codes,
                                                        w.batch_size, w.softmax_scale, window=window)
        o = out.float().cpu().double().numpy()
        l = lse.cpu().double().numpy()
        seen = np.isfinite(ref_lse)
        assert_out_close(o, ref, dtype, f"window {window}")
        assert np.abs(l[seen] - ref_lse[seen]).max() <= LSE_ATOL, window
        assert np.all(np.isneginf(l[~seen])), window
        assert np.all(o[~seen.any(axis=0)] == 0.0), window


def test_unbounded_window_is_the_plain_call_bit_for_bit():
    w, codes = _batch(128, torch.bfloat16, seed=3)
    dev = to_device(w)
    c = torch.from_numpy(codes).cuda()
    a = vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], dev["padded"], dev["padded"], c,
                         w.batch_size, w.max_seqlen, w.softmax_scale)
    b = _fwd(w, codes, (-1, -1), dev)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("window", [(5, 0), (0, 3), (40, 20)])
def test_window_with_separate_q_kv_sequences(window):
    lq = [250, 300, 7, 200, 130]
    lkv = [100, 64, 40, 129, 0]
    codes = np.array([2, 1, 2, 0, 1], np.uint8)
    qs = np.array([0, 250, 550, 557, 757], np.int32)
    ks = np.array([887, 987, 1051, 1091, 1220], np.int32)
    w = workloads.from_lengths("rectw", [1230], [0], heads_q=4, heads_kv=2, head_dim=128, dtype=torch.bfloat16,
                               seed=9)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lkv)]).astype(np.int32)
    dv = lambda a: torch.from_numpy(a).cuda()
    out, lse = vlp.thd_attn_fwd(w.q.cuda(), w.k.cuda(), w.v.cuda(), dv(cu_q), dv(cu_k), dv(qs), dv(ks), dv(codes), 5,
                                300, w.softmax_scale, window=window)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.thd_attention_fwd_general(w.q, w.k, w.v, cu_q, cu_k, qs, ks, codes, 5, w.softmax_scale,
                                                    window=window)
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    seen = np.isfinite(ref_lse)
    assert_out_close(o, ref, torch.bfloat16, "window cross")
    assert np.abs(l[seen] - ref_lse[seen]).max() <= LSE_ATOL
    assert np.all(np.isneginf(l[~seen])) and np.all(o[~seen.any(axis=0)] == 0.0)


@pytest.mark.parametrize("d,dtype,window", [(128, torch.bfloat16, (64, -1)), (64, torch.float16, (100, 50)),
                                            (128, torch.float16, (0, 0)), (64, torch.bfloat16, (300, 0))])
def test_window_backward_matches_oracle(d, dtype, window):
    w, codes = _batch(d, dtype, seed=20 + d)
    dev = to_device(w)
    c = torch.from_numpy(codes).cuda()
    out, lse = vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], dev["padded"], dev["padded"], c,
                                w.batch_size, w.max_seqlen, w.softmax_scale, window=window)
    dout = workloads.grad_output(w, 7)
    dq, dk, dvv = vlp.thd_attn_bwd(dev["q"], dev["k"], dev["v"], out, lse, dout.cuda(), dev["cu"], dev["cu"],
                                   dev["padded"], dev["padded"], c, w.batch_size, w.max_seqlen, w.softmax_scale,
                                   window=window)
    torch.cuda.synchronize()
    ref = oracle.thd_attention_bwd(w.q, w.k, w.v, dout, w.cu_seqlens, w.cu_seqlens, w.cu_seqlens_padded,
                                   w.cu_seqlens_padded, codes, w.batch_size, w.softmax_scale, window=window)
    # dQ and dK are sums of dS = P (dP - D) terms; with a zero-width band P = 1 and dP = D
    # in exact arithmetic, so the reference is ~0 and the rounding of the terms sets the
    # scale: the tolerance uses max(max|ref|, scale * max|k| * max|dV|), dV = P^T dO being
    # the size of dP - D's parts.
    term = w.softmax_scale * float(np.abs(w.k.double().numpy()).max()) * np.abs(ref[2]).max()
    for g, r, name in zip((dq, dk, dvv), ref, ("dq", "dk", "dv")):
        g = g.float().cpu().double().numpy()
        scale = max(np.abs(r).max(), term if name != "dv" else 0.0)
        assert np.abs(g - r).max() <= REL[dtype] * scale + 1e-6, (name, window)


def test_long_context_window_sampled_rows():
    """The full-size long-context batch with the window bench.py times, (2048, 2048), in the
    same call: sampled rows (tile and band edges, random rows) of two heads of every sequence
    against the fp64 oracle."""
    w = workloads.make("long_context")
    dev = to_device(w)
    window = (2048, 2048)
    out, lse = vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], None, None, dev["causal"],
                                w.batch_size, w.max_seqlen, w.softmax_scale, window=window)
    torch.cuda.synchronize()
    rng = np.random.default_rng(88)
    group = w.num_heads_q // w.num_heads_kv
    acc = OutErrors(w.dtype, f"long_context window {window}")   # the count over every sampled row
    for b in range(w.batch_size):
        s, L = int(w.starts[b]), int(w.lengths[b])
        edges = [0, 1, 127, 128, 2047, 2048, 2049, L - 2049, L - 2048, L - 1]
        rows = np.unique(np.clip(np.r_[edges, rng.integers(0, L, 6)], 0, L - 1))
        for h in rng.choice(w.num_heads_q, size=2, replace=False):
            ref_o, ref_l = oracle.thd_attention_rows(w.q, w.k, w.v, s, s, L, bool(w.causal[b]), int(h), group,
                                                     w.softmax_scale, rows, window=window)
            idx = s + torch.from_numpy(rows).cuda()
            acc.add(out[idx, int(h)].float().cpu().double().numpy(), ref_o, f"b={b} h={int(h)}")
            assert np.abs(lse[int(h), idx].cpu().double().numpy() - ref_l).max() <= LSE_ATOL
    acc.check()
