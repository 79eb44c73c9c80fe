"""thd_attn_bwd on the GPU against the fp64 backward oracle (dQ, dK, dV).

The oracle's gradients come from the inputs (q, k, v, dO) alone; the GPU backward
consumes the GPU forward's out and lse, as a training step would.

Tolerance (no bound is stated for gradients; derived from the backward's rounding steps,
see thd_testutil.gradient_bounds): where the oracle computes whole sequences each element
is checked against |g - ref| <= 2 u M + 1.5 T + 2 u |ref| (u the input type's unit
roundoff, M the sum of the absolute values of the element's terms, T the known effect of
the GPU's rounded forward output on D = rowsum(dO * O)).  The long batch whose oracle
runs on sampled dQ rows keeps a bound relative to the largest magnitude (2e-2 for bf16,
4e-3 for fp16).  Exact zeros are required wherever the gradient is structurally zero.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from thd_testutil import UNIT, gradient_bounds, to_device, valid_rows

pytestmark = pytest.mark.gpu
vlp = pytest.importorskip("variable_length_packed_gb300")

REL = {torch.bfloat16: 2e-2, torch.float16: 4e-3}
def run_bwd(w, seed, codes=None, cu_kv=None, pad_q=None, pad_kv=None):
    dev = to_device(w)
    causal = dev["causal"] if codes is None else torch.from_numpy(codes).cuda()
    cu_q = dev["cu"]
    cu_k = cu_q if cu_kv is None else torch.from_numpy(cu_kv).cuda()
    pq = dev["padded"] if pad_q is None else torch.from_numpy(pad_q).cuda()
    pk = dev["padded"] if pad_kv is None else torch.from_numpy(pad_kv).cuda()
    out, lse = vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], cu_q, cu_k, pq, pk, causal, w.batch_size,
                                w.max_seqlen, w.softmax_scale)
    dout = workloads.grad_output(w, seed)
    dq, dk, dv = vlp.thd_attn_bwd(dev["q"], dev["k"], dev["v"], out, lse, dout.cuda(), cu_q, cu_k, pq, pk, causal,
                                  w.batch_size, w.max_seqlen, w.softmax_scale)
    torch.cuda.synchronize()
    meta = (cu_q.cpu().numpy(), cu_k.cpu().numpy(), None if pq is None else pq.cpu().numpy(),
            None if pk is None else pk.cpu().numpy(), causal.cpu().numpy(), w.batch_size)
    ref = oracle.thd_attention_bwd(w.q, w.k, w.v, dout, *meta[:5], w.batch_size, w.softmax_scale)
    bounds = gradient_bounds(w, dout, out, *meta)
    return (dq, dk, dv), ref, bounds


def structural_zero_rows(T, cu_q, cu_kv, pad_q, pad_kv, codes, batch):
    """Rows whose gradient is zero by construction: query rows of no sequence or that see no
    key (dQ), key rows of no sequence or that no query sees (dK, dV)."""
    qs, ql = oracle.sequence_spans(cu_q, pad_q, batch)
    ks, kl = oracle.sequence_spans(cu_kv, pad_kv, batch)
    zq = np.ones(T, bool)
    zk = np.ones(T, bool)
    for b in range(batch):
        Lq, Lkv = int(ql[b]), int(kl[b])
        code = 0 if codes is None else int(codes[b])
        if Lq <= 0 or Lkv <= 0:
            continue
        nv = np.array([oracle.visible_keys(i, Lq, Lkv, code) for i in range(Lq)])
        zq[qs[b]:qs[b] + Lq] = nv == 0
        zk[ks[b]:ks[b] + nv.max()] = False
    return zq, zk


def check(w, got, ref, name, zeros=None, bounds=None):
    """Errors within the per-element bounds (when given), else within REL of the tensor's largest
    magnitude; structural zeros exact."""
    report, fails = [], []
    for i, (g, r, label) in enumerate(zip(got, ref, ("dq", "dk", "dv"))):
        g = g.float().cpu().double().numpy()
        scale = np.abs(r).max()
        err = np.abs(g - r)
        report.append(f"{name} {label}: max|err| {err.max():.3e} max|ref| {scale:.3e} "
                      f"rel {err.max() / max(scale, 1e-30):.3e}")
        if bounds is not None:
            bound = bounds[i] + 2 * UNIT[w.dtype] * np.abs(r) + 1e-6 * max(scale, 1e-30)
            used = float((err / bound).max())
            report[-1] += f", largest share of the per-element bound {used:.3f}"
            if used > 1.0:
                fails.append(report[-1])
        elif err.max() > REL[w.dtype] * scale + 1e-6:
            fails.append(report[-1])
        if zeros is not None:
            z = zeros[0] if label == "dq" else zeros[1]
            if not np.all(g[z] == 0):
                fails.append(f"{name} {label}: structural zeros not exact")
    print("\n".join(report))
    assert not fails, fails


def layout_zeros(w):
    return structural_zero_rows(w.total_tokens, w.cu_seqlens, w.cu_seqlens, w.cu_seqlens_padded,
                                w.cu_seqlens_padded, w.seq_is_causal, w.batch_size)


@pytest.mark.parametrize("name", ["tiny_mixed", "padded_gaps"])
def test_small_workloads(name):
    w = workloads.make(name)
    got, ref, bounds = run_bwd(w, seed=7)
    check(w, got, ref, name, layout_zeros(w), bounds)


@pytest.mark.parametrize("d,dtype,group", [(64, torch.bfloat16, 1), (128, torch.bfloat16, 4), (64, torch.float16, 2),
                                           (128, torch.float16, 1)])
def test_mixed_lengths_and_groups(d, dtype, group):
    lens = [1, 127, 128, 129, 300, 5]
    causal = [1, 0, 1, 0, 1, 0]
    w = workloads.from_lengths("bwdmix", lens, causal, gaps_before=[3, 0, 64, 1, 7, 2], trailing=5, heads_q=4,
                               heads_kv=4 // group, head_dim=d, dtype=dtype, seed=d + group)
    got, ref, bounds = run_bwd(w, seed=3)
    check(w, got, ref, f"mix d{d} g{group}", layout_zeros(w), bounds)


def test_large_trailing_region():
    """T far above the batch's rows: dK / dV of the rows after the last sequence (zeroed by
    every block of the first launch in equal shares) are exact zeros, dQ there too, and
    the sequences' gradients are within the per-element bounds."""
    w = workloads.from_lengths("trail", [100, 300, 37], [1, 0, 1], gaps_before=[5, 0, 9], trailing=30000,
                               heads_q=4, heads_kv=2, head_dim=128, dtype=torch.bfloat16, seed=16)
    got, ref, bounds = run_bwd(w, seed=17)
    check(w, got, ref, "trail", layout_zeros(w), bounds)


def test_mask_types_separate_q_kv():
    import test_merge_gpu as tm
    w, cu_q, cu_k, qs, ks, codes = tm.rect_batch(128, torch.bfloat16, seed=5)
    w.batch_size = 5
    w.cu_seqlens = cu_q
    got, ref, bounds = run_bwd(w, seed=11, codes=codes, cu_kv=cu_k, pad_q=qs, pad_kv=ks)
    check(w, got, ref, "rect", structural_zero_rows(w.total_tokens, cu_q, cu_k, qs, ks, codes, 5), bounds)


def test_mixed_gqa_sampled_sequences():
    """The 64-sequence GQA batch on the GPU; the oracle computes the gradients of four
    sequences (each sequence's gradients depend on that sequence only)."""
    w = workloads.make("mixed_gqa")
    dev = to_device(w)
    out, lse = vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], dev["padded"], dev["padded"],
                                dev["causal"], w.batch_size, w.max_seqlen, w.softmax_scale)
    dout = workloads.grad_output(w, 13)
    dq, dk, dv = vlp.thd_attn_bwd(dev["q"], dev["k"], dev["v"], out, lse, dout.cuda(), dev["cu"], dev["cu"],
                                  dev["padded"], dev["padded"], dev["causal"], w.batch_size, w.max_seqlen,
                                  w.softmax_scale)
    torch.cuda.synchronize()
    order = np.argsort(-w.lengths)
    for b in [int(order[0]), int(order[1]), int(order[-1]), 17]:
        s, L = int(w.starts[b]), int(w.lengths[b])
        sub = slice(s, s + L)
        ref = oracle.thd_attention_bwd(w.q[sub], w.k[sub], w.v[sub], dout[sub], [0, L], [0, L], None, None,
                                       [int(w.causal[b])], 1, w.softmax_scale)
        ws = workloads.Workload(name="seq", batch_size=1, lengths=np.array([L]), causal=w.causal[b:b + 1],
                                starts=np.array([0]), cu_seqlens=np.array([0, L], np.int32), cu_seqlens_padded=None,
                                seq_is_causal=w.seq_is_causal[b:b + 1], total_tokens=L, num_heads_q=w.num_heads_q,
                                num_heads_kv=w.num_heads_kv, head_dim=w.head_dim, dtype=w.dtype,
                                softmax_scale=w.softmax_scale, max_seqlen=L, q=w.q[sub], k=w.k[sub], v=w.v[sub])
        bounds = gradient_bounds(ws, dout[sub], out[sub], [0, L], [0, L], None, None, [int(w.causal[b])], 1)
        check(w, (dq[sub], dk[sub], dv[sub]), ref, f"gqa b={b} L={L}", bounds=bounds)
    pad = torch.from_numpy(~valid_rows(w)).cuda()
    assert torch.all(dq[pad] == 0) and torch.all(dk[pad] == 0) and torch.all(dv[pad] == 0)


def test_long_context_backward_sampled_dq_rows():
    """The full-size long-context batch in the configuration bench.py times (its own
    max_seqlen hint): dQ of sampled rows (tile edges and random rows) of two heads of every
    sequence against the row-wise fp64 oracle.  (dK / dV need every query row of a sequence;
    they are checked element by element on the smaller batches above.)"""
    w = workloads.make("long_context")
    dev = to_device(w)
    out, lse = vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], dev["padded"], dev["padded"],
                                dev["causal"], w.batch_size, w.max_seqlen, w.softmax_scale)
    dout = workloads.grad_output(w, 7)
    dq, _, _ = vlp.thd_attn_bwd(dev["q"], dev["k"], dev["v"], out, lse, dout.cuda(), dev["cu"], dev["cu"],
                                dev["padded"], dev["padded"], dev["causal"], w.batch_size, w.max_seqlen,
                                w.softmax_scale)
    torch.cuda.synchronize()
    rng = np.random.default_rng(77)
    group = w.num_heads_q // w.num_heads_kv
    for b in range(w.batch_size):
        s, L = int(w.starts[b]), int(w.lengths[b])
        for h in rng.choice(w.num_heads_q, size=2, replace=False):
            rows = np.unique(np.r_[0, 1, 127, 128, L - 129, L - 1, rng.integers(0, L, 6)])
            ref = oracle.thd_attention_bwd_dq_rows(w.q, w.k, w.v, dout, s, s, L, bool(w.causal[b]), int(h), group,
                                                   w.softmax_scale, rows)
            got = dq[s + torch.from_numpy(rows).cuda(), int(h)].float().cpu().double().numpy()
            err = np.abs(got - ref).max()
            assert err <= REL[w.dtype] * np.abs(ref).max(), (b, int(h), err, np.abs(ref).max())
