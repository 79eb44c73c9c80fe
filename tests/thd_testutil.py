"""Helpers shared by the GPU parity tests: move a workload to the device, call the library,
compare with the fp64 oracle at the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import variable_length_packed_gb300 as vlp

# Acceptance bounds: output absolute error 1e-2 (bf16 inputs) / 2e-3 (fp16 inputs),
# LSE absolute error 1e-3; pad rows and the mask bit-exact.
OUT_ATOL = {torch.bfloat16: 1e-2, torch.float16: 2e-3}
LSE_ATOL = 1e-3


def out_bound(ref, dtype):
    """Per-element bound on |out - ref|: OUT_ATOL plus half a unit in the last place of the
    output type at |ref|.  The output is stored in the input type, and from |ref| = 4 on a bf16
    value correctly rounded from the exact one can itself be up to 0.0156 away from it, so the
    flat 1e-2 cannot hold there; an element above OUT_ATOL passes only within this bound."""
    mant = 7 if dtype == torch.bfloat16 else 10
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return OUT_ATOL[dtype] + np.where(a > 0, np.exp2(e - mant - 1), 0.0)


def assert_out_close(got, ref, dtype, what=""):
    """|got - ref| within out_bound everywhere, and above the flat OUT_ATOL in at most one
    element in 10^4 (so the half-ulp allowance cannot hide a systematic error).  Returns the
    largest error."""
    acc = OutErrors(dtype, what)
    acc.add(got, ref)
    return acc.check()


class OutErrors:
    """Output errors gathered over many samples (e.g. every sampled (sequence, head, row) of a
    batch), checked once: each element against out_bound, and the one-in-10^4 count of
    elements above the flat OUT_ATOL over the whole sample, not per piece, so that one
    over-bound element per (sequence, head) cannot pass where pieces are small."""

    def __init__(self, dtype, what=""):
        self.dtype = dtype
        self.what = what
        self.n = 0
        self.over = 0
        self.worst = 0.0

    def add(self, got, ref, where=""):
        got = np.asarray(got, dtype=np.float64)
        ref = np.asarray(ref, dtype=np.float64)
        err = np.abs(got - ref)
        if err.size == 0:
            return
        worst = float(err.max())
        bound = out_bound(ref, self.dtype)
        assert np.all(err <= bound), f"{self.what} {where}: max |out err| {worst:.3e}, above the rounding bound"
        self.n += err.size
        self.over += int((err > OUT_ATOL[self.dtype]).sum())
        self.worst = max(self.worst, worst)

    def check(self):
        """The count over everything added; returns the largest error."""
        allowed = max(1, self.n // 10000)
        if self.n:
            print(f"{self.what}: {self.over} of {self.n} elements above {OUT_ATOL[self.dtype]} "
                  f"(allowed {allowed}), max |err| {self.worst:.3e}")
        assert self.over <= allowed, f"{self.what}: {self.over} of {self.n} elements above {OUT_ATOL[self.dtype]}"
        return self.worst


def to_device(w, device="cuda"):
    dev = torch.device(device)
    d = dict(
        q=w.q.to(dev), k=w.k.to(dev), v=w.v.to(dev),
        cu=torch.from_numpy(w.cu_seqlens).to(dev),
        padded=None if w.cu_seqlens_padded is None else torch.from_numpy(w.cu_seqlens_padded).to(dev),
        causal=torch.from_numpy(w.seq_is_causal).to(dev),
    )
    return d


def run_gpu(w, dev=None, workspace=None, **over):
    dev = dev or to_device(w)
    args = dict(cu_seqlens_q_padded=dev["padded"], cu_seqlens_kv_padded=dev["padded"],
                seq_is_causal=dev["causal"], batch_size=w.batch_size, max_seqlen=w.max_seqlen,
                softmax_scale=w.softmax_scale, workspace=workspace)
    args.update(over)
    out, lse = vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], **args)
    torch.cuda.synchronize()
    return out, lse


def valid_rows(w):
    m = np.zeros(w.total_tokens, dtype=bool)
    for s, L in zip(w.starts, w.lengths):
        m[int(s):int(s) + int(L)] = True
    return m


def check_pad_rows(w, out, lse):
    """Rows of no sequence: exact zeros, LSE exactly -inf."""
    pad = torch.from_numpy(~valid_rows(w)).to(out.device)
    if pad.any():
        assert torch.all(out[pad] == 0), "pad rows not exact zero"
        if lse is not None:
            assert torch.all(torch.isneginf(lse[:, pad])), "pad LSE not -inf"


def compare_full(w, out, lse, ref_out=None, ref_lse=None):
    """Element-wise comparison of every row against the whole-batch oracle."""
    if ref_out is None:
        ref_out, ref_lse = oracle.thd_attention_fwd(
            w.q, w.k, w.v, w.cu_seqlens, w.cu_seqlens, w.cu_seqlens_padded, w.cu_seqlens_padded,
            w.seq_is_causal, w.batch_size, w.softmax_scale)
    o = out.float().cpu().double().numpy()
    vr = valid_rows(w)
    worst = assert_out_close(o[vr], ref_out[vr], w.dtype, w.name)
    if lse is not None:
        l = lse.cpu().double().numpy()
        lerr = np.abs(l[:, vr] - ref_lse[:, vr])
        assert lerr.max(initial=0.0) <= LSE_ATOL, f"{w.name}: max |lse err| {lerr.max():.3e}"
    check_pad_rows(w, out, lse)
    return worst


def compare_sampled(w, out, lse, pairs, rows_for):
    """Compare selected rows of selected (sequence, head) pairs against the oracle, row by row.
    The output bound applies per element and its count over all samples together."""
    group = w.num_heads_q // w.num_heads_kv
    acc = OutErrors(w.dtype, w.name)
    for b, h in pairs:
        s, L = int(w.starts[b]), int(w.lengths[b])
        rows = np.unique(np.clip(np.asarray(rows_for(L)), 0, L - 1))
        ref_o, ref_l = oracle.thd_attention_rows(w.q, w.k, w.v, s, s, L, bool(w.causal[b]), h, group,
                                                 w.softmax_scale, rows)
        got = out[s + torch.from_numpy(rows).to(out.device), h, :].float().cpu().double().numpy()
        acc.add(got, ref_o, f"b={b} h={h}")
        if lse is not None:
            gl = lse[h, s + torch.from_numpy(rows).to(lse.device)].cpu().double().numpy()
            lerr = np.abs(gl - ref_l).max()
            assert lerr <= LSE_ATOL, f"{w.name} b={b} h={h}: |lse err| {lerr:.3e}"
    worst = acc.check()
    check_pad_rows(w, out, lse)
    return worst


def boundary_rows(L, rng, extra=6):
    base = [0, 1, 2, 63, 64, 127, 128, 129, 255, 256, L // 2, L - 2, L - 1]
    return base + list(rng.integers(0, L, size=extra))


# Unit roundoff of the input types (the backward rounds P and dS to these).
UNIT = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}


def gradient_bounds(w, dout, out_gpu, cu_q, cu_kv, pad_q, pad_kv, codes, batch):
    """Per-element error bounds (dq, dk, dv) of a backward that rounds once to the input type
    where its MMAs take a computed operand.  No bound is stated for gradients ("Add
    per-sequence causal policy to packed THD attention", Validation, asks for parity only);
    this one follows from the steps of the chain rule the backward takes.

    Every gradient element is a sum of terms in which one factor was rounded once:
        dV_j = sum_i P_ij dO_i            P rounded (the P^T dO MMA)
        dK_j = scale sum_i dS_ij Q_i      dS rounded
        dQ_i = scale sum_j dS_ij K_j      dS rounded
    With u the unit roundoff (2^-8 bf16, 2^-11 fp16) each term is off by at most u of its
    own magnitude, so a sum is off by at most u M, M the sum of the terms' absolute values.
    One more difference is known exactly: D = rowsum(dO * O) is formed from the rounded
    forward output out_gpu, not the exact one, so dS moves by P * (D_gpu - D); its effect
    on dK and dQ is T.  Returned: 2 u M + 1.5 T per element (the factors cover the fp32
    products, sums and exponentials, each far below u); the caller adds 2 u |ref| for the
    output's own rounding.  dK / dV sum the group's query heads."""
    q, k, v = (t.double().numpy() for t in (w.q, w.k, w.v))
    do = dout.double().numpy()
    og = out_gpu.float().cpu().double().numpy()
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    group = Hq // Hkv
    scale = w.softmax_scale
    u = UNIT[w.dtype]
    mq, tq = np.zeros_like(q), np.zeros_like(q)
    mk, tk = np.zeros_like(k), np.zeros_like(k)
    mv = np.zeros_like(v)
    qs, ql = oracle.sequence_spans(cu_q, pad_q, batch)
    ks, kl = oracle.sequence_spans(cu_kv, pad_kv, batch)
    for b in range(batch):
        Lq, Lkv = int(ql[b]), int(kl[b])
        if Lq <= 0 or Lkv <= 0:
            continue
        code = 0 if codes is None else int(codes[b])
        ranges = np.array([oracle.visible_range(i, Lq, Lkv, code) for i in range(Lq)])
        keys = np.arange(Lkv)[None, :]
        visible = (keys >= ranges[:, :1]) & (keys < ranges[:, 1:])
        sq, sk = slice(qs[b], qs[b] + Lq), slice(ks[b], ks[b] + Lkv)
        for h in range(Hq):
            g = h // group
            Q, K, V, dO, Og = q[sq, h], k[sk, g], v[sk, g], do[sq, h], og[sq, h]
            Z = np.where(visible, scale * (Q @ K.T), -np.inf)
            zmax = np.where(visible.any(axis=1), Z.max(axis=1), 0.0)
            E = np.where(visible, np.exp(Z - zmax[:, None]), 0.0)
            den = E.sum(axis=1)
            P = E / np.where(den > 0, den, 1.0)[:, None]
            dP = dO @ V.T
            D = (dO * (P @ V)).sum(axis=1)
            dD = np.abs((dO * Og).sum(axis=1) - D)
            dS = P * (dP - D[:, None])
            mv[sk, g] += np.abs(P).T @ np.abs(dO)
            mk[sk, g] += scale * (np.abs(dS).T @ np.abs(Q))
            tk[sk, g] += scale * ((P * dD[:, None]).T @ np.abs(Q))
            mq[sq, h] += scale * (np.abs(dS) @ np.abs(K))
            tq[sq, h] += scale * dD[:, None] * (P @ np.abs(K))
    return 2 * u * mq + 1.5 * tq, 2 * u * mk + 1.5 * tk, 2 * u * mv
