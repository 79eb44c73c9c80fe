"""The parity tests' output bound (thd_testutil.out_bound / assert_out_close), on the CPU.

The stated absolute bound (1e-2 for bf16, 2e-3 for fp16) is kept wherever it can hold; an
element above it passes only within half an output-type ulp more, and only one element in
10^4 may use that allowance.  These checks pin that reading: correctly rounded outputs of
attention-like magnitude pass, outputs off by more than the rounding fail, a systematic excess
fails the count, and the count is strict where many outputs are large.
"""
import numpy as np
import pytest
import torch

from thd_testutil import OUT_ATOL, OutErrors, assert_out_close, out_bound


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_correctly_rounded_outputs_pass(dtype):
    """Correctly rounded outputs of attention-like magnitude (rows of N(0, 1) values mixed by a
    softmax; here N(0, 1) itself, the widest case) pass, although for bf16 a few of them are
    more than 1e-2 from the exact value."""
    rng = np.random.default_rng(3)
    ref = rng.normal(0.0, 1.0, size=200000)
    got = torch.from_numpy(ref).to(dtype).double().numpy()
    assert_out_close(got, ref, dtype, "rounded")


def test_count_guard_is_strict_for_large_outputs():
    """The one-in-10^4 guard is deliberately strict: when many outputs exceed 4 in magnitude,
    even correctly rounded bf16 values fail it (their rounding alone reaches 0.0156)."""
    ref = np.random.default_rng(4).normal(0.0, 2.5, size=200000)
    got = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    with pytest.raises(AssertionError):
        assert_out_close(got, ref, torch.bfloat16, "large")


def test_flat_bound_is_kept_where_rounding_is_small():
    ref = np.array([0.3, -0.7, 0.9])
    assert np.all(out_bound(ref, torch.bfloat16) < 0.0125)
    with pytest.raises(AssertionError):
        assert_out_close(ref + 0.0125, ref, torch.bfloat16, "off")


def test_error_beyond_the_rounding_allowance_fails():
    ref = np.array([5.0, 1.0, 2.0])
    got = ref.copy()
    got[0] += 0.03   # above 1e-2 + half a bf16 ulp at 5 (0.0156)
    with pytest.raises(AssertionError):
        assert_out_close(got, ref, torch.bfloat16, "big")


def test_systematic_excess_fails_the_count():
    ref = np.full(10000, 5.0)
    got = ref + 0.012   # each within the allowance, but all above the flat bound
    assert np.all(np.abs(got - ref) <= out_bound(ref, torch.bfloat16))
    with pytest.raises(AssertionError):
        assert_out_close(got, ref, torch.bfloat16, "systematic")
    got[1:] = ref[1:] + 0.005   # one element above the flat bound is allowed
    assert_out_close(got, ref, torch.bfloat16, "single") == pytest.approx(0.012)
    assert OUT_ATOL[torch.bfloat16] == 1e-2 and OUT_ATOL[torch.float16] == 2e-3


def test_count_is_taken_over_the_whole_sample_not_per_piece():
    """Sampled parity gathers every (sequence, head) piece before counting: one planted
    over-flat element in each of 600 small pieces (64 rows x 64 columns, the size of the
    many-short batch's sampled pairs) is 600 of 2.46M elements, above the one-in-10^4
    allowance (245), so it fails, although each piece alone would pass its own count."""
    rng = np.random.default_rng(11)
    acc = OutErrors(torch.bfloat16, "planted")
    for _ in range(600):
        ref = rng.normal(0.0, 0.5, size=(64, 64))
        got = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
        i, j = rng.integers(0, 64, size=2)
        ref[i, j] = 3.0
        got[i, j] = 3.0 + 0.0105   # above 1e-2, within the half-ulp allowance at 3
        assert_out_close(got, ref, torch.bfloat16, "one piece")   # passes alone
        acc.add(got, ref)
    with pytest.raises(AssertionError):
        acc.check()


def test_whole_sample_count_passes_correctly_rounded_pieces():
    rng = np.random.default_rng(12)
    acc = OutErrors(torch.bfloat16, "rounded pieces")
    for _ in range(200):
        ref = rng.normal(0.0, 1.0, size=(37, 128))
        acc.add(torch.from_numpy(ref).to(torch.bfloat16).double().numpy(), ref)
    assert acc.check() < 0.0157


# --- the backward's per-element gradient bound -------------------------------------------

def _emulated_backward(w, dout, drop_d=False, slip=0.0):
    """A backward that rounds exactly where the GPU's does (forward output O, P before the
    P^T dO product, dS before the dS Q / dS K products, and each gradient), in fp64 otherwise.
    ``drop_d`` and ``slip`` plant mistakes: dS without the D term, a relative error on dK."""
    import oracle
    dt = w.dtype
    rnd = lambda x: torch.from_numpy(x).to(dt).double().numpy()
    q, k, v = (t.double().numpy() for t in (w.q, w.k, w.v))
    do = dout.double().numpy()
    Hq, group, sc = q.shape[1], q.shape[1] // k.shape[1], w.softmax_scale
    dq, dk, dv, out = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v), np.zeros_like(q)
    starts, lens = oracle.sequence_spans(w.cu_seqlens, w.cu_seqlens_padded, w.batch_size)
    for b in range(w.batch_size):
        L, s = int(lens[b]), slice(int(starts[b]), int(starts[b]) + int(lens[b]))
        if L <= 0:
            continue
        r = np.array([oracle.visible_range(i, L, L, int(w.seq_is_causal[b])) for i in range(L)])
        vis = (np.arange(L)[None] >= r[:, :1]) & (np.arange(L)[None] < r[:, 1:])
        for h in range(Hq):
            g = h // group
            Q, K, V, dO = q[s, h], k[s, g], v[s, g], do[s, h]
            Z = np.where(vis, sc * Q @ K.T, -np.inf)
            E = np.where(vis, np.exp(Z - Z.max(axis=1)[:, None]), 0.0)
            P = E / E.sum(axis=1)[:, None]
            O = rnd(P @ V)
            out[s, h] = O
            D = 0.0 if drop_d else (dO * O).sum(axis=1)[:, None]
            dS = rnd(P * (dO @ V.T - D))
            dv[s, g] += rnd(P).T @ dO
            dk[s, g] += sc * (dS.T @ Q) * (1.0 + slip)
            dq[s, h] += sc * dS @ K
    return [rnd(x) for x in (dq, dk, dv)], torch.from_numpy(out).to(dt)


def _largest_share(w, got, out, dout):
    import oracle
    from thd_testutil import UNIT, gradient_bounds
    meta = (w.cu_seqlens, w.cu_seqlens, w.cu_seqlens_padded, w.cu_seqlens_padded, w.seq_is_causal, w.batch_size)
    ref = oracle.thd_attention_bwd(w.q, w.k, w.v, dout, *meta, w.softmax_scale)
    bounds = gradient_bounds(w, dout, out, *meta)
    shares = []
    for g, r, b in zip(got, ref, bounds):
        bound = b + 2 * UNIT[w.dtype] * np.abs(r) + 1e-6 * np.abs(r).max()
        shares.append(float((np.abs(g - r) / bound).max()))
    return shares


@pytest.fixture(scope="module", params=[torch.bfloat16, torch.float16])
def small_backward(request):
    import workloads
    w = workloads.from_lengths("bound", [1, 37, 130, 64], [1, 0, 1, 0], gaps_before=[2, 0, 5, 1], trailing=3,
                               heads_q=4, heads_kv=2, head_dim=64, dtype=request.param, seed=21)
    return w, workloads.grad_output(w, 5)


def test_gradient_bound_holds_for_the_rounding_it_models(small_backward):
    w, dout = small_backward
    got, out = _emulated_backward(w, dout)
    assert max(_largest_share(w, got, out, dout)) < 0.9


def test_gradient_bound_catches_a_dropped_d_term(small_backward):
    w, dout = small_backward
    got, out = _emulated_backward(w, dout, drop_d=True)
    dq, dk, dv = _largest_share(w, got, out, dout)
    assert dq > 1.0 and dk > 1.0 and dv < 1.0


def test_gradient_bound_catches_a_slip_of_eight_roundoffs(small_backward):
    """dK off by 8 u relative (3.1 % in bf16, 0.4 % in fp16) fails: the bound is a few u of the
    terms' magnitude, not a fraction of the tensor's largest value."""
    from thd_testutil import UNIT
    w, dout = small_backward
    got, out = _emulated_backward(w, dout, slip=8 * UNIT[w.dtype])
    dq, dk, dv = _largest_share(w, got, out, dout)
    assert dk > 1.0 and dq < 1.0 and dv < 1.0
