"""thd_attn_fwd on the GPU against the fp64 oracle, element by element.

Small workloads are compared on every row; the large ones (mixed-policy GQA, long
context, many short sequences) on sampled (sequence, head, row) triples computed one by
one by the oracle, plus every pad row (exact zero / -inf LSE).  Tolerances: |out| 1e-2
for bf16 inputs, 2e-3 for fp16 (an element above them passes only within that plus half an
output-type ulp of the exact value, at most one in 10^4: see thd_testutil.out_bound), |LSE| 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from conftest import read_golden
from thd_testutil import (LSE_ATOL, assert_out_close, boundary_rows, check_pad_rows, compare_full,
                          compare_sampled, run_gpu, to_device, valid_rows)

pytestmark = pytest.mark.gpu
vlp = pytest.importorskip("variable_length_packed_gb300")


def status_word(ws):
    return int(ws[8:12].cpu().numpy().view(np.uint32)[0])


def workspace():
    return torch.zeros(vlp.thd_attn_workspace_size(), dtype=torch.uint8, device="cuda")


# --- small workloads: every row -------------------------------------------------------------

@pytest.mark.parametrize("name", ["page1", "page1_pad", "tiny_mixed", "padded_gaps"])
def test_small_workloads_every_row(name):
    w = workloads.make(name)
    ws = workspace()
    out, lse = run_gpu(w, workspace=ws)
    assert status_word(ws) == 0
    compare_full(w, out, lse)


def test_page1_printed_values_on_gpu():
    g = read_golden("page1_full_attention.txt")
    for name in ("page1", "page1_pad"):
        w = workloads.make(name)
        out, lse = run_gpu(w)
        o = out.float().cpu().numpy()
        for r in range(7):
            assert np.all(np.abs(o[r, 0] - float(g[f"row {r}"])) <= 0.5e-4), (name, r, o[r, 0])
        if name == "page1_pad":
            assert np.all(o[7] == 0.0) and torch.isneginf(lse[0, 7])


def test_two_call_identity_on_gpu():
    """out(causal call) + out(full call) with the page's arrays equals the mixed-policy call."""
    g = read_golden("page2_two_call.txt")
    w = workloads.make("tiny_mixed")
    dev = to_device(w)
    ints = lambda key: torch.tensor([int(t) for t in g[key].split()], dtype=torch.int32, device="cuda")
    out_c, lse_c = vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], ints("causal_call.cu_seqlens"),
                                    ints("causal_call.cu_seqlens"), ints("causal_call.cu_seqlens_padded"),
                                    ints("causal_call.cu_seqlens_padded"),
                                    torch.ones(4, dtype=torch.bool, device="cuda"), 4, 3, w.softmax_scale)
    out_f, lse_f = vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], ints("full_call.cu_seqlens"),
                                    ints("full_call.cu_seqlens"), ints("full_call.cu_seqlens_padded"),
                                    ints("full_call.cu_seqlens_padded"), None, 3, 4, w.softmax_scale)
    out, lse = run_gpu(w, dev=dev)
    torch.cuda.synchronize()
    # The three calls pack their sequences into tiles differently (a sequence's keys sit
    # at other tile columns, so sums round in another order): the sum of the two calls and
    # the mixed call are each held to the oracle's tolerances.
    compare_full(w, out_c + out_f, torch.logaddexp(lse_c, lse_f))
    compare_full(w, out, lse)


# --- large workloads: sampled rows ----------------------------------------------------------

def test_mixed_gqa_sampled():
    w = workloads.make("mixed_gqa")
    ws = workspace()
    out, lse = run_gpu(w, workspace=ws)
    assert status_word(ws) == 0
    rng = np.random.default_rng(20)
    order = np.argsort(-w.lengths)
    seqs = list(order[:3]) + list(rng.choice(w.batch_size, size=5, replace=False))
    pairs = [(int(b), int(h)) for b in seqs for h in rng.choice(w.num_heads_q, size=3, replace=False)]
    compare_sampled(w, out, lse, pairs, lambda L: boundary_rows(L, rng, extra=24))


def test_long_context_sampled():
    w = workloads.make("long_context")
    ws = workspace()
    out, lse = run_gpu(w, workspace=ws)
    assert status_word(ws) == 0
    rng = np.random.default_rng(30)
    pairs = [(b, int(h)) for b in range(w.batch_size) for h in rng.choice(w.num_heads_q, size=2, replace=False)]
    compare_sampled(w, out, lse, pairs, lambda L: boundary_rows(L, rng, extra=16))


def test_many_short_sampled():
    w = workloads.make("many_short")
    ws = workspace()
    out, lse = run_gpu(w, workspace=ws)
    assert status_word(ws) == 0
    rng = np.random.default_rng(40)
    seqs = rng.choice(w.batch_size, size=150, replace=False)
    pairs = [(int(b), int(h)) for b in seqs for h in rng.choice(w.num_heads_q, size=4, replace=False)]
    compare_sampled(w, out, lse, pairs, lambda L: np.arange(L))


def test_long_sequences_in_a_late_chunk():
    """1500 sequences (three scheduler chunks of 512) whose four longest sit in the last chunk:
    every CTA visits the chunks longest first, which changes the order of the work, not its
    results.  Sampled rows of every head of the long sequences and of 40 short ones."""
    w = workloads.make("late_long")
    ws = workspace()
    out, lse = run_gpu(w, workspace=ws)
    assert status_word(ws) == 0
    rng = np.random.default_rng(60)
    pairs = [(b, h) for b in range(w.batch_size - 4, w.batch_size) for h in range(w.num_heads_q)]
    pairs += [(int(b), int(rng.integers(0, w.num_heads_q))) for b in rng.choice(w.batch_size - 4, 40, replace=False)]
    compare_sampled(w, out, lse, pairs, lambda L: boundary_rows(L, rng, extra=8))


# --- edge cases -----------------------------------------------------------------------------

@pytest.mark.parametrize("d,dtype", [(8, torch.float16), (16, torch.bfloat16), (32, torch.float16),
                                     (40, torch.bfloat16), (64, torch.float16), (72, torch.bfloat16),
                                     (96, torch.float16), (128, torch.float16), (128, torch.bfloat16)])
def test_head_dims_and_tile_boundaries(d, dtype):
    lens = [1, 127, 128, 129, 255, 256, 257, 3]
    causal = [1, 0, 1, 0, 1, 0, 1, 1]
    w = workloads.from_lengths(f"edge_d{d}", lens, causal, gaps_before=[5, 0, 1, 7, 0, 64, 2, 9], trailing=3,
                               heads_q=4, heads_kv=2, head_dim=d, dtype=dtype, seed=d)
    out, lse = run_gpu(w)
    compare_full(w, out, lse)


@pytest.mark.parametrize("hint", [0, 128])
@pytest.mark.parametrize("d,dtype", [(64, torch.float16), (128, torch.bfloat16)])
def test_paired_short_tiles_across_chunks(d, dtype, hint):
    """Sequences of at most 128 rows run as short tiles, two per unit ((sequence, head) tiles
    with the hint 0, runs of consecutive short sequences packed into 128-row tiles with the
    hint 128), longer ones as 256-row blocks: 700 sequences (two scheduler chunks of 512),
    three query heads on one KV head (odd tile counts per chunk), zero-length sequences (they
    end a run), lengths 128 / 129."""
    rng = np.random.default_rng(70 + d)
    B = 700
    lens = rng.integers(1, 129, size=B)
    lens[rng.choice(B, 60, replace=False)] = rng.integers(129, 400, size=60)
    lens[rng.choice(B, 20, replace=False)] = 0
    lens[:5] = [128, 129, 1, 0, 128]
    causal = rng.random(B) < 0.5
    gaps = rng.integers(0, 9, size=B)
    w = workloads.from_lengths("paired", lens, causal, gaps_before=gaps, trailing=5, heads_q=3, heads_kv=1,
                               head_dim=d, dtype=dtype, seed=d, with_padded=True)
    ws = workspace()
    out, lse = run_gpu(w, workspace=ws, max_seqlen=hint)
    assert status_word(ws) == 0
    compare_full(w, out, lse)


@pytest.mark.parametrize("d,dtype", [(64, torch.bfloat16), (128, torch.float16)])
def test_paired_short_cross_sequences(d, dtype):
    """Short sequences with separate query / key spans and all three mask types (bottom-right
    with fewer keys than queries leaves leading rows without keys; empty key spans)."""
    rng = np.random.default_rng(90 + d)
    B = 41
    lq = rng.integers(1, 129, size=B)
    lkv = rng.integers(0, 129, size=B)
    lkv[:3] = [0, 128, 5]
    lq[:3] = [9, 128, 100]
    codes = rng.integers(0, 3, size=B).astype(np.uint8)
    q_starts = np.concatenate([[0], np.cumsum(lq + 3)[:-1]]).astype(np.int32)
    kv_starts = (np.concatenate([[0], np.cumsum(lkv + 1)[:-1]]) + 7).astype(np.int32)
    T = int(max(q_starts[-1] + lq[-1], kv_starts[-1] + lkv[-1]) + 2)
    w = workloads.from_lengths("cross", [T], [0], heads_q=2, heads_kv=2, head_dim=d, dtype=dtype, seed=d)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lkv)]).astype(np.int32)
    dev = lambda a: torch.from_numpy(a).cuda()
    ws = workspace()
    out, lse = vlp.thd_attn_fwd(w.q.cuda(), w.k.cuda(), w.v.cuda(), dev(cu_q), dev(cu_k), dev(q_starts),
                                dev(kv_starts), dev(codes), B, 128, w.softmax_scale, workspace=ws)
    torch.cuda.synchronize()
    assert status_word(ws) == 0
    ref, ref_lse = oracle.thd_attention_fwd_general(w.q, w.k, w.v, cu_q, cu_k, q_starts, kv_starts, codes, B,
                                                    w.softmax_scale)
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    seen = np.isfinite(ref_lse)
    assert_out_close(o, ref, dtype, "cross")
    assert np.abs(l[seen] - ref_lse[seen]).max() <= LSE_ATOL
    assert np.all(np.isneginf(l[~seen]))
    assert np.all(o[~seen.any(axis=0)] == 0.0)
    assert (~seen).sum() > 0


@pytest.mark.parametrize("d,dtype", [(64, torch.float16), (128, torch.bfloat16)])
def test_packed_tiles_of_tiny_sequences(d, dtype):
    """Runs of tiny sequences without gaps fill a packed tile with up to 128 sequences of one
    row; runs that end exactly at a tile's last row or key; all three mask types; members
    whose key span is empty or longer / shorter than their query span."""
    rng = np.random.default_rng(110 + d)
    B = 600
    lq = rng.integers(1, 4, size=B)
    lq[:128] = 1                                   # one group of 128 one-row sequences
    lq[128:130] = [64, 64]                         # a group that ends at row 127
    lkv = lq.copy()
    sel = rng.choice(np.arange(130, B), 80, replace=False)
    lkv[sel] = rng.integers(0, 6, size=80)
    codes = rng.integers(0, 3, size=B).astype(np.uint8)
    q_gap = np.where(rng.random(B) < 0.2, rng.integers(1, 5, size=B), 0)
    q_gap[:130] = 0
    q_starts = np.concatenate([[0], np.cumsum(lq + q_gap)[:-1]]).astype(np.int32)
    kv_starts = (np.concatenate([[0], np.cumsum(lkv)[:-1]]) + 3).astype(np.int32)
    T = int(max(q_starts[-1] + lq[-1], kv_starts[-1] + lkv[-1]) + 4)
    w = workloads.from_lengths("tiny", [T], [0], heads_q=4, heads_kv=2, head_dim=d, dtype=dtype, seed=d + 3)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lkv)]).astype(np.int32)
    dev = lambda a: torch.from_numpy(a).cuda()
    ws = workspace()
    out, lse = vlp.thd_attn_fwd(w.q.cuda(), w.k.cuda(), w.v.cuda(), dev(cu_q), dev(cu_k), dev(q_starts),
                                dev(kv_starts), dev(codes), B, 8, w.softmax_scale, workspace=ws)
    torch.cuda.synchronize()
    assert status_word(ws) == 0
    ref, ref_lse = oracle.thd_attention_fwd_general(w.q, w.k, w.v, cu_q, cu_k, q_starts, kv_starts, codes, B,
                                                    w.softmax_scale)
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    seen = np.isfinite(ref_lse)
    assert_out_close(o, ref, dtype, "tiny")
    assert np.array_equal(np.isfinite(l), seen)
    assert np.abs(l[seen] - ref_lse[seen]).max() <= LSE_ATOL


def test_packed_groups_without_keys():
    """Packed groups whose sequences have no keys at all (the tile visits no KV tile), next
    to groups that have some: rows without keys are exact zeros with -inf LSE."""
    lq = np.array([5, 7, 3, 9, 2, 4, 6, 1], dtype=np.int64)
    lkv = np.array([0, 0, 0, 0, 3, 4, 0, 2], dtype=np.int64)
    codes = np.array([0, 1, 2, 0, 1, 2, 0, 0], dtype=np.uint8)
    q_starts = np.concatenate([[0], np.cumsum(lq)[:-1]]).astype(np.int32)
    q_starts[4:] += 200   # a second run, in another group
    kv_starts = np.concatenate([[0], np.cumsum(lkv)[:-1]]).astype(np.int32) + 50
    B = len(lq)
    T = int(max(q_starts[-1] + lq[-1], kv_starts[-1] + lkv[-1]) + 3)
    w = workloads.from_lengths("nokeys", [T], [0], heads_q=2, heads_kv=1, head_dim=64, dtype=torch.bfloat16,
                               seed=41)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lkv)]).astype(np.int32)
    dev = lambda a: torch.from_numpy(a).cuda()
    ws = workspace()
    out, lse = vlp.thd_attn_fwd(w.q.cuda(), w.k.cuda(), w.v.cuda(), dev(cu_q), dev(cu_k), dev(q_starts),
                                dev(kv_starts), dev(codes), B, 16, w.softmax_scale, workspace=ws)
    torch.cuda.synchronize()
    assert status_word(ws) == 0
    ref, ref_lse = oracle.thd_attention_fwd_general(w.q, w.k, w.v, cu_q, cu_k, q_starts, kv_starts, codes, B,
                                                    w.softmax_scale)
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    seen = np.isfinite(ref_lse)
    assert_out_close(o, ref, torch.bfloat16, "no keys")
    assert np.array_equal(np.isfinite(l), seen)
    assert np.abs(l[seen] - ref_lse[seen]).max() <= LSE_ATOL
    assert np.all(o[:, :, :][~seen.any(axis=0)] == 0.0)
    assert (~seen[:, q_starts[0]:q_starts[3] + lq[3]]).all()   # the first run sees no key


def test_packing_is_decided_per_chunk():
    """One launch, two scheduler chunks: in the first, every short sequence is followed by a
    long one (nothing to pack: one tile per (sequence, head)); in the second, runs of tiny
    sequences are packed.  Both kinds of short tile and the long blocks in one launch."""
    rng = np.random.default_rng(123)
    B = 700
    lens = np.empty(B, dtype=np.int64)
    lens[:512:2] = rng.integers(1, 129, size=256)
    lens[1:512:2] = rng.integers(129, 300, size=256)
    lens[512:] = rng.integers(1, 12, size=B - 512)
    causal = rng.random(B) < 0.5
    gaps = rng.integers(0, 4, size=B)
    w = workloads.from_lengths("chunks", lens, causal, gaps_before=gaps, trailing=3, heads_q=2, heads_kv=1,
                               head_dim=64, dtype=torch.bfloat16, seed=31, with_padded=True)
    ws = workspace()
    out, lse = run_gpu(w, workspace=ws, max_seqlen=256)   # the packing layout
    assert status_word(ws) == 0
    compare_full(w, out, lse)


@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_gqa_groups(group):
    w = workloads.from_lengths("gqa", [200, 77, 300], [1, 0, 1], gaps_before=[0, 3, 1], heads_q=8,
                               heads_kv=8 // group, head_dim=64, dtype=torch.bfloat16, seed=group)
    out, lse = run_gpu(w)
    compare_full(w, out, lse)


def test_empty_batch_zeroes_everything():
    w = workloads.make("tiny_mixed")
    dev = to_device(w)
    out = torch.full_like(dev["q"], 7.0)
    lse = torch.zeros((w.num_heads_q, w.total_tokens), dtype=torch.float32, device="cuda")
    vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], batch_size=0, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_zero_length_sequences_and_lse_optional():
    w = workloads.from_lengths("zeros", [5, 0, 7, 0, 130], [1, 1, 0, 0, 1], gaps_before=[0, 2, 0, 4, 1],
                               heads_q=2, head_dim=64, dtype=torch.bfloat16, seed=8, with_padded=True)
    out, lse = run_gpu(w)
    compare_full(w, out, lse)
    out2, lse2 = run_gpu(w, return_lse=False)
    assert lse2 is None and torch.equal(out2, out)


def test_gap_contents_do_not_leak():
    outs = []
    for fill in (100.0, -1e4, 0.0):
        w = workloads.from_lengths("leak", [100, 300, 31], [1, 0, 1], gaps_before=[17, 64, 3], trailing=9,
                                   heads_q=2, head_dim=128, dtype=torch.bfloat16, seed=12, gap_fill=fill)
        out, lse = run_gpu(w)
        vr = torch.from_numpy(valid_rows(w)).cuda()
        outs.append((out[vr], lse[:, vr]))
        check_pad_rows(w, out, lse)
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


@pytest.mark.parametrize("hint,d", [(140, 64), (4096, 128)])   # the packing and the plain instantiation
def test_large_trailing_region_is_zeroed(hint, d):
    """A buffer with many more rows than the batch holds (T sized for a larger batch): the
    rows after the last sequence, which every CTA zeroes a share of, are exact zeros with
    -inf LSE over outputs that held NaN, and the sequences' rows match the oracle."""
    w = workloads.from_lengths("trail", [100, 300, 37], [1, 0, 1], gaps_before=[5, 0, 9], trailing=40000,
                               heads_q=4, head_dim=d, dtype=torch.bfloat16, seed=15)
    dev = to_device(w)
    out = torch.full_like(dev["q"], float("nan"))
    lse = torch.full((w.num_heads_q, w.total_tokens), float("nan"), dtype=torch.float32, device="cuda")
    vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], dev["padded"], dev["padded"],
                     dev["causal"], w.batch_size, hint, w.softmax_scale, out=out, lse=lse)
    torch.cuda.synchronize()
    check_pad_rows(w, out, lse)
    compare_full(w, out, lse)


def test_garbage_past_batch_is_ignored_and_deterministic():
    w = workloads.from_lengths("tail", [50, 260, 9], [0, 1, 1], heads_q=2, head_dim=64, dtype=torch.float16,
                               seed=13, capacity=16, rng=np.random.default_rng(5))
    out1, lse1 = run_gpu(w)
    out2, lse2 = run_gpu(w)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    compare_full(w, out1, lse1)


@pytest.mark.parametrize("hint", [140, 4096])   # the packing and the plain instantiation
def test_writes_stay_inside_out_and_lse(hint):
    w = workloads.from_lengths("guard", [33, 140], [1, 0], gaps_before=[2, 5], trailing=4, heads_q=2,
                               head_dim=64, dtype=torch.bfloat16, seed=14)
    dev = to_device(w)
    T, H, d = w.total_tokens, w.num_heads_q, w.head_dim
    g = 64
    obuf = torch.full((T + 2 * g, H, d), 3.0, dtype=w.dtype, device="cuda")
    lbuf = torch.full((H * T + 2 * 1024,), 5.0, dtype=torch.float32, device="cuda")
    out = obuf[g:g + T]
    lse = lbuf[1024:1024 + H * T].view(H, T)
    vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], dev["padded"], dev["padded"],
                     dev["causal"], w.batch_size, hint, w.softmax_scale, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(obuf[:g] == 3.0) and torch.all(obuf[g + T:] == 3.0)
    assert torch.all(lbuf[:1024] == 5.0) and torch.all(lbuf[1024 + H * T:] == 5.0)
    compare_full(w, out, lse)


@pytest.mark.parametrize("hint", [40, 4096])   # the packing and the plain instantiation
def test_non_monotone_metadata_does_not_fault(hint):
    """Invalid device metadata: unspecified output, but the call completes without a fault.
    Also short sequences whose rows overlap (a later one starting before an earlier one
    ends), which the packing must not put in one tile."""
    w = workloads.from_lengths("bad", [40, 40, 40], [1, 0, 1], heads_q=2, head_dim=64, dtype=torch.bfloat16,
                               seed=15)
    dev = to_device(w)
    cases = [([0, 100, 20, 10000], [-50, 90, 119, 3], dev["causal"]),
             ([0, 10, 20, 30], [5, 0, 3, 30], dev["causal"]),
             ([0, 30, 31, 60], [60, 100, 90, 120], dev["causal"]),
             (list(range(0, 45, 5)), [0, 5, 10, 15, 12, 20, 30, 35, 40], None)]
    for cu, pad, causal in cases:
        bad_cu = torch.tensor(cu, dtype=torch.int32, device="cuda")
        bad_pad = torch.tensor(pad, dtype=torch.int32, device="cuda")
        ws = workspace()
        vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], bad_cu, bad_cu, bad_pad, bad_pad, causal, len(cu) - 1, hint,
                         0.125, workspace=ws)
        torch.cuda.synchronize()
        assert status_word(ws) == 0


def test_max_seqlen_hint_picks_the_layout_not_the_result():
    """max_seqlen sizes the claim batches and, up to 256, selects packed tiles for short
    sequences: hints on the same side of 256 give the same bits, every hint is within the
    oracle's bounds, and only rows of short sequences can differ across the two sides."""
    lens = [700, 1, 129, 90, 300, 0, 257, 41, 128, 513, 7, 60, 3] * 3
    w = workloads.from_lengths("hint", lens, [i % 3 == 0 for i in range(len(lens))], heads_q=4, heads_kv=2,
                               head_dim=64, dtype=torch.bfloat16, seed=21)
    dev = to_device(w)
    plain = [run_gpu(w, dev=dev, max_seqlen=hint) for hint in (w.max_seqlen, 0, 257, 1 << 20)]
    packed = [run_gpu(w, dev=dev, max_seqlen=hint) for hint in (1, 16, 256)]
    for group in (plain, packed):
        for o, l in group[1:]:
            assert torch.equal(o, group[0][0]) and torch.equal(l, group[0][1])
        compare_full(w, *group[0])
    rows = torch.zeros(w.total_tokens, dtype=torch.bool)
    for st, L in zip(w.starts, w.lengths):
        if L > 128:
            rows[int(st):int(st) + int(L)] = True
    rows = rows.cuda()
    assert torch.equal(plain[0][0][rows], packed[0][0][rows])


def test_binding_rejects_short_metadata_and_wrong_outputs():
    """The kernels read batch_size + 1 cu_seqlens entries: a shorter buffer, or an output of
    the wrong shape, is refused before anything is launched."""
    w = workloads.make("tiny_mixed")
    dev = to_device(w)
    B = w.batch_size
    with pytest.raises(ValueError):
        vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], batch_size=B + 1)
    with pytest.raises(ValueError):
        vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], seq_is_causal=dev["causal"][:B - 1],
                         batch_size=B)
    with pytest.raises(ValueError):
        vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], batch_size=B,
                         out=torch.empty_like(dev["q"])[:-1])
    with pytest.raises(ValueError):
        vlp.thd_padding_mask(dev["cu"], B + 1, 8)
    with pytest.raises(ValueError):
        vlp.thd_padding_mask(dev["cu"], B, 8, mask=torch.empty(B * 8 - 1, dtype=torch.bool, device="cuda"))
