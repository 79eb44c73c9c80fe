"""Pins for the fp64 attention oracle: each check rests on something other than the oracle.

* the values the Megatron-LM context-parallel issue prints (tests/golden/page1_*.txt);
* closed forms of the constant-input case (full and causal policies);
* the per-sequence policy definition and the two-call ``pad_between_seqs`` identity of the
  TransformerEngine per-sequence causal policy PR (tests/golden/page2_two_call.txt);
* torch's fp64 ``scaled_dot_product_attention`` on CPU (a library routine) per sequence;
* brute force with scalar ``math.exp`` on tiny inputs;
* invariants: pad rows, gap-content independence, buffer tails never read.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from conftest import read_golden

S8 = math.sqrt(8.0)


def run_oracle(w, **over):
    args = dict(q=w.q, k=w.k, v=w.v, cu_seqlens_q=w.cu_seqlens, cu_seqlens_kv=w.cu_seqlens,
                cu_seqlens_q_padded=w.cu_seqlens_padded, cu_seqlens_kv_padded=w.cu_seqlens_padded,
                seq_is_causal=w.seq_is_causal, batch_size=w.batch_size,
                softmax_scale=w.softmax_scale)
    args.update(over)
    return oracle.thd_attention_fwd(**args)


def fp16(x):
    return torch.tensor(np.asarray(x), dtype=torch.float64).to(torch.float16).double().numpy()


# --- page 1: constant-input case -------------------------------------------------------

def test_page1_printed_values():
    g = read_golden("page1_full_attention.txt")
    w = workloads.make("page1")
    out, _ = run_oracle(w)
    for r in range(int(g["rows"])):
        printed = float(g[f"row {r}"])
        got = fp16(out[r, 0, :])
        # printed with 4 decimals: the fp16 value must round to it
        assert np.all(np.abs(got - printed) <= 0.5e-4 + 1e-12), (r, got, printed)


def test_page1_closed_form_full():
    w = workloads.make("page1")
    out, lse = run_oracle(w)
    # logits are sqrt(8)*q*k; four keys equal 1, three equal 2
    o1 = (4 + 6 * math.exp(S8)) / (4 + 3 * math.exp(S8))
    o2 = (4 + 6 * math.exp(2 * S8)) / (4 + 3 * math.exp(2 * S8))
    l1 = math.log(4 * math.exp(S8) + 3 * math.exp(2 * S8))
    l2 = math.log(4 * math.exp(2 * S8) + 3 * math.exp(4 * S8))
    np.testing.assert_allclose(out[:4, 0, :], o1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(out[4:, 0, :], o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0, :4], l1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 4:], l2, rtol=0, atol=1e-12)
    assert abs(o1 - 1.92694929) < 1e-8 and abs(o2 - 1.99536361) < 1e-8


def test_page1_closed_form_causal():
    w = workloads.make("page1")
    out, lse = run_oracle(w, seq_is_causal=np.array([1], dtype=np.uint8))
    e2 = math.exp(2 * S8)
    np.testing.assert_array_equal(out[:4, 0, :], 1.0)      # only ones are visible
    np.testing.assert_allclose(out[4, 0, :], (4 + 2 * e2) / (4 + e2), atol=1e-13)
    np.testing.assert_allclose(out[5, 0, :], (4 + 4 * e2) / (4 + 2 * e2), atol=1e-13)
    np.testing.assert_allclose(out[6, 0, :], (4 + 6 * e2) / (4 + 3 * e2), atol=1e-13)
    for i in range(4):   # row i sees i+1 keys with logit sqrt(8)
        assert abs(lse[0, i] - (S8 + math.log(i + 1))) < 1e-12


def test_page1_pad_row_is_zero_and_ignored():
    w = workloads.make("page1_pad")
    out, lse = run_oracle(w)
    ref, ref_lse = run_oracle(workloads.make("page1"))
    np.testing.assert_array_equal(out[:7], ref)
    np.testing.assert_array_equal(lse[:, :7], ref_lse)
    assert np.all(out[7] == 0.0) and np.isneginf(lse[0, 7])


def test_page1_cp_dump_rank0():
    """The buggy CP run equals full attention over 3 ones + 3 twos (rank-0 rows)."""
    g = read_golden("page1_cp_dump.txt")
    x = torch.tensor([1.0] * 3 + [2.0] * 3, dtype=torch.float16)[:, None, None].expand(6, 1, 8)
    out, _ = oracle.thd_attention_fwd(x, x, x, [0, 6], [0, 6], None, None, None, 1,
                                      1.0 / S8)
    for r in range(3):
        assert abs(fp16(out[r, 0, 0]) - float(g[f"rank0 row {r}"])) <= 0.5e-4


# --- page 2: per-sequence policy -----------------------------------------------------------

def test_mixed_policy_equals_per_sequence_scalar_policy():
    w = workloads.make("tiny_mixed")
    out, lse = run_oracle(w)
    for b in range(w.batch_size):
        s, L = int(w.starts[b]), int(w.lengths[b])
        sub = slice(s, s + L)
        o1, l1 = oracle.thd_attention_fwd(w.q[sub], w.k[sub], w.v[sub], [0, L], [0, L], None,
                                          None, [int(w.causal[b])], 1, w.softmax_scale)
        np.testing.assert_array_equal(out[sub], o1)
        np.testing.assert_array_equal(lse[:, sub], l1)


def test_two_call_pad_between_seqs_sum():
    g = read_golden("page2_two_call.txt")
    toks = g["tokens"]
    w = workloads.make("tiny_mixed")
    assert len(toks) == w.total_tokens
    # policy of each sequence as the token string states it
    runs, prev = [], None
    for c in toks:
        if c != prev:
            runs.append(c)
        prev = c
    assert [c.isdigit() for c in runs] == list(w.causal)
    ints = lambda key: np.array([int(t) for t in g[key].split()], dtype=np.int32)
    out_c, lse_c = run_oracle(w, cu_seqlens_q=ints("causal_call.cu_seqlens"),
                              cu_seqlens_kv=ints("causal_call.cu_seqlens"),
                              cu_seqlens_q_padded=ints("causal_call.cu_seqlens_padded"),
                              cu_seqlens_kv_padded=ints("causal_call.cu_seqlens_padded"),
                              seq_is_causal=np.ones(4, np.uint8), batch_size=4)
    out_f, lse_f = run_oracle(w, cu_seqlens_q=ints("full_call.cu_seqlens"),
                              cu_seqlens_kv=ints("full_call.cu_seqlens"),
                              cu_seqlens_q_padded=ints("full_call.cu_seqlens_padded"),
                              cu_seqlens_kv_padded=ints("full_call.cu_seqlens_padded"),
                              seq_is_causal=None, batch_size=3)
    out, lse = run_oracle(w)
    np.testing.assert_array_equal(out_c + out_f, out)
    # each call has -inf LSE exactly on the other policy's rows
    np.testing.assert_array_equal(np.logaddexp(lse_c, lse_f), lse)
    causal_rows = np.array([c.isdigit() for c in toks])
    assert np.all(np.isneginf(lse_c[:, ~causal_rows])) and np.all(np.isneginf(lse_f[:, causal_rows]))


# --- library routine: torch SDPA in fp64 on CPU ---------------------------------------------

@pytest.mark.parametrize("name", ["tiny_mixed", "padded_gaps"])
def test_against_torch_sdpa_fp64(name):
    w = workloads.make(name)
    if name == "padded_gaps":   # keep the CPU time small: 4 heads
        w.q, w.k, w.v = w.q[:, :4].contiguous(), w.k[:, :4].contiguous(), w.v[:, :4].contiguous()
    out, lse = run_oracle(w)
    for b in range(w.batch_size):
        s, L = int(w.starts[b]), int(w.lengths[b])
        q = w.q[s:s + L].double().transpose(0, 1)
        k = w.k[s:s + L].double().transpose(0, 1)
        v = w.v[s:s + L].double().transpose(0, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, is_causal=bool(w.causal[b]), scale=w.softmax_scale)
        np.testing.assert_allclose(out[s:s + L], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
        z = (q @ k.transpose(-1, -2)) * w.softmax_scale
        if w.causal[b]:
            z = z.masked_fill(~torch.ones(L, L, dtype=torch.bool).tril(), float("-inf"))
        np.testing.assert_allclose(lse[:, s:s + L], torch.logsumexp(z, -1).numpy(), atol=1e-12)


def test_gqa_against_torch_sdpa_fp64():
    rng = np.random.default_rng(11)
    w = workloads.from_lengths("gqa_small", [5, 17, 9], [1, 0, 1], gaps_before=[2, 3, 1],
                               heads_q=8, heads_kv=2, head_dim=16, seed=11)
    out, _ = run_oracle(w)
    for b in range(3):
        s, L = int(w.starts[b]), int(w.lengths[b])
        q = w.q[s:s + L].double().transpose(0, 1)
        k = w.k[s:s + L].double().repeat_interleave(4, dim=1).transpose(0, 1)
        v = w.v[s:s + L].double().repeat_interleave(4, dim=1).transpose(0, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, is_causal=bool(w.causal[b]), scale=w.softmax_scale)
        np.testing.assert_allclose(out[s:s + L], ref.transpose(0, 1).numpy(), atol=1e-12)
    del rng


# --- brute force on tiny inputs --------------------------------------------------------------

def test_brute_force_scalar_loops():
    w = workloads.from_lengths("bf", [1, 4, 3], [1, 0, 1], gaps_before=[1, 0, 2], trailing=1,
                               heads_q=2, heads_kv=1, head_dim=4, seed=5)
    out, lse = run_oracle(w)
    q, k, v = w.q.double().tolist(), w.k.double().tolist(), w.v.double().tolist()
    valid = set()
    for b in range(3):
        s, L = int(w.starts[b]), int(w.lengths[b])
        for h in range(2):
            for i in range(L):
                valid.add(s + i)
                ws = []
                for j in range(L):
                    if w.causal[b] and j > i:
                        continue
                    dot = sum(q[s + i][h][c] * k[s + j][0][c] for c in range(4))
                    ws.append((math.exp(dot * w.softmax_scale), j))
                tot = sum(e for e, _ in ws)
                for c in range(4):
                    ref = sum(e * v[s + j][0][c] for e, j in ws) / tot
                    assert abs(out[s + i, h, c] - ref) < 1e-13
                assert abs(lse[h, s + i] - math.log(tot)) < 1e-13
    for r in range(w.total_tokens):
        if r not in valid:
            assert np.all(out[r] == 0) and np.all(np.isneginf(lse[:, r]))


# --- invariants ------------------------------------------------------------------------------

def test_gap_contents_do_not_matter():
    base = workloads.from_lengths("gaps", [7, 1, 12], [1, 1, 0], gaps_before=[3, 5, 2],
                                  trailing=4, heads_q=2, head_dim=8, seed=9)
    outs = []
    for fill in (100.0, 0.0, -1e4):
        w = workloads.from_lengths("gaps", [7, 1, 12], [1, 1, 0], gaps_before=[3, 5, 2],
                                   trailing=4, heads_q=2, head_dim=8, seed=9, gap_fill=fill)
        outs.append(run_oracle(w))
    for o, l in outs[1:]:
        np.testing.assert_array_equal(o, outs[0][0])
        np.testing.assert_array_equal(l, outs[0][1])
    out, lse = run_oracle(base)
    np.testing.assert_array_equal(out, outs[0][0])


def test_causal_first_row_is_first_value_and_rows_are_convex():
    w = workloads.from_lengths("inv", [6, 9], [1, 1], heads_q=1, head_dim=8, seed=3)
    out, _ = run_oracle(w)
    for b in range(2):
        s = int(w.starts[b])
        np.testing.assert_array_equal(out[s, 0], w.v[s, 0].double().numpy())
    # V == 1 everywhere: every output row of a valid token is exactly a convex combination of 1s
    w.v = torch.ones_like(w.v)
    out1, _ = run_oracle(w)
    np.testing.assert_allclose(out1, 1.0, atol=1e-15)


def test_buffer_tail_never_read():
    w = workloads.make("long_context")   # buffers sized for 64 sequences, garbage past 8
    assert len(w.cu_seqlens) == 65 and w.batch_size == 8
    starts, lengths = oracle.sequence_spans(w.cu_seqlens, None, w.batch_size)
    assert lengths.sum() == 131072 and np.all(lengths >= 1)
    np.testing.assert_array_equal(starts, np.concatenate([[0], np.cumsum(lengths)[:-1]]))


def test_empty_batch():
    w = workloads.make("tiny_mixed")
    out, lse = run_oracle(w, batch_size=0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
