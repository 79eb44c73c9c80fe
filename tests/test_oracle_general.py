"""Pins for the general attention oracle (separate q / kv sequences, per-sequence mask type),
the partial-result merge and the cross-attention padding mask.

* The context-parallel example of the Megatron-LM issue: split the 7 keys into the two
  ranks' chunks (keys 0-3 and 4-6), attend every query to each chunk, merge: the result
  must be the printed full-attention output (tests/golden/page1_full_attention.txt).
* The two-call pad_between_seqs example: merging the two calls gives the mixed call.
* torch's fp64 scaled_dot_product_attention with a boolean mask (a library routine) on
  rectangular (Lq != Lkv) sequences for each mask type.
* Special cases: equal lengths (bottom-right == top-left, and the self-attention oracle),
  a single query under bottom-right (sees every key), merge with an empty partial.
* The cross-attention mask space of the padding-mask PR's Equivalence section: 202100 cases.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from conftest import read_golden

S8 = math.sqrt(8.0)


def fp16(x):
    return torch.tensor(np.asarray(x), dtype=torch.float64).to(torch.float16).double().numpy()


def test_page1_context_parallel_merge_gives_printed_output():
    g = read_golden("page1_full_attention.txt")
    x = workloads.make("page1").q            # [7, 1, 8]: four ones then three twos
    cu_q = np.array([0, 7], np.int32)
    out_a, lse_a = oracle.thd_attention_fwd_general(x, x, x, cu_q, np.array([0, 4], np.int32), None,
                                                    np.array([0], np.int32), None, 1, 1 / S8)
    out_b, lse_b = oracle.thd_attention_fwd_general(x, x, x, cu_q, np.array([0, 3], np.int32), None,
                                                    np.array([4], np.int32), None, 1, 1 / S8)
    out, lse = oracle.merge_partials(out_a, lse_a, out_b, lse_b)
    for r in range(7):
        assert np.all(np.abs(fp16(out[r, 0]) - float(g[f"row {r}"])) <= 0.5e-4)
    # each chunk alone is a convex combination of constant values
    np.testing.assert_allclose(out_a[:, 0, :], 1.0, atol=1e-15)
    np.testing.assert_allclose(out_b[:, 0, :], 2.0, atol=1e-15)
    assert abs(lse[0, 0] - math.log(4 * math.exp(S8) + 3 * math.exp(2 * S8))) < 1e-12


def test_two_call_merge_equals_mixed_call():
    g = read_golden("page2_two_call.txt")
    w = workloads.make("tiny_mixed")
    ints = lambda key: np.array([int(t) for t in g[key].split()], dtype=np.int32)
    oc, lc = oracle.thd_attention_fwd_general(w.q, w.k, w.v, ints("causal_call.cu_seqlens"),
                                              ints("causal_call.cu_seqlens"),
                                              ints("causal_call.cu_seqlens_padded"),
                                              ints("causal_call.cu_seqlens_padded"), [1] * 4, 4,
                                              w.softmax_scale)
    of, lf = oracle.thd_attention_fwd_general(w.q, w.k, w.v, ints("full_call.cu_seqlens"),
                                              ints("full_call.cu_seqlens"),
                                              ints("full_call.cu_seqlens_padded"),
                                              ints("full_call.cu_seqlens_padded"), None, 3, w.softmax_scale)
    out, lse = oracle.merge_partials(oc, lc, of, lf)
    ref, ref_lse = oracle.thd_attention_fwd(w.q, w.k, w.v, w.cu_seqlens, w.cu_seqlens, None, None,
                                            w.seq_is_causal, w.batch_size, w.softmax_scale)
    np.testing.assert_allclose(out, ref, atol=1e-14)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-13)


def _rect_case(seed, lq, lkv, heads_q=4, heads_kv=2, d=16):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(lq, heads_q, d, generator=g).to(torch.bfloat16)
    k = torch.randn(lkv, heads_kv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(lkv, heads_kv, d, generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("lq,lkv", [(5, 9), (9, 5), (1, 7), (7, 1), (12, 12), (3, 30)])
@pytest.mark.parametrize("mtype", [0, 1, 2])
def test_general_against_torch_sdpa_with_mask(lq, lkv, mtype):
    q, k, v = _rect_case(lq * 100 + lkv, lq, lkv)
    scale = 0.3
    out, lse = oracle.thd_attention_fwd_general(q, k, v, [0, lq], [0, lkv], None, None, [mtype], 1, scale)
    i = torch.arange(lq)[:, None]
    j = torch.arange(lkv)[None, :]
    if mtype == 0:
        allowed = torch.ones(lq, lkv, dtype=torch.bool)
    elif mtype == 1:
        allowed = j <= i
    else:
        allowed = j <= i + (lkv - lq)
    qq = q.double().transpose(0, 1)
    kk = k.double().repeat_interleave(2, dim=1).transpose(0, 1)
    vv = v.double().repeat_interleave(2, dim=1).transpose(0, 1)
    rows = allowed.any(dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(qq[:, rows], kk, vv, attn_mask=allowed[rows],
                                                           scale=scale)
    np.testing.assert_allclose(out[rows.numpy()], ref.transpose(0, 1).numpy(), atol=1e-12)
    assert np.all(out[~rows.numpy()] == 0) and np.all(np.isneginf(lse[:, ~rows.numpy()]))
    z = (qq @ kk.transpose(-1, -2) * scale).masked_fill(~allowed, float("-inf"))
    np.testing.assert_allclose(lse[:, rows.numpy()], torch.logsumexp(z[:, rows], -1).numpy(), atol=1e-12)


def test_general_reduces_to_self_attention_and_mask_types_coincide():
    w = workloads.from_lengths("gen", [5, 17, 9, 1], [1, 0, 1, 1], gaps_before=[2, 3, 1, 4], trailing=2,
                               heads_q=4, heads_kv=2, head_dim=16, seed=21)
    ref, ref_lse = oracle.thd_attention_fwd(w.q, w.k, w.v, w.cu_seqlens, w.cu_seqlens, w.cu_seqlens_padded,
                                            w.cu_seqlens_padded, w.seq_is_causal, w.batch_size, w.softmax_scale)
    for codes in (w.seq_is_causal, np.where(w.seq_is_causal > 0, 2, 0)):   # top-left and bottom-right
        out, lse = oracle.thd_attention_fwd_general(w.q, w.k, w.v, w.cu_seqlens, w.cu_seqlens,
                                                    w.cu_seqlens_padded, w.cu_seqlens_padded, codes,
                                                    w.batch_size, w.softmax_scale)
        np.testing.assert_allclose(out, ref, atol=1e-13)
        np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


def test_single_query_bottom_right_sees_every_key():
    q, k, v = _rect_case(3, 1, 11)
    full = oracle.thd_attention_fwd_general(q, k, v, [0, 1], [0, 11], None, None, [0], 1, 0.25)
    br = oracle.thd_attention_fwd_general(q, k, v, [0, 1], [0, 11], None, None, [2], 1, 0.25)
    tl = oracle.thd_attention_fwd_general(q, k, v, [0, 1], [0, 11], None, None, [1], 1, 0.25)
    np.testing.assert_array_equal(full[0], br[0])
    np.testing.assert_allclose(tl[0][0], v[0].double().repeat_interleave(2, dim=0).numpy(), atol=1e-15)


@pytest.mark.parametrize("split", [1, 4, 13, 31])
def test_merge_of_key_split_equals_full(split):
    q, k, v = _rect_case(50 + split, 20, 32)
    full = oracle.thd_attention_fwd_general(q, k, v, [0, 20], [0, 32], None, None, [0], 1, 0.2)
    a = oracle.thd_attention_fwd_general(q, k, v, [0, 20], [0, split], None, [0], [0], 1, 0.2)
    b = oracle.thd_attention_fwd_general(q, k, v, [0, 20], [0, 32 - split], None, [split], [0], 1, 0.2)
    out, lse = oracle.merge_partials(*a, *b)
    np.testing.assert_allclose(out, full[0], atol=1e-13)
    np.testing.assert_allclose(lse, full[1], atol=1e-12)
    out2, lse2 = oracle.merge_partials(*b, *a)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_merge_with_empty_partial_is_identity():
    rng = np.random.default_rng(4)
    out_a = rng.standard_normal((6, 2, 8))
    lse_a = rng.standard_normal((2, 6))
    lse_a[1, 3] = -np.inf
    out_a[3, 1] = 0.0
    out_b = np.zeros_like(out_a)
    lse_b = np.full_like(lse_a, -np.inf)
    out, lse = oracle.merge_partials(out_a, lse_a, out_b, lse_b)
    np.testing.assert_array_equal(out, out_a)
    np.testing.assert_array_equal(lse, lse_a)


def enumerate_cross_cases():
    for sq in range(1, 6):
        for skv in range(1, 6):
            for B in range(1, 4):
                pairs = list(itertools.product(range(sq + 1), range(skv + 1)))
                for combo in itertools.product(pairs, repeat=B):
                    lq = [p[0] for p in combo]
                    lk = [p[1] for p in combo]
                    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
                    ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
                    yield cq, ck, B, sq, skv


def test_cross_mask_exhaustive_case_count_and_forms_agree():
    expected = int(read_golden("mask_case_counts.txt")["cross_attention_cases"])
    n = 0
    for cq, ck, B, sq, skv in enumerate_cross_cases():
        a = oracle.padding_mask_cross_loop(cq, ck, B, sq, skv)
        b = oracle.padding_mask_cross_formula(cq, ck, B, sq, skv)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
        n += 1
    assert n == expected
