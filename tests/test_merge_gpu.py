"""GPU tests of the §(f) additions: per-sequence mask types with separate q / kv sequences,
the partial-result merge, and the cross-attention padding masks.  Expected values come
from the fp64 oracle on the same seeded inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from conftest import read_golden
from test_oracle_general import enumerate_cross_cases
from thd_testutil import LSE_ATOL, assert_out_close

pytestmark = pytest.mark.gpu
vlp = pytest.importorskip("variable_length_packed_gb300")


def rect_batch(d, dtype, seed):
    """Five sequences whose query and key/value spans differ in length and position."""
    lq = [250, 300, 7, 200, 130]
    lkv = [100, 64, 40, 129, 0]
    codes = [2, 1, 2, 0, 1]     # bottom-right with Lkv < Lq: the first 150 rows see no key
    qs = [0, 250, 550, 557, 757]
    ks = [887, 987, 1051, 1091, 1220]
    T = 1230
    w = workloads.from_lengths("rect", [T], [0], heads_q=4, heads_kv=2, head_dim=d, dtype=dtype, seed=seed)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lkv)]).astype(np.int32)
    return w, cu_q, cu_k, np.array(qs, np.int32), np.array(ks, np.int32), np.array(codes, np.uint8)


@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float16)])
def test_packed_short_sequences_with_separate_q_kv(d, dtype):
    """The packing instantiation (a max_seqlen hint of 128) on 300 short sequences whose
    query and key/value spans differ in length and position, with every mask type and
    sequences without keys; rows of no sequence and rows that see no key: zero out, -inf LSE."""
    rng = np.random.default_rng(d + 1)
    B = 300
    lq = rng.integers(1, 101, B)
    lkv = np.where(rng.random(B) < 0.05, 0, rng.integers(1, 121, B))
    codes = rng.integers(0, 3, B).astype(np.uint8)
    qs = np.cumsum(np.r_[0, lq[:-1] + rng.integers(0, 6, B - 1)])
    ks = qs[-1] + lq[-1] + 7 + np.cumsum(np.r_[0, lkv[:-1] + rng.integers(0, 6, B - 1)])
    T = int(ks[-1] + lkv[-1] + 3)
    w = workloads.from_lengths("rect_short", [T], [0], heads_q=4, heads_kv=2, head_dim=d, dtype=dtype, seed=d + 2)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lkv)]).astype(np.int32)
    qs, ks = qs.astype(np.int32), ks.astype(np.int32)
    dev = lambda a: torch.from_numpy(a).cuda()
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    out, lse = vlp.thd_attn_fwd(q, k, v, dev(cu_q), dev(cu_k), dev(qs), dev(ks), dev(codes), B, 128,
                                w.softmax_scale)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.thd_attention_fwd_general(w.q, w.k, w.v, cu_q, cu_k, qs, ks, codes, B, w.softmax_scale)
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    seen = np.isfinite(ref_lse)
    assert_out_close(o, ref, dtype, "packed cross")
    assert np.abs(l[seen] - ref_lse[seen]).max() <= LSE_ATOL
    assert np.all(np.isneginf(l[~seen]))
    rows_none = ~seen.any(axis=0)
    assert np.all(o[rows_none] == 0)


@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float16), (40, torch.bfloat16)])
def test_mask_types_with_separate_q_kv(d, dtype):
    w, cu_q, cu_k, qs, ks, codes = rect_batch(d, dtype, seed=d)
    dev = lambda a: torch.from_numpy(a).cuda()
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    out, lse = vlp.thd_attn_fwd(q, k, v, dev(cu_q), dev(cu_k), dev(qs), dev(ks), dev(codes), 5, 300,
                                w.softmax_scale)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.thd_attention_fwd_general(w.q, w.k, w.v, cu_q, cu_k, qs, ks, codes, 5,
                                                    w.softmax_scale)
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    seen = np.isfinite(ref_lse)
    assert_out_close(o, ref, dtype, "merge")
    assert np.abs(l[seen] - ref_lse[seen]).max() <= LSE_ATOL
    assert np.all(np.isneginf(l[~seen]))
    rows_none = ~seen.any(axis=0)
    assert np.all(o[rows_none] == 0.0)           # rows of no sequence and rows that see no key
    assert (~seen).sum() > 0                     # bottom-right rows before the diagonal, empty kv


def test_merge_matches_oracle_on_synthetic_partials():
    for d, dtype in ((128, torch.bfloat16), (64, torch.float16), (8, torch.bfloat16), (40, torch.float16)):
        oa, la, ob, lb = workloads.merge_inputs(517, 3, d, dtype, seed=d)
        out, lse = vlp.thd_attn_merge(oa.cuda(), la.cuda(), ob.cuda(), lb.cuda())
        torch.cuda.synchronize()
        ref, ref_lse = oracle.merge_partials(oa, la.numpy(), ob, lb.numpy())
        o = out.float().cpu().double().numpy()
        l = lse.cpu().double().numpy()
        fin = np.isfinite(ref_lse)
        assert_out_close(o, ref, dtype, f"merge d={d}")
        assert np.abs(l[fin] - ref_lse[fin]).max() <= 1e-5
        assert np.all(np.isneginf(l[~fin])) and np.all(o[~fin.T] == 0)


def test_merge_in_place_and_identity():
    oa, la, ob, lb = workloads.merge_inputs(300, 2, 64, torch.bfloat16, seed=7)
    ref, ref_lse = vlp.thd_attn_merge(oa.cuda(), la.cuda(), ob.cuda(), lb.cuda())
    a_out, a_lse = oa.cuda(), la.cuda()
    vlp.thd_attn_merge(a_out, a_lse, ob.cuda(), lb.cuda(), out=a_out, lse=a_lse)
    torch.cuda.synchronize()
    assert torch.equal(a_out, ref) and torch.equal(a_lse, ref_lse)
    empty_o = torch.zeros_like(oa).cuda()
    empty_l = torch.full_like(la, float("-inf")).cuda()
    o, l = vlp.thd_attn_merge(oa.cuda(), la.cuda(), empty_o, empty_l)
    torch.cuda.synchronize()
    assert torch.equal(o.cpu(), oa) and torch.equal(l.cpu(), la)


def test_page1_context_parallel_split_merged_on_gpu():
    """Each 'rank' attends every query to its own key chunk; merging gives the printed output."""
    g = read_golden("page1_full_attention.txt")
    w = workloads.make("page1")
    x = w.q.cuda()
    cu_q = torch.tensor([0, 7], dtype=torch.int32, device="cuda")
    pad_q = torch.tensor([0], dtype=torch.int32, device="cuda")
    part = []
    for lo, n in ((0, 4), (4, 3)):
        cu_k = torch.tensor([0, n], dtype=torch.int32, device="cuda")
        pad_k = torch.tensor([lo], dtype=torch.int32, device="cuda")
        part.append(vlp.thd_attn_fwd(x, x, x, cu_q, cu_k, pad_q, pad_k, None, 1, 8, 1 / math.sqrt(8)))
    out, lse = vlp.thd_attn_merge(*part[0], *part[1])
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    for r in range(7):
        assert np.all(np.abs(o[r, 0] - float(g[f"row {r}"])) <= 0.5e-4), (r, o[r, 0])


@pytest.mark.parametrize("split", [1, 128, 200, 383])
def test_key_split_attention_merged_equals_full(split):
    """Attention over keys [0, split) and [split, L) of each sequence, merged, against the
    oracle's full attention.  Bound: the partials' own 1e-2 (bf16) plus the merged value's
    rounding (half a bf16 ulp below 4: 7.8e-3) plus 2e-3 for the LSE weights: 2e-2."""
    L = 384
    w = workloads.from_lengths("split", [L, L], [0, 0], heads_q=4, heads_kv=2, head_dim=128,
                               dtype=torch.bfloat16, seed=split)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    cu_q = torch.tensor([0, L, 2 * L], dtype=torch.int32, device="cuda")
    pad_q = torch.tensor([0, L], dtype=torch.int32, device="cuda")
    parts = []
    for lo, n in ((0, split), (split, L - split)):
        cu_k = torch.tensor([0, n, 2 * n], dtype=torch.int32, device="cuda")
        pad_k = torch.tensor([lo, L + lo], dtype=torch.int32, device="cuda")
        parts.append(vlp.thd_attn_fwd(q, k, v, cu_q, cu_k, pad_q, pad_k, None, 2, L, w.softmax_scale))
    out, lse = vlp.thd_attn_merge(*parts[0], *parts[1])
    torch.cuda.synchronize()
    ref, ref_lse = oracle.thd_attention_fwd(w.q, w.k, w.v, w.cu_seqlens, w.cu_seqlens, None, None, None, 2,
                                            w.softmax_scale)
    assert np.abs(out.float().cpu().double().numpy() - ref).max() <= 2e-2
    assert np.abs(lse.cpu().double().numpy() - ref_lse).max() <= LSE_ATOL


def test_cross_mask_exhaustive_space():
    """Every case of the Equivalence section's cross-attention space (202100), batched: cases
    with the same (max_seqlen_q, max_seqlen_kv) are concatenated into one call, since each
    mask row depends only on its own two cu_seqlens entries."""
    expected = int(read_golden("mask_case_counts.txt")["cross_attention_cases"])
    groups = {}
    n = 0
    for cq, ck, B, sq, skv in enumerate_cross_cases():
        groups.setdefault((sq, skv), []).append((np.diff(cq), np.diff(ck)))
        n += 1
    assert n == expected
    for (sq, skv), cases in groups.items():
        lq = np.concatenate([c[0] for c in cases])
        lk = np.concatenate([c[1] for c in cases])
        cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
        ck = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
        B = len(lq)
        mq, mk = vlp.thd_padding_mask_cross(torch.from_numpy(cq).cuda(), torch.from_numpy(ck).cuda(), B, sq, skv)
        rq, rk = oracle.padding_mask_cross_formula(cq, ck, B, sq, skv)
        assert np.array_equal(mq.cpu().numpy(), rq) and np.array_equal(mk.cpu().numpy(), rk), (sq, skv)
