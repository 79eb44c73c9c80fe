"""thd_attn_fwd_noalloc: the entry point for callers that cannot allocate device memory.

It must give the same result as thd_attn_fwd (within the parity tolerances) while taking
its workspace from the library's fixed per-device buffer.  Two calls in a row also check
that the buffer's leftover state from one call does not leak into the next.  This file is
collected last, so a failure here does not hide any other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from thd_testutil import OUT_ATOL, LSE_ATOL, to_device

pytestmark = pytest.mark.gpu
vlp = pytest.importorskip("variable_length_packed_gb300")


@pytest.fixture(scope="module")
def lib():
    from variable_length_packed_gb300 import build as vbuild
    vbuild.build()
    return vlp.load_library()


@pytest.mark.parametrize("name", ["padded_gaps", "tiny_mixed", "page1_pad"])
def test_noalloc_matches_workspace_entry_point(lib, name):
    w = workloads.make(name)
    dev = to_device(w)
    ref_out, ref_lse = vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], dev["padded"],
                                        dev["padded"], dev["causal"], w.batch_size, w.max_seqlen,
                                        w.softmax_scale)
    torch.cuda.synchronize()
    P = ctypes.c_void_p
    dtype = 0 if w.dtype == torch.bfloat16 else 1
    stream = P(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full_like(dev["q"], float("nan"))
        lse = torch.full((w.num_heads_q, w.total_tokens), float("nan"), dtype=torch.float32, device="cuda")
        st = lib.thd_attn_fwd_noalloc(
            P(dev["q"].data_ptr()), P(dev["k"].data_ptr()), P(dev["v"].data_ptr()), P(dev["cu"].data_ptr()),
            P(dev["cu"].data_ptr()), P(None if dev["padded"] is None else dev["padded"].data_ptr()),
            P(None if dev["padded"] is None else dev["padded"].data_ptr()), P(dev["causal"].data_ptr()),
            w.batch_size, w.max_seqlen, ctypes.c_float(w.softmax_scale), P(out.data_ptr()), P(lse.data_ptr()),
            w.total_tokens, w.num_heads_q, w.num_heads_kv, w.head_dim, dtype, stream)
        assert st == 0, vlp.thd_status_string(st)
        torch.cuda.synchronize()
        diff = (out.float() - ref_out.float()).abs().max().item()
        assert diff <= OUT_ATOL[w.dtype], (call, diff)
        both_inf = torch.isneginf(lse) & torch.isneginf(ref_lse)
        ldiff = torch.where(both_inf, torch.zeros_like(lse), (lse - ref_lse).abs()).max().item()
        assert ldiff <= LSE_ATOL, (call, ldiff)
        assert not torch.isnan(out).any() and not torch.isnan(lse).any()


@pytest.mark.parametrize("with_lse", [True, False])
@pytest.mark.parametrize("name", ["padded_gaps", "tiny_mixed"])
def test_noalloc_python_wrapper(lib, name, with_lse):
    """The public wrapper (argument checks, marshalling, the current stream) with outputs the
    caller allocated beforehand, with and without lse, twice in a row; the buffer's status
    word, read through thd_attn_noalloc_status, stays clear."""
    w = workloads.make(name)
    dev = to_device(w)
    ref_out, ref_lse = vlp.thd_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], dev["padded"],
                                        dev["padded"], dev["causal"], w.batch_size, w.max_seqlen,
                                        w.softmax_scale)
    out = torch.empty_like(dev["q"])
    lse = torch.empty((w.num_heads_q, w.total_tokens), dtype=torch.float32, device="cuda") if with_lse else None
    for call in range(2):
        out.fill_(float("nan"))
        if lse is not None:
            lse.fill_(float("nan"))
        o, l = vlp.thd_attn_fwd_noalloc(dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], dev["padded"],
                                        dev["padded"], dev["causal"], w.batch_size, w.max_seqlen, w.softmax_scale,
                                        out, lse)
        assert o is out and l is lse
        assert vlp.thd_attn_noalloc_status() == 0
        diff = (out.float() - ref_out.float()).abs().max().item()
        assert diff <= OUT_ATOL[w.dtype], (call, diff)
        if lse is not None:
            both_inf = torch.isneginf(lse) & torch.isneginf(ref_lse)
            ldiff = torch.where(both_inf, torch.zeros_like(lse), (lse - ref_lse).abs()).max().item()
            assert ldiff <= LSE_ATOL, (call, ldiff)
        assert not torch.isnan(out).any()


def test_noalloc_reports_a_wait_that_ran_out(lib):
    """A wait that runs out inside the no-allocation call (the failure path's test setting:
    a 1 ns limit and the injected wait) is reported through thd_attn_noalloc_status, and the
    next normal call clears the word and gives the bits of a call made before it."""
    w = workloads.make("long_context_small")
    dev = to_device(w)
    out = torch.empty_like(dev["q"])
    lse = torch.empty((w.num_heads_q, w.total_tokens), dtype=torch.float32, device="cuda")
    args = (dev["q"], dev["k"], dev["v"], dev["cu"], dev["cu"], dev["padded"], dev["padded"], dev["causal"],
            w.batch_size, w.max_seqlen, w.softmax_scale, out, lse)
    before = [t.clone() for t in vlp.thd_attn_fwd_noalloc(*args)]
    assert vlp.thd_attn_noalloc_status() == 0
    prev = vlp.thd_set_wait_limit_ns(1)
    assert vlp.thd_set_wait_injection(True) is False
    try:
        vlp.thd_attn_fwd_noalloc(*args)
        status = vlp.thd_attn_noalloc_status()
    finally:
        assert vlp.thd_set_wait_injection(False) is True
        assert vlp.thd_set_wait_limit_ns(prev) == 1
    assert status & vlp.STATUS_WAIT_TIMEOUT, status
    after = vlp.thd_attn_fwd_noalloc(*args)
    assert vlp.thd_attn_noalloc_status() == 0
    assert torch.equal(after[0], before[0]) and torch.equal(after[1], before[1])
