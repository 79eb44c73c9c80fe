"""thd_padding_mask on the GPU against the mask oracle: byte-exact.

Covers the exhaustive space of "[PyTorch] Build the attention padding mask without host
syncs" (Equivalence: lengths in [0, S], S = 1..8, B = 1..4, with and without a longer
cu_seqlens buffer: 35368 cases), the 4096 x 8192 workload, unaligned output pointers,
rows longer than max_seqlen and non-monotone buffers.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from test_oracle_mask import enumerate_self_cases

pytestmark = pytest.mark.gpu
vlp = pytest.importorskip("variable_length_packed_gb300")


def gpu_mask(cu_np, B, S, offset=0):
    cu = torch.from_numpy(np.asarray(cu_np, dtype=np.int32)).cuda()
    buf = torch.full((B * S + offset + 32,), 0xAB, dtype=torch.uint8, device="cuda")
    view = buf[offset:offset + B * S]
    vlp.thd_padding_mask(cu, B, S, mask=view)
    host = buf.cpu().numpy()
    assert np.all(host[:offset] == 0xAB) and np.all(host[offset + B * S:] == 0xAB), "write outside mask"
    return host[offset:offset + B * S].reshape(B, 1, 1, S)


def test_exhaustive_small_space():
    n = 0
    bad = 0
    for cu, B, S in enumerate_self_cases():
        got = gpu_mask(cu, B, S, offset=n % 16)
        ref = oracle.padding_mask_formula(cu, B, S).astype(np.uint8)
        bad += int(not np.array_equal(got, ref))
        n += 1
    assert n == 35368 and bad == 0


def test_large_workload_bit_exact():
    mw = workloads.make_mask()
    got = gpu_mask(mw.cu_seqlens, mw.batch_size, mw.max_seqlen)
    ref = oracle.padding_mask_formula(mw.cu_seqlens, mw.batch_size, mw.max_seqlen).astype(np.uint8)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("B,S,offset", [(3, 5, 1), (7, 33, 3), (5, 16, 0), (9, 17, 15), (1, 1, 7), (64, 100, 9),
                                         (33, 48, 0), (130, 256, 0), (3, 8192, 0), (2000, 32, 0), (11, 64, 4)])
def test_shapes_and_alignment(B, S, offset):
    rng = np.random.default_rng(B * 100 + S)
    lens = rng.integers(0, S + 3, size=B)             # includes rows longer than S
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cu = np.concatenate([cu, rng.integers(-1000, 1000, size=5).astype(np.int32)])  # garbage tail
    got = gpu_mask(cu, B, S, offset)
    ref = oracle.padding_mask_formula(cu, B, S).astype(np.uint8)
    assert np.array_equal(got, ref)


def test_non_monotone_and_returned_tensor():
    cu = np.array([10, 3, 3, 40, 2], dtype=np.int32)   # negative and oversized lengths
    for S in (12, 32):                                 # flat and row-per-warp paths
        got = gpu_mask(cu, 4, S)
        assert np.array_equal(got, oracle.padding_mask_formula(cu, 4, S).astype(np.uint8))
    m = vlp.thd_padding_mask(torch.tensor([0, 2, 5], dtype=torch.int32, device="cuda"), 2, 4)
    assert m.dtype == torch.bool and m.shape == (2, 1, 1, 4)
    assert m.cpu().numpy().reshape(2, 4).tolist() == [[False, False, True, True], [False, False, False, True]]
