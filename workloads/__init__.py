"""Seeded synthetic inputs for packed variable-length (THD) attention.

This module only *draws* inputs: sequence lengths, per-sequence causal flags,
inter-sequence gaps, the cumulative-length buffers that describe them, and the
Q/K/V token tensors.  It holds none of the attention or mask arithmetic, so the
fp64 oracle (``oracle/``) and the CUDA library (``variable_length_packed_gb300``)
can both be fed from it without sharing any of the method's code.

Recipe (the same for every workload):

* metadata comes from ``numpy.random.default_rng(seed)``, drawn in the order
  lengths, policies, gaps (then any garbage that fills oversized buffers);
* Q/K/V come from ``torch.Generator('cpu').manual_seed(seed)``: ``randn`` in
  fp32 for Q, then K, then V, each cast to the workload dtype;
* rows that belong to no sequence ("gap" rows) keep their random values unless
  the workload says otherwise (``gap_fill``).

Workloads follow the shapes of the pages' own examples: the 7-sequence
``[111aaa222bb3344cccc]`` batch of the TransformerEngine per-sequence causal
policy PR (review comment with the ``pad_between_seqs`` example), the 7-token
constant-input case of the Megatron-LM context-parallel padding issue, and
larger packed batches with the length mixes listed in ``WORKLOADS``.
"""
from __future__ import annotations

from dataclasses import dataclass, field
import math

import numpy as np
import torch

__all__ = ["Workload", "MaskWorkload", "WORKLOADS", "make", "make_mask", "from_lengths"]


@dataclass
class Workload:
    """One packed THD batch.

    ``cu_seqlens`` / ``cu_seqlens_padded`` / ``seq_is_causal`` are the host
    copies of the device buffers a caller would pass; they may be longer than
    ``batch_size + 1`` (resp. ``batch_size``), in which case the tail holds
    garbage that must never be read.  ``cu_seqlens_padded`` is ``None`` when the
    batch has no gaps.
    """

    name: str
    batch_size: int
    lengths: np.ndarray            # int64 [B] valid tokens per sequence
    causal: np.ndarray             # bool  [B]
    starts: np.ndarray             # int64 [B] first row of each sequence in the packed buffer
    cu_seqlens: np.ndarray         # int32 [>= B+1]
    cu_seqlens_padded: np.ndarray | None  # int32 [>= B+1] or None
    seq_is_causal: np.ndarray      # uint8 [>= B]
    total_tokens: int
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    dtype: torch.dtype
    softmax_scale: float
    max_seqlen: int
    q: torch.Tensor = field(repr=False)   # [T, Hq, d] CPU, dtype
    k: torch.Tensor = field(repr=False)   # [T, Hkv, d]
    v: torch.Tensor = field(repr=False)   # [T, Hkv, d]
    seed: int = 0                         # the seed Q/K/V are drawn from
    gap_fill: float | None = None         # value of every gap row of Q/K/V (None: random like the rest)


@dataclass
class MaskWorkload:
    name: str
    batch_size: int
    max_seqlen: int
    lengths: np.ndarray       # int64 [B]
    cu_seqlens: np.ndarray    # int32 [>= B+1]


def _qkv(seed, T, hq, hkv, d, dtype):
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn((T, hq, d), generator=g, dtype=torch.float32).to(dtype)
    k = torch.randn((T, hkv, d), generator=g, dtype=torch.float32).to(dtype)
    v = torch.randn((T, hkv, d), generator=g, dtype=torch.float32).to(dtype)
    return q, k, v


def _layout(lengths, gaps_before, trailing=0):
    """Row offsets of each sequence when sequence b is preceded by gaps_before[b] pad rows."""
    lengths = np.asarray(lengths, dtype=np.int64)
    gaps_before = np.asarray(gaps_before, dtype=np.int64)
    starts = np.zeros(len(lengths), dtype=np.int64)
    pos = 0
    for b in range(len(lengths)):
        pos += int(gaps_before[b])
        starts[b] = pos
        pos += int(lengths[b])
    return starts, pos + int(trailing)


def _buffers(lengths, starts, total, causal, capacity=None, rng=None):
    B = len(lengths)
    cap = B if capacity is None else capacity
    cu = np.zeros(cap + 1, dtype=np.int64)
    cu[1:B + 1] = np.cumsum(lengths)
    padded = np.zeros(cap + 1, dtype=np.int64)
    padded[:B] = starts
    padded[B] = total
    flags = np.zeros(max(cap, 1), dtype=np.uint8)
    flags[:B] = causal.astype(np.uint8)
    if cap > B:
        assert rng is not None
        cu[B + 1:] = rng.integers(-2**31, 2**31 - 1, size=cap - B, dtype=np.int64)
        padded[B + 1:] = rng.integers(-2**31, 2**31 - 1, size=cap - B, dtype=np.int64)
        flags[B:] = rng.integers(0, 256, size=cap - B, dtype=np.uint8)
    return cu.astype(np.int32), padded.astype(np.int32), flags


def from_lengths(name, lengths, causal, *, gaps_before=None, trailing=0, heads_q=1,
                 heads_kv=None, head_dim=64, dtype=torch.bfloat16, seed=0,
                 softmax_scale=None, gap_fill=None, capacity=None, rng=None,
                 with_padded=None):
    """Build a Workload from explicit lengths / flags / gaps (Q/K/V drawn from ``seed``)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    causal = np.asarray(causal, dtype=bool)
    B = len(lengths)
    if gaps_before is None:
        gaps_before = np.zeros(B, dtype=np.int64)
    starts, T = _layout(lengths, gaps_before, trailing)
    if with_padded is None:
        with_padded = bool(np.any(np.asarray(gaps_before) != 0) or trailing != 0)
    heads_kv = heads_q if heads_kv is None else heads_kv
    cu, padded, flags = _buffers(lengths, starts, T, causal, capacity, rng)
    if _MAKE_TENSORS:
        q, k, v = _qkv(seed, T, heads_q, heads_kv, head_dim, dtype)
    else:
        q = k = v = None
    if gap_fill is not None and q is not None:
        valid = np.zeros(T, dtype=bool)
        for s, L in zip(starts, lengths):
            valid[s:s + L] = True
        pad_rows = torch.from_numpy(~valid)
        for t in (q, k, v):
            t[pad_rows] = gap_fill
    scale = 1.0 / math.sqrt(head_dim) if softmax_scale is None else softmax_scale
    return Workload(
        name=name, batch_size=B, lengths=lengths, causal=causal, starts=starts,
        cu_seqlens=cu, cu_seqlens_padded=padded if with_padded else None,
        seq_is_causal=flags, total_tokens=int(T), num_heads_q=heads_q,
        num_heads_kv=heads_kv, head_dim=head_dim, dtype=dtype,
        softmax_scale=float(scale), max_seqlen=int(lengths.max()) if B else 0,
        q=q, k=k, v=v, seed=int(seed), gap_fill=gap_fill)


# ---------------------------------------------------------------------------
# The five packed batches (plus the page-1 constant case)
# ---------------------------------------------------------------------------

def tiny_mixed():
    """The 19-token batch 111aaa222bb3344cccc: numbered sequences causal, lettered full."""
    return from_lengths("tiny_mixed", [3, 3, 3, 2, 2, 2, 4], [1, 0, 1, 0, 1, 1, 0],
                        heads_q=2, head_dim=64, dtype=torch.bfloat16, seed=0,
                        softmax_scale=1.0 / 8.0)


def page1_constant(pad_row=False):
    """7 tokens, one head, d=8, fp16: Q=K=V=1 on tokens 0-3 and 2 on tokens 4-6, full context.

    With ``pad_row`` the buffer holds an 8th token set to 100 (the padded token of the
    context-parallel example), and ``cu_seqlens_padded = [0, 8]`` marks it as pad.
    """
    T = 8 if pad_row else 7
    x = torch.empty((T, 1, 8), dtype=torch.float16)
    x[:4] = 1.0
    x[4:7] = 2.0
    if pad_row:
        x[7] = 100.0
    lengths = np.array([7], dtype=np.int64)
    starts = np.array([0], dtype=np.int64)
    cu = np.array([0, 7], dtype=np.int32)
    padded = np.array([0, T], dtype=np.int32)
    return Workload(
        name="page1_pad" if pad_row else "page1", batch_size=1, lengths=lengths,
        causal=np.array([False]), starts=starts, cu_seqlens=cu,
        cu_seqlens_padded=padded if pad_row else None,
        seq_is_causal=np.zeros(1, dtype=np.uint8), total_tokens=T, num_heads_q=1,
        num_heads_kv=1, head_dim=8, dtype=torch.float16,
        softmax_scale=1.0 / math.sqrt(8.0), max_seqlen=8,
        q=x.clone(), k=x.clone(), v=x.clone())


def padded_gaps(seed=1):
    """16 causal sequences, lengths U{1..512}, each slot start rounded up to a multiple of 64,
    pad rows filled with 100.0."""
    rng = np.random.default_rng(seed)
    B = 16
    lengths = rng.integers(1, 513, size=B)
    causal = np.ones(B, dtype=bool)
    gaps = np.zeros(B, dtype=np.int64)
    pos = 0
    for b in range(B):
        start = -(-pos // 64) * 64
        gaps[b] = start - pos
        pos = start + lengths[b]
    trailing = -(-pos // 64) * 64 - pos
    return from_lengths("padded_gaps", lengths, causal, gaps_before=gaps, trailing=trailing,
                        heads_q=16, head_dim=128, dtype=torch.bfloat16, seed=seed,
                        gap_fill=100.0, with_padded=True)


def mixed_gqa(seed=2):
    """64 sequences, lengths log-uniform in [128, 4096], causal ~ Bernoulli(0.5),
    gaps U{0..63} between sequences, 32 query heads over 8 KV heads, d=128."""
    rng = np.random.default_rng(seed)
    B = 64
    lengths = np.rint(np.exp(rng.uniform(math.log(128), math.log(4096), size=B))).astype(np.int64)
    causal = rng.random(B) < 0.5
    gaps = np.zeros(B, dtype=np.int64)
    gaps[1:] = rng.integers(0, 64, size=B - 1)
    return from_lengths("mixed_gqa", lengths, causal, gaps_before=gaps, heads_q=32,
                        heads_kv=8, head_dim=128, dtype=torch.bfloat16, seed=seed,
                        with_padded=True)


def long_context_lengths(rng, B=8, total=131072):
    raw = rng.uniform(8192, 32768, size=B)
    scaled = raw * (total / raw.sum())
    base = np.floor(scaled).astype(np.int64)
    rem = total - int(base.sum())
    order = np.argsort(-(scaled - base), kind="stable")
    base[order[:rem]] += 1
    return base


def long_context(seed=3):
    """8 sequences, lengths U(8192, 32768) rescaled to 131072 tokens, 6 causal / 2 full,
    no gaps; metadata buffers sized for 64 sequences with garbage past the batch."""
    rng = np.random.default_rng(seed)
    B = 8
    lengths = long_context_lengths(rng, B)
    causal = np.zeros(B, dtype=bool)
    causal[rng.permutation(B)[:6]] = True
    return from_lengths("long_context", lengths, causal, heads_q=16, head_dim=128,
                        dtype=torch.bfloat16, seed=seed, capacity=64, rng=rng,
                        with_padded=False)


def long_context_small(seed=3):
    """The long-context mix at a quarter of the size (4 sequences, 32768 tokens, 3 causal /
    1 full, 16 heads, d=128, bf16): Q/K/V still larger than L2, one launch about a millisecond.
    Used for profiler captures of the same kernel."""
    lengths = long_context_lengths(np.random.default_rng(seed), 4, total=32768)
    causal = np.array([True, True, False, True])
    return from_lengths("long_context_small", lengths, causal, heads_q=16, head_dim=128,
                        dtype=torch.bfloat16, seed=seed, with_padded=False)


def many_short(seed=4):
    """4096 sequences, lengths geometric (mean 64) clipped to [1, 256], causal ~ Bernoulli(0.3),
    gaps U{0..15} between sequences, 32 heads, d=64, fp16."""
    rng = np.random.default_rng(seed)
    B = 4096
    lengths = np.clip(rng.geometric(1.0 / 64.0, size=B), 1, 256).astype(np.int64)
    causal = rng.random(B) < 0.3
    gaps = np.zeros(B, dtype=np.int64)
    gaps[1:] = rng.integers(0, 16, size=B - 1)
    return from_lengths("many_short", lengths, causal, gaps_before=gaps, heads_q=32,
                        head_dim=64, dtype=torch.float16, seed=seed, with_padded=True)


def late_long(seed=6, long_first=False):
    """1500 sequences, three scheduler chunks of 512: 1496 with lengths U{32..256} (causal ~
    Bernoulli(0.5)) and 4 of 12288 tokens (causal, full, causal, full) placed last, in the last
    chunk (long_first: the same sequences with the 4 long ones first); 4 heads, d=128, bf16, no
    gaps.  The long sequences' blocks are the longest units of the launch."""
    rng = np.random.default_rng(seed)
    short = rng.integers(32, 257, size=1496)
    short_causal = rng.random(1496) < 0.5
    long_ = np.full(4, 12288)
    long_causal = np.array([True, False, True, False])
    if long_first:
        lengths, causal = np.r_[long_, short], np.r_[long_causal, short_causal]
    else:
        lengths, causal = np.r_[short, long_], np.r_[short_causal, long_causal]
    return from_lengths("late_long_first" if long_first else "late_long", lengths, causal, heads_q=4,
                        head_dim=128, dtype=torch.bfloat16, seed=seed, with_padded=False)


WORKLOADS = {
    "tiny_mixed": tiny_mixed,
    "page1": lambda: page1_constant(False),
    "page1_pad": lambda: page1_constant(True),
    "padded_gaps": padded_gaps,
    "mixed_gqa": mixed_gqa,
    "long_context": long_context,
    "long_context_small": long_context_small,
    "many_short": many_short,
    "late_long": late_long,
    "late_long_first": lambda: late_long(long_first=True),
}


_MAKE_TENSORS = True


def make(name, tensors=True):
    """Build workload `name`.  With tensors=False only the metadata is drawn (q/k/v are
    None); device_qkv() then draws same-shaped tensors directly on a GPU."""
    global _MAKE_TENSORS
    _MAKE_TENSORS = tensors
    try:
        return WORKLOADS[name]()
    finally:
        _MAKE_TENSORS = True


def device_qkv(w, device, seed=None):
    """Q/K/V of w's shapes and dtype drawn with a seeded generator on `device`
    (N(0,1) in fp32, then cast), for timing runs that need no host copy.  The seed is the
    workload's own unless given; gap rows get the workload's gap_fill when it has one.
    (A device generator draws other numbers than the CPU one, with the same distribution.)"""
    seed = w.seed if seed is None else seed
    g = torch.Generator(device=device).manual_seed(seed)
    shape_q = (w.total_tokens, w.num_heads_q, w.head_dim)
    shape_kv = (w.total_tokens, w.num_heads_kv, w.head_dim)
    q = torch.randn(shape_q, generator=g, device=device, dtype=torch.float32).to(w.dtype)
    k = torch.randn(shape_kv, generator=g, device=device, dtype=torch.float32).to(w.dtype)
    v = torch.randn(shape_kv, generator=g, device=device, dtype=torch.float32).to(w.dtype)
    if w.gap_fill is not None:
        valid = torch.zeros(w.total_tokens, dtype=torch.bool)
        for s, L in zip(w.starts, w.lengths):
            valid[int(s):int(s) + int(L)] = True
        pad = (~valid).to(device)
        for t in (q, k, v):
            t[pad] = w.gap_fill
    return q, k, v


def make_mask(name="mask_many", seed=4):
    """Padding-mask workload: batch 4096, max_seqlen 8192, lengths U{0..8192}."""
    if name != "mask_many":
        raise KeyError(name)
    rng = np.random.default_rng(seed)
    B, S = 4096, 8192
    lengths = rng.integers(0, S + 1, size=B).astype(np.int64)
    cu = np.zeros(B + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    return MaskWorkload(name=name, batch_size=B, max_seqlen=S, lengths=lengths,
                        cu_seqlens=cu.astype(np.int32))


def merge_inputs(T, H, d, dtype, seed):
    """Two partial attention results for merge tests: out_* uniform in [-2, 2] ([T, H, d],
    dtype), lse_* ~ N(0, 3^2) ([H, T], float32); about 5 % of (head, row) entries have
    lse_a = -inf, 5 % lse_b = -inf and 2 % both, with the matching out rows zero."""
    g = torch.Generator("cpu").manual_seed(seed)
    out_a = (torch.rand((T, H, d), generator=g) * 4 - 2).to(dtype)
    out_b = (torch.rand((T, H, d), generator=g) * 4 - 2).to(dtype)
    lse_a = torch.randn((H, T), generator=g) * 3
    lse_b = torch.randn((H, T), generator=g) * 3
    u = torch.rand((H, T), generator=g)
    none_a = u < 0.05
    none_b = (u >= 0.05) & (u < 0.10)
    both = (u >= 0.10) & (u < 0.12)
    for lse, out, m in ((lse_a, out_a, none_a | both), (lse_b, out_b, none_b | both)):
        lse[m] = float("-inf")
        out.permute(1, 0, 2)[m] = 0
    return out_a, lse_a, out_b, lse_b


def grad_output(w, seed):
    """dO for backward tests: N(0, 1) of out's shape [T, Hq, d] in w's dtype (CPU)."""
    g = torch.Generator("cpu").manual_seed(seed)
    return torch.randn((w.total_tokens, w.num_heads_q, w.head_dim), generator=g,
                       dtype=torch.float32).to(w.dtype)
