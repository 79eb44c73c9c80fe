"""The kernels' failure path, made to run on purpose: every wait of a kernel on its own
pipeline is bounded, and thd_set_wait_limit_ns shortens the bound so that waits run out.

A call whose waits run out must return, set THD_STATUS_WAIT_TIMEOUT in its status word,
and leave the device usable: a normal call right after it, in the same process, gives
the same bits as a call made before it, and those bits agree with the fp64 oracle.  The
limit is a plain host-side setting read into each launch's parameters; nothing faults,
traps or hangs: the waits that run out end the kernel's loops, and each CTA then lets
the copies and MMAs it started finish before it releases its tensor memory.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from thd_testutil import compare_full, compare_sampled, run_gpu, to_device

pytestmark = pytest.mark.gpu
vlp = pytest.importorskip("variable_length_packed_gb300")

SHORT_LIMIT_NS = 1   # a wait still pending after its first poll runs out


def status_word(ws):
    return int(ws[8:12].cpu().numpy().view(np.uint32)[0])


def workspace(n=None):
    return torch.zeros(n or vlp.thd_attn_workspace_size(), dtype=torch.uint8, device="cuda")


class short_waits:
    """A short wait limit, and the injected wait that runs out whatever the timing (a
    pipeline fast enough that every wait completes within the hardware's first suspended
    poll would otherwise let no wait run out)."""

    def __enter__(self):
        self.prev = vlp.thd_set_wait_limit_ns(SHORT_LIMIT_NS)
        assert vlp.thd_set_wait_injection(True) is False

    def __exit__(self, *exc):
        assert vlp.thd_set_wait_injection(False) is True
        assert vlp.thd_set_wait_limit_ns(self.prev) == SHORT_LIMIT_NS


def test_limit_setter_round_trip():
    prev = vlp.thd_set_wait_limit_ns(123)
    assert prev == 2_000_000_000                 # the default
    assert vlp.thd_set_wait_limit_ns(0) == 123   # 0 restores the default
    assert vlp.thd_set_wait_limit_ns(0) == 2_000_000_000


@pytest.mark.parametrize("name,hint", [("long_context_small", None), ("padded_gaps", None), ("padded_gaps", 512),
                                       ("many_short_tiny", 128)])
def test_forward_waits_run_out_then_recover(name, hint):
    """The warp-specialised forward (the plain instantiation on long sequences, and the
    packing one with a short max_seqlen hint): waits run out, the status bit is set, and
    the next normal call gives the bits of the call made before."""
    if name == "many_short_tiny":
        rng = np.random.default_rng(7)
        lens = np.clip(rng.geometric(1 / 24, size=900), 1, 128)
        w = workloads.from_lengths(name, lens, rng.random(900) < 0.3, gaps_before=rng.integers(0, 4, 900),
                                   heads_q=8, head_dim=64, dtype=torch.float16, seed=7, with_padded=True)
    else:
        w = workloads.make(name)
    dev = to_device(w)
    over = {} if hint is None else {"max_seqlen": hint}
    ws = workspace()
    before = run_gpu(w, dev=dev, workspace=ws, **over)
    assert status_word(ws) == 0
    with short_waits():
        run_gpu(w, dev=dev, workspace=ws, **over)
        torch.cuda.synchronize()
    assert status_word(ws) & vlp.STATUS_WAIT_TIMEOUT, "no wait ran out under the short limit"
    after = run_gpu(w, dev=dev, workspace=ws, **over)
    assert status_word(ws) == 0
    assert torch.equal(after[0], before[0]) and torch.equal(after[1], before[1])
    if w.total_tokens <= 8192:
        compare_full(w, *after)
    else:
        rng = np.random.default_rng(3)
        pairs = [(b, int(h)) for b in range(w.batch_size) for h in rng.choice(w.num_heads_q, 2, replace=False)]
        compare_sampled(w, after[0], after[1], pairs, lambda L: [0, 127, 128, L // 2, L - 1])


def test_serial_forward_recovers_after_short_waits():
    """The kernel for other head dims (here 40): its waits are on its own MMAs, which
    may complete within the first polls, so the bit is not required; the call returns,
    and the next normal call gives the earlier bits."""
    w = workloads.from_lengths("serial", [700, 129, 3000, 64], [1, 0, 1, 0], gaps_before=[0, 3, 9, 1],
                               heads_q=4, heads_kv=2, head_dim=40, dtype=torch.bfloat16, seed=17)
    dev = to_device(w)
    ws = workspace()
    before = run_gpu(w, dev=dev, workspace=ws)
    with short_waits():
        run_gpu(w, dev=dev, workspace=ws)
        torch.cuda.synchronize()
    after = run_gpu(w, dev=dev, workspace=ws)
    assert status_word(ws) == 0
    assert torch.equal(after[0], before[0]) and torch.equal(after[1], before[1])
    compare_full(w, *after)


def test_backward_waits_run_out_then_recover():
    w = workloads.make("long_context_small")
    dev = to_device(w)
    out, lse = run_gpu(w, dev=dev)
    dout = workloads.grad_output(w, 9).cuda()
    need = vlp.load_library().thd_attn_bwd_workspace_size(w.total_tokens, w.num_heads_q, w.head_dim)
    ws = workspace(need)

    def bwd():
        g = vlp.thd_attn_bwd(dev["q"], dev["k"], dev["v"], out, lse, dout, dev["cu"], dev["cu"], None, None,
                             dev["causal"], w.batch_size, w.max_seqlen, w.softmax_scale, workspace=ws)
        torch.cuda.synchronize()
        return g

    before = bwd()
    assert status_word(ws) == 0
    with short_waits():
        bwd()
    assert status_word(ws) & vlp.STATUS_WAIT_TIMEOUT, "no wait ran out under the short limit"
    after = bwd()
    assert status_word(ws) == 0
    # dK and dV accumulate in a fixed order (bit for bit); dQ tiles are added to an fp32
    # accumulator by atomic reductions whose order varies from run to run, so dQ is compared
    # to its own scale: far below the parity bound (2e-2 of the largest gradient)
    assert torch.equal(after[1], before[1]) and torch.equal(after[2], before[2])
    dq_a, dq_b = after[0].float(), before[0].float()
    assert (dq_a - dq_b).abs().max().item() <= 2e-3 * dq_b.abs().max().item()
