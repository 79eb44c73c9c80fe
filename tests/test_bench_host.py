"""Host-side checks of bench.py: the effective-FLOP count, the multi-rank timing path
(two gloo ranks on CPU) and the reference (oracle) arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import torch

import bench
import workloads
from conftest import ROOT


def test_effective_flops_counts_unmasked_pairs():
    w = workloads.from_lengths("f", [1, 5, 3, 8], [1, 0, 1, 1], heads_q=3, head_dim=16, seed=0)
    pairs = 0
    for L, c in zip(w.lengths, w.causal):
        pairs += sum(1 for i in range(L) for j in range(L) if (j <= i or not c))
    assert bench.effective_flops(w) == 4 * 16 * 3 * pairs


def test_window_pairs_match_the_oracle_band():
    import oracle
    w = workloads.from_lengths("wp", [1, 37, 300, 129], [1, 0, 1, 0], heads_q=2, head_dim=16, seed=0)
    for left, right in ((-1, -1), (5, 0), (0, 0), (64, 64), (-1, 3), (1000, 7)):
        ref = 0
        for L, c in zip(w.lengths, w.causal):
            for i in range(int(L)):
                lo, hi = oracle.visible_range(i, int(L), int(L), 1 if c else 0, (left, right))
                ref += hi - lo
        assert bench.window_pairs(w, left, right) == ref, (left, right)


def test_attn_bytes_formula():
    w = workloads.from_lengths("b", [4, 6], [1, 0], heads_q=4, heads_kv=2, head_dim=8, seed=0)
    T = w.total_tokens
    assert bench.attn_bytes(w) == T * 4 * 8 * 2 * 2 + T * 2 * 8 * 2 * 2 + T * 4 * 4


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench as b
    ws, r, _ = b.dist_setup()
    assert dist.get_backend() == "gloo"
    b.barrier(ws)
    t = b.max_over_ranks(1.5 * (r + 1), ws, torch.device("cpu"))
    q.put((r, ws, t))
    dist.destroy_process_group()


def test_two_rank_max_over_ranks_gloo():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 3.0), (1, 2, 3.0)]


def test_reference_arm_prints_oracle_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny_mixed", "--steps", "1", "--warmup", "3", "--ref-budget", "0.2"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["warmup"] >= 3


def test_recorded_traffic_follows_the_workload():
    """The committed DRAM record applies to the workload it was captured on (its own figure)
    and to the one it was scaled to; any other workload reports no traffic."""
    import bench
    full = bench.recorded_traffic("attn_fwd", "long_context")
    small = bench.recorded_traffic("attn_fwd", "long_context_small")
    if full is None:   # the record no longer matches the kernel sources
        assert small is None
        return
    assert small is not None and abs(full - 4 * small) < 1.0
    assert bench.recorded_traffic("attn_fwd", "many_short") is None
    assert bench.recorded_traffic("attn_fwd") == full


def test_other_workloads_use_their_own_seed_and_gap_fill():
    """The batches timed beside the step draw Q/K/V from their own seed (padded gaps 1,
    mixed GQA 2, long context 3, many short 4), with the gap rows as the batch states."""
    for name, seed in (("padded_gaps", 1), ("mixed_gqa", 2), ("long_context", 3), ("many_short", 4)):
        assert workloads.make(name, tensors=False).seed == seed, name
    ow, q, k, v = bench.other_inputs("padded_gaps", "cpu")
    rq, rk, rv = workloads.device_qkv(ow, "cpu", seed=1)
    assert torch.equal(q, rq) and torch.equal(k, rk) and torch.equal(v, rv)
    valid = torch.zeros(ow.total_tokens, dtype=torch.bool)
    for s, L in zip(ow.starts, ow.lengths):
        valid[int(s):int(s) + int(L)] = True
    assert (~valid).any() and torch.all(q[~valid] == 100.0) and torch.all(v[~valid] == 100.0)
    assert not torch.any(q[valid] == 100.0)


def test_library_rebuild_follows_source_contents(tmp_path, monkeypatch):
    """build._stale() compares a hash of the sources' contents (and the flags) with the one
    stored beside the library: a newer file time alone does not rebuild, a changed byte does."""
    from variable_length_packed_gb300 import build as vbuild
    csrc, inc = tmp_path / "pkg" / "csrc", tmp_path / "include"
    csrc.mkdir(parents=True)
    inc.mkdir()
    (csrc / "a.cu").write_text("int a;\n")
    (inc / "h.h").write_text("#define X 1\n")
    lib = tmp_path / "pkg" / "lib.so"
    monkeypatch.setattr(vbuild, "CSRC", str(csrc))
    monkeypatch.setattr(vbuild, "ROOT", str(tmp_path))
    monkeypatch.setattr(vbuild, "LIB", str(lib))
    monkeypatch.setattr(vbuild, "STAMP", str(lib) + ".sha256")
    assert vbuild._stale()                                   # no library
    lib.write_bytes(b"\0")
    assert vbuild._stale()                                   # no stamp
    (tmp_path / "pkg" / "lib.so.sha256").write_text(vbuild.source_hash() + "\n")
    assert not vbuild._stale()
    os.utime(csrc / "a.cu", (4e9, 4e9))                      # newer time, same bytes
    assert not vbuild._stale()
    (inc / "h.h").write_text("#define X 2\n")                # same size, other bytes
    assert vbuild._stale()
    (inc / "h.h").write_text("#define X 1\n")
    assert not vbuild._stale()
    assert vbuild._stale(["-DTHD_EXTRA"])                    # other flags
