"""Benchmark: packed THD attention forward (+ padding mask) on GB300.

One step = the whole hot path over one synthetic packed batch: thd_attn_fwd on the
long-context workload (8 sequences, 131072 tokens, 16 heads, d=128, bf16, 6 causal /
2 full-context, metadata buffers sized for 64 sequences) followed by thd_padding_mask
for the same cu_seqlens.  `value` is effective attention TFLOP/s over all ranks
(4*d*Hq per unmasked query-key pair), inputs resident in HBM.  The padding mask is also
timed alone on the 4096 x 8192 mask workload (GB/s against HBM peak).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs its own replica of the workload (weak scaling, no
collective on the data path; the barrier and max-over-ranks timing use the process
group).  `--impl reference` times the fp64 CPU oracle on host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
_NCORES = len(os.sched_getaffinity(0))
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_NCORES))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "THD attn fwd effective TFLOP/s and % of GB300 dense BF16 peak; mask GB/s"
WORKLOAD = "long_context"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Sources of each kernel whose profiler counters are recorded under profiles/ (a counter
# record is used only while these files are unchanged).
KERNEL_SOURCES = {
    "attn_fwd": ["variable_length_packed_gb300/csrc/" + f for f in ("ptx.cuh", "attn_common.cuh", "attn_fwd_ws.cuh")],
    "padding_mask": ["variable_length_packed_gb300/csrc/padding_mask.cu"],
}


def effective_flops(w):
    """4 * d * Hq per unmasked (query, key) pair: QK^T and PV, multiply-adds counted as 2."""
    L = w.lengths.astype(np.float64)
    pairs = np.where(w.causal, L * (L + 1) / 2, L * L).sum()
    return 4.0 * w.head_dim * w.num_heads_q * pairs


def window_pairs(w, left, right):
    """Visible (query, key) pairs of a self-attention batch under a sliding window: query i of a
    sequence sees keys max(0, i - left) .. min(L - 1, i + right) (right 0 for causal sequences),
    the band of thd_attn_fwd_window with shift 0."""
    pairs = 0
    for L, c in zip(w.lengths, w.causal):
        i = np.arange(int(L), dtype=np.int64)
        lo = np.maximum(0, i - left) if left >= 0 else np.zeros_like(i)
        r = 0 if c else right
        hi = np.minimum(int(L) - 1, i + r) if r >= 0 else np.full_like(i, int(L) - 1)
        pairs += int(np.maximum(hi - lo + 1, 0).sum())
    return float(pairs)


def attn_bytes(w):
    """Algorithmic HBM bytes of one attention launch: Q, K, V read once, O and LSE written once."""
    T, e = w.total_tokens, 2
    return T * (2 * w.num_heads_q + 2 * w.num_heads_kv) * w.head_dim * e + T * w.num_heads_q * 4


def other_inputs(name, dev):
    """Metadata of batch `name` and its Q/K/V drawn on `dev` from the batch's own seed (gap rows
    filled as the batch states)."""
    ow = workloads.make(name, tensors=False)
    return (ow, *workloads.device_qkv(ow, dev))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_sources_sha(kind):
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        path = os.path.join(ROOT, rel)
        if os.path.exists(path):
            with open(path, "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kind, workload=None):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current sources
    and the workload: the captured workload's own figure, the scaled figure for the workload
    it was scaled to, None for any other workload."""
    path = os.path.join(ROOT, "profiles", f"{kind}_traffic.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, _, v = line.partition(":")
                vals[k.strip()] = v.strip()
    if vals.get("kernel_sources_sha256") != kernel_sources_sha(kind):
        return None
    captured, _, scaled = vals.get("workload", "").partition("->")
    captured = captured.strip()
    scaled = scaled.split("(")[0].strip() or captured
    try:
        if workload is None or workload == scaled:
            return float(vals["dram_bytes_per_launch_full_workload"])
        if workload == captured:
            return float(vals["dram_bytes_per_launch_capture"])
    except (KeyError, ValueError):
        return None
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.result = self._finish()

    def _finish(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return ws, rank, local


def max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------------------------
# oracle on host cores (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------------------------

def oracle_sample(w, budget_s):
    """Time the fp64 oracle on whole query-row blocks of the workload until `budget_s` elapses.

    Returns (effective FLOP/s, description)."""
    import oracle
    group = w.num_heads_q // w.num_heads_kv
    done_pairs = 0.0
    rows_done = 0
    t0 = time.perf_counter()
    blocks = []
    for b in np.argsort(-w.lengths):
        L = int(w.lengths[b])
        for r0 in range(0, L, 512):
            blocks.append((int(b), r0, min(L, r0 + 512)))
    rng = np.random.default_rng(0)
    rng.shuffle(blocks)
    it = 0
    while time.perf_counter() - t0 < budget_s and it < len(blocks):
        b, r0, r1 = blocks[it]
        h = it % w.num_heads_q
        it += 1
        s, L = int(w.starts[b]), int(w.lengths[b])
        rows = np.arange(r0, r1)
        oracle.thd_attention_rows(w.q, w.k, w.v, s, s, L, bool(w.causal[b]), h, group, w.softmax_scale, rows)
        done_pairs += float((rows + 1).sum()) if w.causal[b] else float(len(rows) * L)
        rows_done += len(rows)
    el = time.perf_counter() - t0
    flops = 4.0 * w.head_dim * done_pairs
    desc = (f"{it} blocks of <=512 query rows (one head each) drawn from {w.name}: {rows_done} rows, "
            f"{done_pairs:.3e} unmasked pairs, {el:.1f} s")
    return flops / el, desc, el


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    w = workloads.make(args.workload)
    eff = effective_flops(w)
    per_step = []
    descs = []
    budget = min(args.ref_budget, 150.0 / (args.warmup + args.steps))
    for i in range(args.warmup + args.steps):
        rate, desc, el = oracle_sample(w, budget)
        if i >= args.warmup:
            per_step.append(rate)
            descs.append(desc)
    rate = statistics.median(per_step)
    value = rate / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": eff / rate * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": _NCORES, "kind": "oracle",
                         "sample": descs[-1]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": "fp64 numpy oracle on host cores; each step times a bounded sample of the workload and "
                "ms_per_step extrapolates that rate to the whole batch",
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    return {"workload": f"{w.name}: {w.batch_size} packed sequences, {w.total_tokens} tokens, "
                        f"{int(w.causal.sum())} causal / {int((~w.causal).sum())} full, no gaps, "
                        f"metadata buffers sized for {len(w.cu_seqlens) - 1} sequences",
            "batch": w.batch_size, "total_tokens": w.total_tokens, "heads_q": w.num_heads_q,
            "heads_kv": w.num_heads_kv, "head_dim": w.head_dim,
            "lengths": [int(x) for x in w.lengths], "causal": [bool(x) for x in w.causal],
            "mask_step": {"batch": w.batch_size, "max_seqlen": int(w.max_seqlen)},
            "l2": "inputs larger than L2 (Q/K/V 1.5 GB per step), no flush needed",
            "parallelism": "one replica per GPU"}


# ---------------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------------

def time_mask(vlp, dev, stream, peaks, reps=200):
    """thd_padding_mask on the 4096 x 8192 mask workload, as a CUDA graph of `reps` back-to-back
    launches that rotate over enough output buffers (each 33.6 MB) to hold at least twice the
    L2 cache, so every launch's lines are written back to HBM while later launches run (one
    buffer rewritten in place would stay in L2).  The same graph on a single buffer is reported
    beside it, as the L2-resident figure."""
    mw = workloads.make_mask()
    mcu = torch.from_numpy(mw.cu_seqlens).to(dev)
    mask_bytes = mw.batch_size * mw.max_seqlen + 4 * (mw.batch_size + 1)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 128 * 2**20)
    nbuf = max(2, -(-2 * l2 // (mw.batch_size * mw.max_seqlen)))
    bufs = [torch.empty((mw.batch_size, 1, 1, mw.max_seqlen), dtype=torch.bool, device=dev) for _ in range(nbuf)]

    def launch(i, rotate=True):
        vlp.thd_padding_mask(mcu, mw.batch_size, mw.max_seqlen, mask=bufs[i % nbuf if rotate else 0])

    for i in range(2 * nbuf):   # plain launches first (a profiler can select them by index)
        launch(i)
    torch.cuda.synchronize()
    per_launch = {}
    for rotate in (True, False):
        g = torch.cuda.CUDAGraph()
        s2 = torch.cuda.Stream(dev)
        s2.wait_stream(stream)
        with torch.cuda.stream(s2):
            with torch.cuda.graph(g, stream=s2):
                for i in range(reps):
                    launch(i, rotate)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        m0.record(stream)
        g.replay()
        m1.record(stream)
        torch.cuda.synchronize()
        per_launch[rotate] = m0.elapsed_time(m1) * 1e3 / reps
        del g
    mask_us = per_launch[True]
    mask_gbs = mask_bytes / (mask_us * 1e-6) / 1e9
    return {"workload": "mask_many: batch 4096, max_seqlen 8192, lengths U{0..8192}",
            "us_per_launch": mask_us, "gbs": mask_gbs, "peak_gbs": peaks["hbm_gbs"],
            "frac": mask_gbs / peaks["hbm_gbs"], "algorithmic_bytes": mask_bytes,
            "timing": f"CUDA graph of {reps} back-to-back launches rotating over {nbuf} output buffers "
                      f"({nbuf * mw.batch_size * mw.max_seqlen / 1e6:.0f} MB, at least twice the "
                      f"{l2 / 2**20:.0f} MiB L2)",
            "traffic": recorded_traffic("padding_mask"),
            "l2_resident_us_per_launch": per_launch[False],
            "l2_resident_note": "the same graph rewriting one buffer, which stays in L2 (not an HBM figure)"}


def run_gpu(args, ws, rank, local):
    import variable_length_packed_gb300 as vlp
    from variable_length_packed_gb300 import build as vbuild

    vbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    if args.mask_only:   # the mask measurement alone (for profiler captures)
        if rank == 0:
            print(json.dumps({"mask": time_mask(vlp, dev, torch.cuda.current_stream(dev), peaks)}), flush=True)
        return 0
    w = workloads.make(args.workload)
    eff = effective_flops(w)
    stream = torch.cuda.current_stream(dev)

    q, k, v = w.q.to(dev), w.k.to(dev), w.v.to(dev)
    cu = torch.from_numpy(w.cu_seqlens).to(dev)
    causal = torch.from_numpy(w.seq_is_causal).to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.num_heads_q, w.total_tokens), dtype=torch.float32, device=dev)
    wsp = torch.zeros(vlp.thd_attn_workspace_size(), dtype=torch.uint8, device=dev)
    S = int(w.max_seqlen)
    mask = torch.empty((w.batch_size, 1, 1, S), dtype=torch.bool, device=dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        vlp.thd_attn_fwd(q, k, v, cu, cu, None, None, causal, w.batch_size, S, w.softmax_scale, out=out,
                         lse=lse, workspace=wsp)
        if ev is not None:
            ev[1].record(stream)
        vlp.thd_padding_mask(cu, w.batch_size, S, mask=mask)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = int(wsp[8:12].cpu().numpy().view(np.uint32)[0])
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(ws)
        torch.cuda.synchronize()
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
    elapsed_ms = t_start.elapsed_time(t_end)
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    elapsed_ms = max_over_ranks(elapsed_ms, ws, dev)
    ms_per_step = elapsed_ms / args.steps
    value = ws * eff / (ms_per_step * 1e-3) / 1e12
    if args.attn_only:
        if rank == 0:
            print(json.dumps({"workload": w.name, "attn_ms_per_launch": attn_ms,
                              "effective_tflops": eff / (attn_ms * 1e-3) / 1e12, "status": status}), flush=True)
        return 0

    # ---- backward on the same batch (dQ, dK, dV; the forward's out / lse as inputs) ----
    backward = None
    if not args.no_backward:
        gdo = torch.Generator(device=dev).manual_seed(5)
        dout = torch.randn(w.q.shape, generator=gdo, device=dev, dtype=torch.float32).to(w.dtype)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        bws = torch.empty(vlp.load_library().thd_attn_bwd_workspace_size(w.total_tokens, w.num_heads_q,
                                                                          w.head_dim), dtype=torch.uint8, device=dev)

        def bcall():
            vlp.thd_attn_bwd(q, k, v, out, lse, dout, cu, cu, None, None, causal, w.batch_size, S, w.softmax_scale,
                             dq=dq, dk=dk, dv=dv, workspace=bws)
        for _ in range(3):
            bcall()
        torch.cuda.synchronize()
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        breps = 5
        b0.record(stream)
        for _ in range(breps):
            bcall()
        b1.record(stream)
        torch.cuda.synchronize()
        bms = b0.elapsed_time(b1) / breps
        beff = 2.5 * eff   # five products (S, dP, dV, dK, dQ) against the forward's two
        backward = {"ms_per_call": bms, "effective_tflops": beff / (bms * 1e-3) / 1e12,
                    "frac_of_bf16_peak": beff / (bms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                    "launches_per_call": 3, "flops_counted": "2.5 x forward effective FLOPs"}
        del dout, dq, dk, dv, bws

    # ---- the other packed batches: attention alone, same kernel, inputs drawn on the device ----
    others = {}
    for name in args.also:
        ow, oq, ok_, ov = other_inputs(name, dev)
        ocu = torch.from_numpy(ow.cu_seqlens).to(dev)
        opad = None if ow.cu_seqlens_padded is None else torch.from_numpy(ow.cu_seqlens_padded).to(dev)
        ocz = torch.from_numpy(ow.seq_is_causal).to(dev)
        oout = torch.empty_like(oq)
        olse = torch.empty((ow.num_heads_q, ow.total_tokens), dtype=torch.float32, device=dev)

        def ocall():
            vlp.thd_attn_fwd(oq, ok_, ov, ocu, ocu, opad, opad, ocz, ow.batch_size, ow.max_seqlen,
                             ow.softmax_scale, out=oout, lse=olse, workspace=wsp)
        for _ in range(3):
            ocall()
        torch.cuda.synchronize()
        reps = 10
        o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        o0.record(stream)
        for _ in range(reps):
            ocall()
        o1.record(stream)
        torch.cuda.synchronize()
        oms = o0.elapsed_time(o1) / reps
        oeff = effective_flops(ow)
        obytes = attn_bytes(ow)
        others[name] = {"ms_per_launch": oms, "effective_tflops": oeff / (oms * 1e-3) / 1e12,
                        "frac_of_bf16_peak": oeff / (oms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                        "algorithmic_gbs": obytes / (oms * 1e-3) / 1e9,
                        "frac_of_hbm": obytes / (oms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                        "tokens": ow.total_tokens, "batch": ow.batch_size, "heads_q": ow.num_heads_q,
                        "heads_kv": ow.num_heads_kv, "head_dim": ow.head_dim, "dtype": str(ow.dtype)}
        del oq, ok_, ov, oout, olse

    # ---- scheduler chunk order: the same 1500 sequences with their 4 longest last / first ----
    chunk_order = None
    if not args.attn_only and not args.no_chunk_order:
        cms = {}
        for name in ("late_long", "late_long_first"):
            ow, oq, ok_, ov = other_inputs(name, dev)
            ocu = torch.from_numpy(ow.cu_seqlens).to(dev)
            ocz = torch.from_numpy(ow.seq_is_causal).to(dev)
            oout = torch.empty_like(oq)
            olse = torch.empty((ow.num_heads_q, ow.total_tokens), dtype=torch.float32, device=dev)

            def ocall():
                vlp.thd_attn_fwd(oq, ok_, ov, ocu, ocu, None, None, ocz, ow.batch_size, ow.max_seqlen,
                                 ow.softmax_scale, out=oout, lse=olse, workspace=wsp)
            for _ in range(3):
                ocall()
            torch.cuda.synchronize()
            o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            o0.record(stream)
            for _ in range(10):
                ocall()
            o1.record(stream)
            torch.cuda.synchronize()
            cms[name] = o0.elapsed_time(o1) / 10
            del oq, ok_, ov, oout, olse
        chunk_order = {"workload": "1500 sequences (3 scheduler chunks): 1496 of U{32..256} tokens and 4 of 12288, "
                                   "4 heads, d=128, bf16",
                       "long_last_ms": cms["late_long"], "long_first_ms": cms["late_long_first"],
                       "long_last_over_long_first": cms["late_long"] / cms["late_long_first"]}

    # ---- sliding window (local attention, +-2048 keys around the diagonal) on the same batch ----
    window = None
    if not args.attn_only and not args.no_window:
        left = right = 2048
        wout = torch.empty_like(q)
        wlse = torch.empty_like(lse)

        def wcall():
            vlp.thd_attn_fwd(q, k, v, cu, cu, None, None, causal, w.batch_size, S, w.softmax_scale, out=wout,
                             lse=wlse, workspace=wsp, window=(left, right))
        for _ in range(3):
            wcall()
        torch.cuda.synchronize()
        wst = int(wsp[8:12].cpu().numpy().view(np.uint32)[0])
        reps = 10
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        for _ in range(reps):
            wcall()
        w1.record(stream)
        torch.cuda.synchronize()
        wms = w0.elapsed_time(w1) / reps
        weff = 4.0 * w.head_dim * w.num_heads_q * window_pairs(w, left, right)
        window = {"window": [left, right], "workload": args.workload, "ms_per_launch": wms,
                  "effective_tflops": weff / (wms * 1e-3) / 1e12,
                  "frac_of_bf16_peak": weff / (wms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                  "flops_counted": "4 * d * Hq per visible (query, key) pair in the band",
                  "device_status_word": wst}
        del wout, wlse

    # ---- padding mask alone on the 4096 x 8192 workload ----
    mask_line = time_mask(vlp, dev, stream, peaks)

    # ---- LSE merge of two partial results of the step's shape (HBM stream) ----
    # Two partial (out, LSE) of this workload's shape, the second from the forward itself
    # and the first a shifted copy: the kernel reads both and writes the merged pair.
    merge = None
    if not args.attn_only:
        mo_a, ml_a = torch.roll(out, 1, 0), torch.roll(lse, 1, 1)
        mo, ml = torch.empty_like(out), torch.empty_like(lse)
        for _ in range(3):
            vlp.thd_attn_merge(mo_a, ml_a, out, lse, out=mo, lse=ml)
        torch.cuda.synchronize()
        mreps = 20
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(mreps):
            vlp.thd_attn_merge(mo_a, ml_a, out, lse, out=mo, lse=ml)
        g1.record(stream)
        torch.cuda.synchronize()
        merge_ms = g0.elapsed_time(g1) / mreps
        Tm, Hm, dm = out.shape
        merge_bytes = Tm * Hm * (3 * dm * out.element_size() + 3 * 4)
        merge_gbs = merge_bytes / (merge_ms * 1e-3) / 1e9
        merge = {"workload": f"{args.workload} shape: two partial outputs [T={Tm}, H={Hm}, d={dm}] and LSEs",
                 "ms_per_launch": merge_ms, "gbs": merge_gbs, "peak_gbs": peaks["hbm_gbs"],
                 "frac": merge_gbs / peaks["hbm_gbs"], "algorithmic_bytes": merge_bytes,
                 "bytes_counted": "two outputs and two LSEs read, one of each written"}
        del mo_a, ml_a, mo, ml

    # ---- end to end through the public API with host buffers ----
    # Every step copies its inputs from pinned host memory and reads its outputs back.
    # Steps are pipelined the way a serving loop would run them: two device buffer sets,
    # the host->device copy of step i+1 and the device->host copy of step i-1 run on copy
    # streams while step i computes.
    hq, hk, hv = (t.pin_memory() for t in (w.q, w.k, w.v))
    hcu = torch.from_numpy(w.cu_seqlens).pin_memory()
    hcausal = torch.from_numpy(w.seq_is_causal).pin_memory()
    hout = torch.empty(w.q.shape, dtype=w.q.dtype).pin_memory()
    hlse = torch.empty((w.num_heads_q, w.total_tokens), dtype=torch.float32).pin_memory()
    hmask = torch.empty((w.batch_size, 1, 1, S), dtype=torch.bool).pin_memory()
    sets = [dict(q=q, k=k, v=v, cu=cu, causal=causal, out=out, lse=lse, mask=mask)]
    sets.append({key: torch.empty_like(t) for key, t in sets[0].items()})
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("inp", "comp", "outp")}

    def e2e_step(i):
        b = i % 2
        d = sets[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev["comp"][b])     # step i-2 finished reading this input set
            d["q"].copy_(hq, non_blocking=True)
            d["k"].copy_(hk, non_blocking=True)
            d["v"].copy_(hv, non_blocking=True)
            d["cu"].copy_(hcu, non_blocking=True)
            d["causal"].copy_(hcausal, non_blocking=True)
            ev["inp"][b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev["inp"][b])
            if i >= 2:
                s_comp.wait_event(ev["outp"][b])   # step i-2's outputs were read back
            vlp.thd_attn_fwd(d["q"], d["k"], d["v"], d["cu"], d["cu"], None, None, d["causal"], w.batch_size, S,
                             w.softmax_scale, out=d["out"], lse=d["lse"], workspace=wsp)
            vlp.thd_padding_mask(d["cu"], w.batch_size, S, mask=d["mask"])
            ev["comp"][b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comp"][b])
            hout.copy_(d["out"], non_blocking=True)
            hlse.copy_(d["lse"], non_blocking=True)
            hmask.copy_(d["mask"], non_blocking=True)
            ev["outp"][b].record(s_out)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    # as many steps as the device-timed region (at least 4): the first step's input copy and
    # the last step's output copy are not hidden behind other steps, and count once per run
    # Three timed runs; the median is reported (the host-memory side of the copies is shared
    # with the rest of the host, and its bandwidth varies from run to run); all three are
    # listed beside it.
    e_steps = max(4, args.steps)
    e2e_trials = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(ws)
        torch.cuda.synchronize()
        e0.record(s_in)
        for i in range(e_steps):
            e2e_step(i)
        e1.record(s_out)
        torch.cuda.synchronize()
        e2e_trials.append(max_over_ranks(e0.elapsed_time(e1) / e_steps, ws, dev))
    e2e_ms = sorted(e2e_trials)[1]
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hcu, hcausal))
    d2h = sum(t.numel() * t.element_size() for t in (hout, hlse, hmask))
    # the box's pinned-copy bandwidths, one copy each way (untimed; explains e2e against value)
    c0, c1, c2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    c0.record(stream)
    q.copy_(hq, non_blocking=True)
    c1.record(stream)
    hout.copy_(out, non_blocking=True)
    c2.record(stream)
    torch.cuda.synchronize()
    copy_gbs = {"h2d_gbs": hq.numel() * hq.element_size() / (c0.elapsed_time(c1) * 1e-3) / 1e9,
                "d2h_gbs": hout.numel() * hout.element_size() / (c1.elapsed_time(c2) * 1e-3) / 1e9}
    del sets[1]

    # ---- check the timed output once against the oracle on a few rows (not timed) ----
    import oracle
    rows = np.array([0, 1, 1000, int(w.lengths[0]) - 1])
    ro, rl = oracle.thd_attention_rows(w.q, w.k, w.v, 0, 0, int(w.lengths[0]), bool(w.causal[0]), 0, 1,
                                       w.softmax_scale, rows)
    got = out[torch.from_numpy(rows).to(dev), 0].float().cpu().double().numpy()
    check_err = float(np.abs(got - ro).max())

    achieved = eff / (attn_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": workload_config(w),
        "pct_of_bf16_peak": 100.0 * achieved / peaks["bf16_tflops"],
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"], "traffic": recorded_traffic("attn_fwd", args.workload),
                     "kernel": "thd attention forward", "peak_source": f"{peak_src} bf16 dense (burst)",
                     "frac_of_sustained_peak": achieved / peaks["bf16_tflops_sustained"],
                     "attn_ms_per_launch": attn_ms, "algorithmic_flops_per_launch": eff,
                     "algorithmic_bytes_per_launch": attn_bytes(w)},
        "mask": mask_line,
        "e2e": {"value": ws * eff / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "copy_bandwidth": copy_gbs,
                "trials_ms_per_step": e2e_trials, "steps_per_trial": e_steps,
                "pipelining": "two buffer sets; step i+1's H2D and step i-1's D2H overlap step i's kernels; "
                              "median of three timed runs"},
        "other_workloads": others,
        "backward": backward,
        "sliding_window": window,
        "chunk_order": chunk_order,
        "merge": merge,
        "gpu_launches": 2 * args.steps,
        "clocks": clk.result,
        "device_status_word": status,
        "sampled_check_max_abs_err": check_err,
    }
    if rank == 0 and not args.no_cpu_baseline:
        rate, desc, el = oracle_sample(w, args.cpu_budget)
        line["cpu_baseline"] = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": _NCORES, "kind": "oracle",
                                "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(workloads.WORKLOADS),
                    help="packed batch to run (default: the long-context workload the metric is quoted on)")
    ap.add_argument("--also", nargs="*", default=["padded_gaps", "mixed_gqa", "many_short"],
                    help="other packed batches whose attention launch is timed alone (after the step)")
    ap.add_argument("--no-backward", action="store_true", help="skip timing the backward pass")
    ap.add_argument("--no-window", action="store_true", help="skip timing the sliding-window forward")
    ap.add_argument("--no-chunk-order", action="store_true",
                    help="skip timing the late-long-sequence batch against its long-first twin")
    ap.add_argument("--mask-only", action="store_true",
                    help="run only the padding-mask measurement and print it; for profiler captures")
    ap.add_argument("--attn-only", action="store_true",
                    help="run only the attention launches (warm-up + timed) and print the line; "
                         "for profiler captures")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)   # timing rule: at least 3 untimed warm-up steps
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, ws, rank)
    return run_gpu(args, ws, rank, local)


if __name__ == "__main__":
    sys.exit(main())
