"""Benchmark of the block-scaled FP8 hot path on GB300.

Workload (one "step"): the dense block-FP8 GEMM shape sweep — m in
{8, 64, 128, 1024, 2048, 4096} x (n, k) in {(4096, 7168), (7168, 18432),
(18432, 7168), (24576, 1536), (32768, 512), (7168, 16384)} — where each of the
36 shapes runs the per-token-group activation quant (1 x 128, fp32 scales)
followed by the block-scaled GEMM against 128 x 128 block-quantized weights.
Inputs are seeded synthetic tensors (activations N(0,1) with 0.1 % x50
outliers, weights N(0, 0.02)), resident in HBM; the weights are quantized on
the GPU before timing (offline, as on the pages).

Metric: effective TFLOP/s of the whole step, sum(2 m n k) / step time, plus
per-shape GEMM microseconds, TFLOP/s, GB/s (the pages' formula, "vLLM DeepGEMM
FP8 Block GEMM 基准测试" §4.3) and fraction of the per-shape roofline.

`--impl reference` times the CPU oracle (the only reference this method has)
on a bounded sample of the same workload.  Under torchrun every rank runs the
same workload on its own GPU (replicas, weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

SWEEP_NK = [(4096, 7168), (7168, 18432), (18432, 7168), (24576, 1536), (32768, 512),
            (7168, 16384)]
SWEEP_M = [8, 64, 128, 1024, 2048, 4096]
METRIC = "block-FP8 GEMM TFLOPS & GB/s per (m,n,k); quant GB/s; % of roofline, 1 GB300"
UNIT = "TFLOP/s"
WORKLOAD = ("dense block-FP8 W8A8 shape sweep: m{8,64,128,1024,2048,4096} x "
            "(n,k){(4096,7168),(7168,18432),(18432,7168),(24576,1536),(32768,512),"
            "(7168,16384)}; per shape: 1x128 activation quant (fp32 scales) + 1x128/128x128 "
            "block-scaled FP8 GEMM, fp32 accumulate, bf16 out")
FP8_PER_BF16 = 2.0  # nominal dense fp8 : bf16 tensor-rate ratio on GB300 (4.5 : 2.25 PF)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# the pages' metric formulas (§4.3)
# ---------------------------------------------------------------------------
def pages_tflops(m, n, k, t_us):
    return 2.0 * m * n * k / (t_us * 1e-6) / 1e12


def pages_gbps(m, n, k, t_us):
    return (m * k + k * n + 2.0 * m * n) / (t_us * 1e-6) / 1e9


def gemm_alg_bytes(m, n, k):
    """Algorithmic bytes of one GEMM launch: fp8 A and W, bf16 out, fp32 scales."""
    align4 = (m + 3) // 4 * 4
    return m * k + n * k + 2 * m * n + align4 * (k // 128) * 4 + ((n + 127) // 128) * (k // 128) * 4


def quant_alg_bytes(m, k):
    """bf16 read + e4m3 write + fp32 column-major scales."""
    return 2 * m * k + m * k + (m + 3) // 4 * 4 * (k // 128) * 4


def max_over_ranks(value: float, dist, device) -> float:
    """The slowest rank's time (the job's time): all-reduce MAX over ranks.
    Returns value unchanged when dist is None (one process)."""
    if dist is None:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# The sources of the sweep's GEMM kernels, whose DRAM traffic the committed
# profile records.
KERNEL_SOURCES = ("block_scaled_fp8_quant_gb300/csrc/gemm_kernels.cu",
                  "block_scaled_fp8_quant_gb300/csrc/gemm_common.cuh",
                  "block_scaled_fp8_quant_gb300/csrc/bfq_device.cuh")


def kernel_source_hash():
    """Hash of the kernel sources' code: comments, trailing blanks and empty
    lines are left out, so that a comment edit keeps the measured profile."""
    import re

    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        code = "\n".join(line.rstrip() for line in src.splitlines() if line.strip())
        h.update(code.encode())
    return h.hexdigest()[:16]


def profile_traffic():
    """DRAM bytes per step of the GEMM launches from the committed ncu summary,
    or None when the summary is missing or was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "gemm_sweep_dram_traffic.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        return float(vals["gemm_dram_bytes_per_launch_avg"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------
SAMPLE_ROWS = 8
SAMPLE_COLS = 1024
CPU_BASELINE_SECONDS = 10.0


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_inputs(cols):
    """Bounded sample inputs (bf16 bits): per (n, k), the first `cols` weight
    rows and 8 activation rows."""
    import numpy as np
    import torch

    import bfq_synth as synth

    out = []
    for n, k in SWEEP_NK:
        w = synth.weight(cols, k, seed=n + k)
        x = synth.activation(SAMPLE_ROWS, k, seed=SAMPLE_ROWS * 31 + n)
        wb = w.contiguous().view(torch.int16).numpy().view(np.uint16)
        xb = x.contiguous().view(torch.int16).numpy().view(np.uint16)
        out.append((k, wb, xb))
    return out


def oracle_sample_step(cols=SAMPLE_COLS, threads=1, inputs=None):
    """One bounded sample of the workload on the CPU oracle: 8 activation rows
    against the first `cols` weight rows of each of the 6 (n, k) shapes (weight
    block quant of that slice, activation quant, GEMM).  With threads > 1 the
    weight rows are shared out over that many host threads in 128-row blocks,
    each thread quantizing its blocks and multiplying them (the oracle's C
    code runs outside the interpreter lock; every block is computed exactly
    as single-threaded).  Returns FLOPs done."""
    import concurrent.futures as cf

    import oracle

    inputs = inputs or _oracle_inputs(cols)
    flops = 0
    acts = [oracle.quant(xb, oracle.FMT_F32) for _, _, xb in inputs]
    blocks = [(i, c0) for i in range(len(inputs)) for c0 in range(0, cols, 128)]

    def block(job):  # weight block quant + GEMM of one 128-row weight block
        i, c0 = job
        wq, sw = oracle.weight_block_quant(inputs[i][1][c0:c0 + 128], False)
        aq, sa = acts[i]
        oracle.gemm(aq, sa, oracle.FMT_F32, wq, sw)

    if threads <= 1:
        for job in blocks:
            block(job)
    else:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(block, blocks))
    for k, _, _ in inputs:
        flops += 2 * SAMPLE_ROWS * cols * k
    return flops


def _time_oracle(threads, seconds, cols=SAMPLE_COLS):
    inputs = _oracle_inputs(cols)
    t0 = time.perf_counter()
    flops, reps = 0, 0
    while reps == 0 or time.perf_counter() - t0 < seconds:
        flops += oracle_sample_step(cols, threads, inputs)
        reps += 1
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, reps, dt


def cpu_baseline():
    """The oracle timed on the host: on every host core (the reported value)
    and on one thread, each for about CPU_BASELINE_SECONDS."""
    import oracle

    oracle.build_oracle()
    oracle.e4m3_encode([0.0])  # build the oracle's tables before threads start
    cores = host_cores()
    v1, r1, d1 = _time_oracle(1, CPU_BASELINE_SECONDS)
    vn, rn, dn = _time_oracle(cores, CPU_BASELINE_SECONDS)
    what = (f"({SAMPLE_ROWS} activation rows x first {SAMPLE_COLS} weight rows of each of the "
            f"6 (n,k) sweep shapes: weight block quant + activation quant + fp64 block GEMM)")
    return {"value": vn, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{rn} x {what}, 128-row weight blocks shared over {cores} host threads "
                      f"({dn:.1f} s)",
            "single_thread": {"value": v1, "unit": UNIT, "cores": 1,
                              "sample": f"{r1} x the same sample, one thread ({d1:.1f} s)"}}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle

    oracle.build_oracle()
    oracle.e4m3_encode([0.0])  # build the oracle's tables before threads start
    cores = host_cores()
    # The weight-row sample shrinks with the number of steps so that the whole
    # run stays near a minute and a half of CPU time (~2 s of single-thread
    # work per step at 1024 rows on the GPU machine's host cores).
    cols = max(128, min(SAMPLE_COLS, SAMPLE_COLS * 40 // max(1, args.steps + args.warmup)
                        // 128 * 128))
    inputs = _oracle_inputs(cols)
    for _ in range(args.warmup):
        oracle_sample_step(cols, cores, inputs)
    t0 = time.perf_counter()
    flops = 0
    for _ in range(args.steps):
        flops += oracle_sample_step(cols, cores, inputs)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": "bounded CPU sample"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{SAMPLE_ROWS} rows x {cols} weight rows per (n,k), "
                                   f"per step, 128-row weight blocks over {cores} host threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def build_problem(bfq, torch, dev, only=None):
    """The 36 sweep shapes.  Every shape gets its own copy of its (n, k)
    weight (quantized once, then cloned), so that no GEMM launch finds its
    weights in L2: between two reads of one copy the step streams ~2.8 GB of
    other weights (> 20x the 129 MB L2), as successive layers of a model do.
    `wq0`/`sw0` keep the group's first copy."""
    import bfq_synth as synth

    shapes = []
    for n, k in SWEEP_NK:
        if only and (only[1], only[2]) != (n, k):
            continue
        w = synth.weight(n, k, seed=n + k, device=dev)
        wq0, sw0 = bfq.weight_block_quant(w, bfq.SCALE_F32)
        del w
        first = True
        for m in SWEEP_M:
            if only and only[0] != m:
                continue
            wq, sw = (wq0, sw0) if first else (wq0.clone(), sw0.clone())
            first = False
            x = synth.activation(m, k, seed=m * 31 + n, device=dev)
            q = torch.empty((m, k), dtype=torch.float8_e4m3fn, device=dev)
            s = torch.empty((k // 128, bfq.align4(m)), dtype=torch.float32, device=dev)
            out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
            ws = bfq.gemm_workspace(m, n, k, dev)
            shapes.append(dict(m=m, n=n, k=k, x=x, q=q, s=s, wq=wq, sw=sw, wq0=wq0, sw0=sw0,
                               out=out, ws=ws))
    torch.cuda.synchronize()
    return shapes


def profile_ue8m0_shape(bfq, torch, dev, shape, calls):
    """One (m, n, k) with UE8M0 scales on both operands (packed activation
    scales, power-of-two weight scales), `calls` eager rounds of quant +
    bfq_gemm_block_fp8_ue8m0, for profiler captures."""
    import bfq_synth as synth

    m, n, k = shape
    w = synth.weight(n, k, seed=n + k, device=dev)
    wq, sw = bfq.weight_block_quant(w, bfq.SCALE_F32_POW2)
    del w
    x = synth.activation(m, k, seed=m * 31 + n, device=dev)
    q = torch.empty((m, k), dtype=torch.float8_e4m3fn, device=dev)
    s = torch.empty((bfq.scale_cols(k, bfq.SCALE_UE8M0_PACKED), bfq.align4(m)), dtype=torch.int32,
                    device=dev)
    out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    for _ in range(calls):
        bfq.bfq_quant(x, q, s, bfq.SCALE_UE8M0_PACKED, s.shape[-1])
        bfq.bfq_gemm_block_fp8_ue8m0(q, s, bfq.SCALE_UE8M0_PACKED, s.shape[-1], wq, sw, out)
    torch.cuda.synchronize()
    if bfq.bfq_poll_device_status() != 0:
        raise RuntimeError("device status set")


def step(bfq, shapes, events=None):
    for i, sh in enumerate(shapes):
        if events is not None:
            events[i][0].record()
        bfq.bfq_quant(sh["x"], sh["q"], sh["s"], bfq.SCALE_F32, sh["s"].shape[-1])
        if events is not None:
            events[i][1].record()
        bfq.bfq_gemm_block_fp8(sh["q"], sh["s"], bfq.SCALE_F32, sh["s"].shape[-1], sh["wq"],
                               sh["sw"], sh["out"], sh["ws"])
        if events is not None:
            events[i][2].record()


class E2EPipeline:
    """End-to-end step through the public API with host buffers: the shapes
    of one (n, k) weight share one pinned host input buffer, one device input
    buffer, one device output buffer and one pinned host output buffer, so
    every step copies each group's activations host->device in one copy,
    quantizes and multiplies every shape of the group, and copies the
    group's results device->host in one copy.  Three streams overlap the
    transfers of one group with the compute of its neighbours; CUDA events
    order each group's copy-in -> compute -> copy-out and keep device buffers
    from being reused before the copy that reads them has finished."""

    def __init__(self, torch, shapes):
        self.torch = torch
        self.groups = []
        i = 0
        while i < len(shapes):
            j = i
            while j < len(shapes) and (shapes[j]["n"], shapes[j]["k"]) == (shapes[i]["n"],
                                                                           shapes[i]["k"]):
                j += 1
            grp = shapes[i:j]
            n_in = sum(s["x"].numel() for s in grp)
            n_out = sum(s["out"].numel() for s in grp)
            dev = grp[0]["x"].device
            g = dict(shapes=grp,
                     d_in=torch.empty(n_in, dtype=torch.bfloat16, device=dev),
                     d_out=torch.empty(n_out, dtype=torch.bfloat16, device=dev),
                     h_in=torch.empty(n_in, dtype=torch.bfloat16).pin_memory(),
                     h_out=torch.empty(n_out, dtype=torch.bfloat16).pin_memory(),
                     xs=[], outs=[])
            a = b = 0
            for s in grp:
                n1, n2 = s["x"].numel(), s["out"].numel()
                g["h_in"][a:a + n1].copy_(s["x"].reshape(-1).cpu())
                g["xs"].append(g["d_in"][a:a + n1].view(s["x"].shape))
                g["outs"].append(g["d_out"][b:b + n2].view(s["out"].shape))
                a, b = a + n1, b + n2
            self.groups.append(g)
            i = j
        self.h2d_bytes = sum(g["h_in"].numel() * 2 for g in self.groups)
        self.d2h_bytes = sum(g["h_out"].numel() * 2 for g in self.groups)
        self.s_in = torch.cuda.Stream()
        self.s_out = torch.cuda.Stream()
        n = len(self.groups)
        self.ev_in = [torch.cuda.Event() for _ in range(n)]
        self.ev_done = [torch.cuda.Event() for _ in range(n)]
        self.ev_out = [torch.cuda.Event() for _ in range(n)]
        self.first = True

    def step(self, bfq):
        torch = self.torch
        comp = torch.cuda.current_stream()
        for i, g in enumerate(self.groups):
            with torch.cuda.stream(self.s_in):
                if not self.first:  # the inputs are free once last step's group ran
                    self.s_in.wait_event(self.ev_done[i])
                g["d_in"].copy_(g["h_in"], non_blocking=True)
                self.ev_in[i].record()
            comp.wait_event(self.ev_in[i])
            if not self.first:  # the outputs are free once last step copied them
                comp.wait_event(self.ev_out[i])
            for sh, x, out in zip(g["shapes"], g["xs"], g["outs"]):
                bfq.bfq_quant(x, sh["q"], sh["s"], bfq.SCALE_F32, sh["s"].shape[-1])
                bfq.bfq_gemm_block_fp8(sh["q"], sh["s"], bfq.SCALE_F32, sh["s"].shape[-1],
                                       sh["wq"], sh["sw"], out, sh["ws"])
            self.ev_done[i].record(comp)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(self.ev_done[i])
                g["h_out"].copy_(g["d_out"], non_blocking=True)
                self.ev_out[i].record()
        self.first = False

    def join(self):
        comp = self.torch.cuda.current_stream()
        comp.wait_stream(self.s_in)
        comp.wait_stream(self.s_out)

    def link_rates(self, reps=3):
        """Copy-engine rates of the host link in GB/s, on the step's two
        largest output buffers: host->device alone (the second largest,
        copied in), device->host alone (the largest, copied out), and both
        at once (one copy on each copy stream).  The step's transfers take
        at least max(H2D bytes / h2d, D2H bytes / d2h)."""
        torch = self.torch
        by_out = sorted(self.groups, key=lambda g: g["h_out"].numel())
        g, g2 = by_out[-1], by_out[-2]
        comp = torch.cuda.current_stream()

        def timed(fn):
            fn()
            torch.cuda.synchronize()
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record()
            for _ in range(reps):
                fn()
            t1.record()
            torch.cuda.synchronize()
            return t0.elapsed_time(t1) / reps * 1e-3

        def h2d():
            g2["d_out"].copy_(g2["h_out"], non_blocking=True)

        def d2h():
            g["h_out"].copy_(g["d_out"], non_blocking=True)

        def both():  # the two largest output buffers, one in each direction
            self.s_in.wait_stream(comp)
            self.s_out.wait_stream(comp)
            with torch.cuda.stream(self.s_in):
                h2d()
            with torch.cuda.stream(self.s_out):
                d2h()
            comp.wait_stream(self.s_in)
            comp.wait_stream(self.s_out)

        b_in, b_out = g2["h_out"].numel() * 2, g["h_out"].numel() * 2
        return {"h2d_GBps": round(b_in / timed(h2d) / 1e9, 1),
                "d2h_GBps": round(b_out / timed(d2h) / 1e9, 1),
                "both_GBps": round((b_in + b_out) / timed(both) / 1e9, 1)}


def timed_launches(bfq, torch, shapes, reps):
    """Per-launch durations (ms) of quant and GEMM for every shape, measured
    with CUDA events on the launching stream.  Each repetition first enqueues
    a short device-side sleep so that the host has queued the whole step
    before the GPU reaches it: host launch latency cannot show up as kernel
    time.  The sleep lies outside every event pair."""
    qt = [[] for _ in shapes]
    gt = [[] for _ in shapes]
    for _ in range(reps):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in shapes]
        torch.cuda._sleep(20_000_000)
        step(bfq, shapes, ev)
        torch.cuda.synchronize()
        for j in range(len(shapes)):
            qt[j].append(ev[j][0].elapsed_time(ev[j][1]))
            gt[j].append(ev[j][1].elapsed_time(ev[j][2]))
    return qt, gt


def measure_calc_diff(bfq, torch, dev, shapes, threads):
    """Per shape, on sampled rows (first, last and two seeded rows): the pages'
    calc_diff ("vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.4: 1 - 2<x,y> /
    (|x|^2 + |y|^2), in fp64) between the GPU's bf16 output and the oracle's
    fp64 result, and the largest error normalised by |A_hat[m]| |W_hat[n]|
    (the 2e-3 gate of the parity tests).  The oracle quantizes the same
    seeded bf16 inputs itself; its weight quant and GEMM are shared out over
    `threads` host threads in 128-row weight blocks."""
    import concurrent.futures as cf

    import numpy as np

    import bfq_synth as synth
    import oracle

    oracle.build_oracle()
    oracle.e4m3_encode([0.0])  # build the oracle's tables before threads start
    res = []
    groups = {}
    for sh in shapes:
        groups.setdefault((sh["n"], sh["k"]), []).append(sh)
    with cf.ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
        for (n, k), grp in groups.items():
            w = synth.weight(n, k, seed=n + k, device=dev)
            wb = w.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
            del w
            blocks = list(range(0, n, 128))
            parts = list(ex.map(lambda r0: oracle.weight_block_quant(wb[r0:r0 + 128], False),
                                blocks))
            wq = np.concatenate([p_[0] for p_ in parts])
            sw = np.concatenate([p_[1] for p_ in parts])
            wn = np.concatenate(list(ex.map(
                lambda p_: np.linalg.norm(oracle.dequant_weight(p_[0], p_[1]), axis=1), parts)))
            for sh in grp:
                m = sh["m"]
                rng = np.random.default_rng(m * 7 + n + k)
                rows = np.unique(np.concatenate([[0, m - 1], rng.integers(0, m, 2)]))
                xb = sh["x"][torch.from_numpy(rows).to(dev)].cpu().contiguous()
                aq, sa = oracle.quant(xb.view(torch.int16).numpy().view(np.uint16),
                                      oracle.FMT_F32)
                ref = np.concatenate(list(ex.map(
                    lambda i: oracle.gemm(aq, sa, oracle.FMT_F32, parts[i][0], parts[i][1]),
                    range(len(parts)))), axis=1)
                got = sh["out"][torch.from_numpy(rows).to(dev)].float().cpu().numpy()
                an = np.linalg.norm(oracle.dequant_rows(aq, sa, oracle.FMT_F32), axis=1)
                x64, y64 = got.astype(np.float64), ref
                den = (x64 * x64 + y64 * y64).sum()
                cd = float(1.0 - 2.0 * (x64 * y64).sum() / den) if den > 0 else 0.0
                err = np.abs(x64 - y64) / (an[:, None] * wn[None, :])
                res.append({"m": m, "n": n, "k": k, "rows": len(rows), "calc_diff": cd,
                            "max_norm_err": float(err.max())})
            del wb, wq, sw, parts
    return res


def measure_pdl_ab(bfq, torch, shapes, replays):
    """Programmatic dependent launch on and off ("vLLM DeepGEMM FP8 Block GEMM
    基准测试" §4.2: the wrapper enables PDL).  (1) The decode chain of the
    smallest dense case, quant 8 x 7168 -> GEMM 8 x 4096 x 7168, back to back
    in one graph over nine weight copies (> 2x L2, so every GEMM reads its
    weights from HBM); (2) the whole sweep step as one graph.  Each graph is
    captured with the switch set, so it holds that launch mode."""
    c0 = next((sh for sh in shapes if (sh["m"], sh["n"], sh["k"]) == (8, 4096, 7168)), None)
    res = {}
    if c0 is not None:
        copies = 9
        wqs = [c0["wq"]] + [c0["wq"].clone() for _ in range(copies - 1)]
        sws = [c0["sw"]] + [c0["sw"].clone() for _ in range(copies - 1)]
        ld = c0["s"].shape[-1]

        def chain(i):
            bfq.bfq_quant(c0["x"], c0["q"], c0["s"], bfq.SCALE_F32, ld)
            bfq.bfq_gemm_block_fp8(c0["q"], c0["s"], bfq.SCALE_F32, ld, wqs[i], sws[i],
                                   c0["out"], c0["ws"])

        def gemm_only(i):
            bfq.bfq_gemm_block_fp8(c0["q"], c0["s"], bfq.SCALE_F32, ld, wqs[i], sws[i],
                                   c0["out"], c0["ws"])

        for name, fn in (("c0_quant_gemm_chain_us", chain), ("c0_gemm_us", gemm_only)):
            res[name] = {}
            for mode in (True, False):
                prev = bfq.bfq_set_programmatic_launch(mode)
                try:
                    t = graph_back_to_back_us(torch, fn, copies, 4 * copies)
                finally:
                    bfq.bfq_set_programmatic_launch(prev)
                res[name]["pdl" if mode else "no_pdl"] = round(t, 2)
        del wqs, sws
    res["step_ms"] = {}
    for mode in (True, False):
        prev = bfq.bfq_set_programmatic_launch(mode)
        try:
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                step(bfq, shapes)
                torch.cuda.synchronize()
                with torch.cuda.graph(g, stream=side):
                    step(bfq, shapes)
            torch.cuda.current_stream().wait_stream(side)
        finally:
            bfq.bfq_set_programmatic_launch(prev)
        g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(replays):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        res["step_ms"]["pdl" if mode else "no_pdl"] = round(e0.elapsed_time(e1) / replays, 4)
        del g
    return res


L2_BYTES = 129 << 20


def per_shape_b2b(bfq, torch, shapes, trials=5):
    """Per shape, device time per call of back-to-back launches captured in one
    CUDA graph (each launch overlapping the previous one's tail through
    programmatic dependent launch, as in a sequence of layers):
      gemm      cycling over the weight copies of the shape's (n, k) group,
                cloned further until they hold 2.5x the L2, so every launch
                reads its weights from HBM;
      gemm_warm one weight copy, which stays in L2 from call to call;
      quant     the shape's activation quant on its one input (L2-resident,
                as the previous layer's output would be).
    Returns {(m, n, k): (gemm_us, gemm_warm_us, quant_us)}."""
    groups = {}
    for sh in shapes:
        groups.setdefault((sh["n"], sh["k"]), []).append(sh)
    res = {}
    for (n, k), grp in groups.items():
        wqs = [sh["wq"] for sh in grp]
        sws = [sh["sw"] for sh in grp]
        need = -(-int(2.5 * L2_BYTES) // (n * k))
        while len(wqs) < need:
            wqs.append(grp[0]["wq"].clone())
            sws.append(grp[0]["sw"].clone())
        copies = len(wqs)
        for sh in grp:
            ld = sh["s"].shape[-1]

            def gemm(i, sh=sh, ld=ld):
                bfq.bfq_gemm_block_fp8(sh["q"], sh["s"], bfq.SCALE_F32, ld, wqs[i], sws[i],
                                       sh["out"], sh["ws"])

            def quant(i, sh=sh, ld=ld):
                bfq.bfq_quant(sh["x"], sh["q"], sh["s"], bfq.SCALE_F32, ld)

            t = graph_back_to_back_us(torch, gemm, copies, max(2 * copies, 12), trials)
            tw = graph_back_to_back_us(torch, lambda i, g=gemm: g(0), 1, 12, trials)
            tq = graph_back_to_back_us(torch, quant, 1, 12, trials)
            res[(sh["m"], n, k)] = (t, tw, tq)
        del wqs, sws
    torch.cuda.synchronize()
    return res


QUANT_M = [8, 128, 4096, 16384]
QUANT_K = [7168, 18432]
MOE_E, MOE_T, MOE_I, MOE_H = 32, 256, 2048, 7168


def gated_times(torch, fn, reps):
    """Per-launch device time (us) of fn(), with the host ahead of the GPU."""
    ts = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(2_000_000)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    ts.sort()
    return ts[len(ts) // 2]


def measure_ue8m0_arms(bfq, torch, dev, fp8_peak, ms=(1024, 4096)):
    """Dense GEMM with UE8M0 scales on both operands (packed activation
    scales, power-of-two 128x128 weight scales; the sweep's (n, k) shapes):
    the block-scaled arm (bfq_gemm_block_fp8_ue8m0, scales applied by the
    MMA) against the promotion kernel (bfq_gemm_block_fp8) on the same
    inputs, back to back in one CUDA graph over weight copies holding 2.5x
    the L2.  The two results agree to within summation order."""
    import bfq_synth as synth

    rows = []
    for n, k in SWEEP_NK:
        w = synth.weight(n, k, seed=n + k + 5, device=dev)
        wq, sw = bfq.weight_block_quant(w, bfq.SCALE_F32_POW2)
        del w
        copies = max(2, -(-int(2.5 * L2_BYTES) // (n * k)))
        wqs = [wq] + [wq.clone() for _ in range(copies - 1)]
        sws = [sw] + [sw.clone() for _ in range(copies - 1)]
        for m in ms:
            x = synth.activation(m, k, seed=m + n + 5, device=dev)
            q, s = bfq.quant(x, bfq.SCALE_UE8M0_PACKED)
            o_bs = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
            o_pr = torch.empty_like(o_bs)
            t_bs = graph_back_to_back_us(
                torch, lambda i: bfq.bfq_gemm_block_fp8_ue8m0(q, s, 2, s.shape[-1], wqs[i], sws[i],
                                                              o_bs), copies, max(4 * copies, 16))
            t_pr = graph_back_to_back_us(
                torch, lambda i: bfq.bfq_gemm_block_fp8(q, s, 2, s.shape[-1], wqs[i], sws[i], o_pr,
                                                        None), copies, max(4 * copies, 16))
            torch.cuda.synchronize()
            diff = (o_bs.float() - o_pr.float()).abs().max().item()
            scale = o_pr.float().abs().max().item()
            fl = 2.0 * m * n * k
            rows.append({"m": m, "n": n, "k": k, "block_scaled_us": round(t_bs, 2),
                         "promotion_us": round(t_pr, 2), "speedup": round(t_pr / t_bs, 3),
                         "block_scaled_tflops": round(fl / t_bs / 1e6, 1),
                         "block_scaled_frac_fp8": round(fl / t_bs / 1e6 / fp8_peak, 3),
                         "promotion_tflops": round(fl / t_pr / 1e6, 1),
                         "max_abs_diff_rel": float(f"{diff / max(scale, 1e-30):.2e}")})
            del q, s, o_bs, o_pr, x
        del wqs, sws, wq, sw
        torch.cuda.empty_cache()
    return {"timing": "back to back in one CUDA graph over weight copies holding 2.5x the L2",
            "plan": "bfq_gemm_block_fp8_ue8m0 runs the promotion plan for M <= 128, K < 1024 or "
                    "fewer tiles than half the SMs",
            "shapes": rows}


def graph_back_to_back_us(torch, fn, copies, calls, trials=5):
    """Per-call device time (us) of fn(i) issued back to back, i cycling over
    `copies` operand sets, as one CUDA graph (no host launch gaps; each launch
    overlaps the previous one's tail through programmatic dependent launch,
    as in a real sequence of calls).  Median over `trials` replays."""
    for i in range(copies):
        fn(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for c in range(calls):
                fn(c % copies)
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(trials):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3 / calls)
    del g
    return statistics.median(ts)


def measure_quant_sweep(bfq, torch, dev, hbm_peak, reps):
    """Standalone per-token-group quant over m x k, fp32 and packed UE8M0 scales.
    `us` is one isolated launch (gated, median of `reps`); `us_b2b` the per-call
    time of back-to-back calls over rotating inputs that together exceed L2
    twice (the pages' benchmark loop repeats a kernel the same way)."""
    import bfq_synth as synth

    rows = []
    for k in QUANT_K:
        for m in QUANT_M:
            copies = max(1, min(8, -(-(300 << 20) // (2 * m * k))))
            xs = [synth.activation(m, k, seed=m + k + c, zero_group=True, device=dev)
                  for c in range(copies)]
            x = xs[0]
            for fmt, name in ((bfq.SCALE_F32, "f32"), (bfq.SCALE_UE8M0_PACKED, "ue8m0_packed")):
                ld = bfq.align4(m)
                q = torch.empty((m, k), dtype=torch.float8_e4m3fn, device=dev)
                sc = torch.empty((bfq.scale_cols(k, fmt), ld), dtype=bfq.scale_dtype(fmt),
                                 device=dev)
                us = gated_times(torch, lambda: bfq.bfq_quant(x, q, sc, fmt, ld), reps)
                us_b2b = graph_back_to_back_us(
                    torch, lambda i: bfq.bfq_quant(xs[i], q, sc, fmt, ld), copies,
                    max(2 * copies, 12))
                nbytes = 3 * m * k + sc.numel() * 4
                gbs = nbytes / (us * 1e-6) / 1e9
                gbs_b2b = nbytes / (us_b2b * 1e-6) / 1e9
                rows.append({"m": m, "k": k, "scales": name, "us": round(us, 2),
                             "gbps": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 3),
                             "us_b2b": round(us_b2b, 2), "gbps_b2b": round(gbs_b2b, 1),
                             "hbm_frac_b2b": round(gbs_b2b / hbm_peak, 3), "bytes": nbytes})
            del xs, x
    return rows


FUSED_SHAPES = [(128, 7168, 18432), (4096, 7168, 18432), (128, 18432, 7168), (4096, 18432, 7168)]


def measure_fused_quant(bfq, torch, dev, hbm_peak):
    """GEMM whose output feeds the next block-FP8 GEMM: the plain GEMM then the
    1 x 128 quant of its bf16 output (two kernels, the output written and read
    back) against the GEMM with the quant fused into its epilogue (with and
    without also writing the bf16 output).  Back-to-back calls over rotating
    weight copies, fp32 scales in and out."""
    import bfq_synth as synth

    rows = []
    for m, n, k in FUSED_SHAPES:
        copies = max(1, min(4, -(-(300 << 20) // (n * k))))
        w = synth.weight(n, k, seed=n + k, device=dev)
        wq0, sw0 = bfq.weight_block_quant(w, bfq.SCALE_F32)
        del w
        wqs = [wq0] + [wq0.clone() for _ in range(copies - 1)]
        sws = [sw0] + [sw0.clone() for _ in range(copies - 1)]
        x = synth.activation(m, k, seed=m * 31 + n, device=dev)
        q, s = bfq.quant(x, bfq.SCALE_F32)
        del x
        ld = bfq.align4(m)
        out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        oq = torch.empty((m, n), dtype=torch.float8_e4m3fn, device=dev)
        osc = torch.empty((n // 128, ld), dtype=torch.float32, device=dev)
        ws = bfq.gemm_workspace(m, n, k, dev)

        def unfused(i):
            bfq.bfq_gemm_block_fp8(q, s, 0, s.shape[-1], wqs[i], sws[i], out, ws)
            bfq.bfq_quant(out, oq, osc, 0, ld)

        def fused(i):
            bfq.bfq_gemm_block_fp8_quant(q, s, 0, s.shape[-1], wqs[i], sws[i], out, 0, oq, osc, ld,
                                         workspace=ws)

        def fused_no_out(i):
            bfq.bfq_gemm_block_fp8_quant(q, s, 0, s.shape[-1], wqs[i], sws[i], None, 0, oq, osc,
                                         ld, workspace=ws)

        calls = max(2 * copies, 8)
        t_u = graph_back_to_back_us(torch, unfused, copies, calls)
        t_f = graph_back_to_back_us(torch, fused, copies, calls)
        t_fn = graph_back_to_back_us(torch, fused_no_out, copies, calls)
        rows.append({"m": m, "n": n, "k": k, "unfused_us": round(t_u, 2),
                     "fused_us": round(t_f, 2), "fused_no_bf16_out_us": round(t_fn, 2),
                     "saved_frac": round(1.0 - t_f / t_u, 3)})
        del wqs, sws, q, s, out, oq, osc
        torch.cuda.empty_cache()
    return rows


def measure_moe(bfq, torch, dev, hbm_peak, fp8_peak, reps):
    """Masked MoE expert slice: up GEMM -> silu-mul-quant -> down GEMM, E=32,
    T_max=256, valid counts ~ U{0..256}, UE8M0 packed activation scales,
    power-of-two 128x128 weight scales."""
    import bfq_synth as synth

    E, T, I, H = MOE_E, MOE_T, MOE_I, MOE_H
    counts = synth.valid_counts(E, T)
    tot = int(counts.sum())
    d_counts = counts.to(dev)
    w_up = torch.empty((E, 2 * I, H), dtype=torch.float8_e4m3fn, device=dev)
    s_up = torch.empty((E, 2 * I // 128, H // 128), dtype=torch.float32, device=dev)
    w_dn = torch.empty((E, H, I), dtype=torch.float8_e4m3fn, device=dev)
    s_dn = torch.empty((E, H // 128, I // 128), dtype=torch.float32, device=dev)
    for e in range(E):  # one expert at a time keeps the bf16 staging small
        wq, sw = bfq.weight_block_quant(synth.weight(2 * I, H, seed=700 + e, device=dev),
                                        bfq.SCALE_F32_POW2)
        w_up[e].copy_(wq)
        s_up[e].copy_(sw)
        wq, sw = bfq.weight_block_quant(synth.weight(H, I, seed=800 + e, device=dev),
                                        bfq.SCALE_F32_POW2)
        w_dn[e].copy_(wq)
        s_dn[e].copy_(sw)
    x = synth.masked_activation(E, T, H, counts, seed=900, device=dev)
    a_up = torch.empty((E, T, H), dtype=torch.float8_e4m3fn, device=dev)
    sa_up = torch.empty((E, bfq.scale_cols(H, 2), T), dtype=torch.int32, device=dev)
    for e in range(E):
        c = int(counts[e])
        if c:
            bfq.bfq_quant(x[e, :c], a_up[e, :c], sa_up[e], bfq.SCALE_UE8M0_PACKED, T)
    h = torch.empty((E, T, 2 * I), dtype=torch.bfloat16, device=dev)
    a_dn = torch.empty((E, T, I), dtype=torch.float8_e4m3fn, device=dev)
    sa_dn = torch.empty((E, bfq.scale_cols(I, 2), T), dtype=torch.int32, device=dev)
    out = torch.empty((E, T, H), dtype=torch.bfloat16, device=dev)

    # UE8M0 scales on both operands: the GEMMs run on the block-scaled arm
    # (scales applied by the MMA), measured faster here than promotion,
    # which is timed beside it
    def up():
        bfq.bfq_gemm_block_fp8_masked_ue8m0(a_up, sa_up, 2, T, w_up, s_up, d_counts, h)

    def act():
        bfq.bfq_silu_mul_quant(h, d_counts, a_dn, sa_dn, 2, T)

    def down():
        bfq.bfq_gemm_block_fp8_masked_ue8m0(a_dn, sa_dn, 2, T, w_dn, s_dn, d_counts, out)

    def up_promotion():
        bfq.bfq_gemm_block_fp8_masked(a_up, sa_up, 2, T, w_up, s_up, d_counts, h)

    def down_promotion():
        bfq.bfq_gemm_block_fp8_masked(a_dn, sa_dn, 2, T, w_dn, s_dn, d_counts, out)

    for fn in (up_promotion, act, down_promotion, up, act, down):
        fn()
    torch.cuda.synchronize()
    active = int((counts > 0).sum())
    res = {"experts": E, "t_max": T, "valid_rows": tot, "active_experts": active}
    for name, fn, fn_pr, n, k in (("up_gemm", up, up_promotion, 2 * I, H),
                                  ("down_gemm", down, down_promotion, H, I)):
        us = gated_times(torch, fn, reps)
        us_b2b = graph_back_to_back_us(torch, lambda i, fn=fn: fn(), 1, 8)
        us_pr = gated_times(torch, fn_pr, reps)
        us_pr_b2b = graph_back_to_back_us(torch, lambda i, fn=fn_pr: fn(), 1, 8)
        flops = 2.0 * tot * n * k
        nbytes = active * n * k + tot * k + 2 * tot * n + active * (n // 128) * (k // 128) * 4 \
            + tot * (k // 512) * 4
        t_roof = max(flops / (fp8_peak * 1e12), nbytes / (hbm_peak * 1e9))
        res[name] = {"n": n, "k": k, "arm": "block_scaled", "us": round(us, 2),
                     "us_b2b": round(us_b2b, 2), "tflops": round(flops / us / 1e6, 1),
                     "gbps": round(nbytes / (us * 1e-6) / 1e9, 1),
                     "roofline_frac": round(t_roof * 1e6 / us, 3),
                     "roofline_frac_b2b": round(t_roof * 1e6 / us_b2b, 3),
                     "bound": "tensor" if flops / (fp8_peak * 1e12) > nbytes / (hbm_peak * 1e9)
                     else "hbm",
                     "promotion_us": round(us_pr, 2), "promotion_us_b2b": round(us_pr_b2b, 2)}
    us = gated_times(torch, act, reps)
    nbytes = tot * (2 * I * 2 + I) + tot * (I // 512) * 4
    gbs = nbytes / (us * 1e-6) / 1e9
    # back to back over rotating inputs (4 x 64 MB, more than twice the L2)
    hs = [h] + [synth.masked_activation(E, T, 2 * I, counts, seed=950 + c, device=dev)
                for c in range(3)]
    us_b2b = graph_back_to_back_us(
        torch, lambda i: bfq.bfq_silu_mul_quant(hs[i], d_counts, a_dn, sa_dn, 2, T), len(hs), 16)
    gbs_b2b = nbytes / (us_b2b * 1e-6) / 1e9
    res["silu_mul_quant"] = {"us": round(us, 2), "gbps": round(gbs, 1),
                             "hbm_frac": round(gbs / hbm_peak, 3), "us_b2b": round(us_b2b, 2),
                             "gbps_b2b": round(gbs_b2b, 1),
                             "hbm_frac_b2b": round(gbs_b2b / hbm_peak, 3), "bytes": nbytes}
    del hs
    # the slice with the up projection's silu-and-mul + quant fused into its
    # epilogue (weights interleaved once, as offline weight preparation)
    w_up_i, s_up_i = bfq.interleave_gate_up(w_up, s_up)

    def up_act_fused():
        bfq.bfq_gemm_block_fp8_masked_silu_quant_ue8m0(a_up, sa_up, 2, T, w_up_i, s_up_i,
                                                       d_counts, 2, a_dn, sa_dn, T)

    def up_act_fused_promotion():
        bfq.bfq_gemm_block_fp8_masked_silu_quant(a_up, sa_up, 2, T, w_up_i, s_up_i, d_counts, 2,
                                                 a_dn, sa_dn, T)

    up_act_fused_promotion()
    up_act_fused()
    torch.cuda.synchronize()
    us_fused = gated_times(torch, up_act_fused, reps)
    us_fused_pr = gated_times(torch, up_act_fused_promotion, reps)
    us_seq = {}
    for name, fns in (("unfused", (up, act, down)), ("fused", (up_act_fused, down)),
                      ("unfused_promotion", (up_promotion, act, down_promotion)),
                      ("fused_promotion", (up_act_fused_promotion, down_promotion))):
        def chain(i, fns=fns):
            for fn in fns:
                fn()
        us_seq[name] = graph_back_to_back_us(torch, chain, 1, 6)
    res["up_silu_quant_fused"] = {"arm": "block_scaled", "us": round(us_fused, 2),
                                  "promotion_us": round(us_fused_pr, 2),
                                  "unfused_up_plus_silu_us": round(res["up_gemm"]["us"] +
                                                                   res["silu_mul_quant"]["us"], 2)}
    res["slice_us_b2b"] = {k: round(v, 2) for k, v in us_seq.items()}
    del w_up_i, s_up_i
    del w_up, w_dn, x, h
    return res


def run_gpu(args, rank, world, local_rank):
    import torch

    import block_scaled_fp8_quant_gb300 as bfq

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    bfq.load_library()
    peaks, peak_src = load_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    fp8_peak = float(peaks["bf16_tflops"]) * FP8_PER_BF16
    fp8_peak_sustained = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])) * FP8_PER_BF16

    if args.moe_only:  # profiling mode: the MoE expert slice only, no report
        measure_moe(bfq, torch, dev, hbm_peak, fp8_peak, 2)
        return 0
    if args.shape and args.ue8m0:  # profiling mode: one shape on the block-scaled arm
        profile_ue8m0_shape(bfq, torch, dev, args.shape, args.warmup + args.steps)
        return 0
    shapes = build_problem(bfq, torch, dev, args.shape)
    n_shapes = len(shapes)
    flops_step = sum(2 * s["m"] * s["n"] * s["k"] for s in shapes)

    dist = None
    if world > 1:
        import torch.distributed as dist

    for _ in range(args.warmup):
        step(bfq, shapes)
    torch.cuda.synchronize()
    if args.shape:  # profiling mode: a few eager steps of one shape, no report
        for _ in range(args.steps):
            step(bfq, shapes)
        torch.cuda.synchronize()
        return 0

    # the whole step (all launches) as one CUDA graph, replayed K times
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(bfq, shapes)  # warm the capture stream
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            step(bfq, shapes)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else
                      int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local_rank])) as clk:
        start.record()
        for _ in range(args.steps):
            graph.replay()
        stop.record()
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    total_ms = max_over_ranks(start.elapsed_time(stop), dist, dev)

    reps = max(3, min(args.steps, 20))
    qts, gts = timed_launches(bfq, torch, shapes, reps)
    parity = measure_calc_diff(bfq, torch, dev, shapes, host_cores()) if rank == 0 else []
    b2b = per_shape_b2b(bfq, torch, shapes)
    status = bfq.bfq_poll_device_status()
    if status != 0:
        raise RuntimeError(f"device watchdog reported status {status}")

    per_shape = []
    gemm_us_total = quant_us_total = 0.0
    for j, sh in enumerate(shapes):
        qt, gt = qts[j], gts[j]
        m, n, k = sh["m"], sh["n"], sh["k"]
        g_us, gw_us, q_us = b2b[(m, n, k)]
        gemm_us_total += g_us
        quant_us_total += q_us
        t_flop = 2.0 * m * n * k / (fp8_peak * 1e12)
        t_byte = gemm_alg_bytes(m, n, k) / (hbm_peak * 1e9)
        per_shape.append({
            "m": m, "n": n, "k": k, "gemm_us": round(g_us, 2),
            "tflops": round(pages_tflops(m, n, k, g_us), 1),
            "gbps_pages": round(pages_gbps(m, n, k, g_us), 1),
            "roofline_frac": round(max(t_flop, t_byte) * 1e6 / g_us, 3),
            "bound": "tensor" if t_flop >= t_byte else "hbm",
            "gemm_us_l2warm": round(gw_us, 2),
            "gemm_us_isolated": round(statistics.median(gt) * 1e3, 2),
            "quant_us": round(q_us, 2),
            "quant_gbps": round(quant_alg_bytes(m, k) / (q_us * 1e-6) / 1e9, 1),
            "quant_us_isolated": round(statistics.median(qt) * 1e3, 2),
        })
        pr = next((r for r in parity if (r["m"], r["n"], r["k"]) == (m, n, k)), None)
        if pr:
            per_shape[-1]["calc_diff"] = float(f"{pr['calc_diff']:.3e}")
            per_shape[-1]["max_norm_err"] = float(f"{pr['max_norm_err']:.3e}")
    gemm_launch_ms = gemm_us_total / n_shapes * 1e-3
    achieved_tflops = flops_step / (gemm_us_total * 1e-6) / 1e12
    gemm_bytes_avg = sum(gemm_alg_bytes(s["m"], s["n"], s["k"]) for s in shapes) / n_shapes
    t_roof_sum = sum(max(2.0 * s["m"] * s["n"] * s["k"] / (fp8_peak * 1e12),
                         gemm_alg_bytes(s["m"], s["n"], s["k"]) / (hbm_peak * 1e9)) for s in shapes)

    # end to end through the public API with host buffers (pinned)
    pipe = E2EPipeline(torch, shapes)
    h2d, d2h = pipe.h2d_bytes, pipe.d2h_bytes
    for _ in range(max(1, args.warmup)):
        pipe.step(bfq)
    pipe.join()
    torch.cuda.synchronize()
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record()
    for _ in range(args.steps):
        pipe.step(bfq)
    pipe.join()
    e_stop.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e_start.elapsed_time(e_stop), dist, dev)
    link = pipe.link_rates()
    link["transfer_bound_ms_per_step"] = round(1e3 * max(
        h2d / (link["h2d_GBps"] * 1e9), d2h / (link["d2h_GBps"] * 1e9)), 3)

    if rank != 0:
        return 0
    ms_per_step = total_ms / args.steps
    traffic = profile_traffic()
    line = {
        "metric": METRIC,
        "value": world * flops_step / (ms_per_step * 1e-3) / 1e12,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8_e4m3",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "shapes": n_shapes, "act_scales": "fp32 col-major",
                   "weight_scales": "fp32 128x128", "parallelism": f"replicas x{world}",
                   "timed": "CUDA graph of the whole step (quant + GEMM per shape), replayed",
                   "l2": "inputs larger than L2: every shape reads its own weight copy "
                         "(~2.8 GB of distinct weights per step, > 20x the 129 MB L2), so no "
                         "GEMM launch finds its weights in L2; per-shape gemm_us_l2warm "
                         "repeats one weight copy"},
        "e2e": {"value": world * flops_step * args.steps / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / args.steps,
                "how": "public C-ABI calls per shape; pinned host buffers, one H2D and one "
                       "D2H per (n,k) group of shapes; H2D, compute and D2H on three streams "
                       "ordered by events (transfers of one group overlap its neighbours' "
                       "compute)",
                "host_link": link},
        "gpu_launches": 2 * n_shapes * args.steps,
        "roofline": {"bound": "tensor", "achieved": round(achieved_tflops, 1),
                     "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": round(achieved_tflops / fp8_peak, 4),
                     "traffic": traffic,
                     "kernel": "block-FP8 GEMM: gemm_block_fp8_kernel and gemm_block_fp8_persistent (all 36 sweep launches)",
                     "peak_source": f"{peak_src} bf16 burst x {FP8_PER_BF16} (fp8:bf16 nominal)",
                     "alg_bytes_per_launch_avg": gemm_bytes_avg,
                     "avg_launch_us": round(gemm_launch_ms * 1e3, 2),
                     "launch_timing": "per shape, back-to-back launches in one CUDA graph over "
                                      "weight copies holding 2.5x the L2 (cold weights), CUDA "
                                      "events on the launching stream",
                     "mixed_frac": round(t_roof_sum * 1e6 / gemm_us_total, 4),
                     "peak_sustained": fp8_peak_sustained,
                     "frac_of_sustained": round(achieved_tflops / fp8_peak_sustained, 4)},
        "quant": {"total_us_per_step": round(quant_us_total, 1), "hbm_peak_gbs": hbm_peak,
                  "timing": "per shape, back-to-back calls on its input in one CUDA graph"},
        "clocks": clk.summary(),
        "shapes": per_shape,
    }
    if parity:
        line["parity"] = {
            "vs": "CPU oracle (fp64 block GEMM of its own quantization of the same inputs)",
            "rows_per_shape": "first, last and two seeded rows, every column",
            "calc_diff_max": float(f"{max(r['calc_diff'] for r in parity):.3e}"),
            "max_norm_err": float(f"{max(r['max_norm_err'] for r in parity):.3e}"),
            "gate": 2e-3}
    if not args.skip_extra:
        line["pdl_ab"] = measure_pdl_ab(bfq, torch, shapes, 10)
        del shapes, pipe
        torch.cuda.empty_cache()
        line["quant_sweep"] = measure_quant_sweep(bfq, torch, dev, hbm_peak, 10)
        line["moe_slice"] = measure_moe(bfq, torch, dev, hbm_peak, fp8_peak, 10)
        line["ue8m0_arms"] = measure_ue8m0_arms(bfq, torch, dev, fp8_peak)
        line["fused_output_quant"] = measure_fused_quant(bfq, torch, dev, hbm_peak)
        if bfq.bfq_poll_device_status() != 0:
            raise RuntimeError("device watchdog fired during the extra measurements")
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--shape", type=lambda v: tuple(int(t) for t in v.split(",")), default=None,
                    help="m,n,k of one sweep shape: run only it, eagerly, and print nothing "
                         "(for profiler captures)")
    ap.add_argument("--ue8m0", action="store_true",
                    help="with --shape: UE8M0 scales on both operands, block-scaled GEMM arm")
    ap.add_argument("--impl", choices=["bfq", "reference"], default="bfq")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--moe-only", action="store_true",
                    help="run only the masked MoE expert slice and print nothing (profiling)")
    ap.add_argument("--skip-extra", action="store_true",
                    help="skip the standalone-quant sweep and the MoE slice measurements")
    args = ap.parse_args(argv)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        return run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
