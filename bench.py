#!/usr/bin/env python
"""Benchmark of the block-scaled backward GEMMs on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl native|reference]

One step = the backward of one layer on one batch of seeded synthetic input, entirely
in libbsq's kernels: for the default workload (MXFP4 4096 x 4096 x 4096, W and X packed
E2M1 with E8M0 per-32 scales) that is bsq_linear_dgrad + bsq_linear_wgrad.  L2 is
flushed (a 256 MiB device memset, outside the timed events) before every timed step.
Prints one JSON line.  ``value`` is TFLOP/s of the timed steps with inputs resident in
HBM; ``e2e`` is the same metric through the same C ABI calls with the step's inputs
copied from pinned host memory and both gradients copied back inside the timed region.
The small-M (M = 16) dgrad of the same weight is reported as GB/s of algorithmic bytes.

With --impl reference the CPU oracle is timed on a bounded sample of the same workload
(the only other place the oracle runs besides the tests and the cpu_baseline leg).
Multi-GPU (torchrun): every rank runs an independent replica (the path has no exchange
step); value = all ranks' FLOPs / the slowest rank's time.
"""

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FMT_BYTES = {0: 2.0, 1: 1.0, 2: 0.5, 3: 0.5}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only the headline workload (not the other four, nor the standalone dequant)")
    ap.add_argument("--profile", default=None,
                    choices=["backward", "dgrad", "wgrad", "grouped_dgrad", "grouped_wgrad", "small_m", "dequant",
                             "forward", "forward_bf16", "e5m2"],
                    help="run only this op of the workload, --warmup + --steps times back to back, and print "
                         "its mean time (a fixed launch sequence for ncu; not a benchmark line)")
    ap.add_argument("--experts", type=int, default=None,
                    help="grouped workloads: scale down to this many experts (same tokens per expert)")
    ap.add_argument("--rows", type=int, default=None,
                    help="workload 4 with --profile: route this many grad_out rows (a decode-sized batch) "
                         "over the same 64 expert weights")
    return ap.parse_args()


def profile_run(args, bsq, synth, dev):
    """--profile: one op of the workload, back to back (no L2 flush in between)."""
    c = synth.make_config(args.config, device=dev, seed=0, experts=args.experts,
                          rows=args.rows if args.config == 4 else None)
    if c["grouped"]:
        c["offsets_dev"] = torch.from_numpy(c["offsets"]).to(dev)
    outs = alloc_outputs(c, dev)
    op = args.profile
    if op == "backward":
        f = lambda: bsq.linear_backward(c["G"], c["W"], c["X"], grad_x=outs["dgrad"], grad_w=outs["wgrad"])
    elif op == "dgrad":
        f = lambda: bsq.linear_dgrad(c["G"], c["W"], out=outs["dgrad"])
    elif op == "wgrad":
        f = lambda: bsq.linear_wgrad(c["G"], c["X"], out=outs["wgrad"])
    elif op == "grouped_dgrad":
        f = lambda: bsq.grouped_dgrad(c["G"], c["W"], c["offsets_dev"], out=outs["grouped_dgrad"])
    elif op == "grouped_wgrad":
        f = lambda: bsq.grouped_wgrad(c["G"], c["X"], c["offsets_dev"], c["E"], out=outs["grouped_wgrad"])
    elif op in ("forward", "forward_bf16"):
        yo = torch.empty((c["M"], c["N"]), dtype=torch.bfloat16, device=dev)
        xf = c["X"] if op == "forward" else synth.make_packed(synth.FMT_BF16, 1, c["M"], c["K"], 1.0, 77, dev)
        f = lambda: bsq.linear_forward(xf, c["W"], out=yo)
    elif op == "e5m2":
        qc = torch.empty(c["G"].shape, dtype=torch.uint8, device=dev)
        qd = torch.empty(c["G"].shape, dtype=torch.bfloat16, device=dev)
        f = lambda: bsq.quantize_e5m2(c["G"], codes=qc, deq=qd)
    elif op == "small_m":
        if "G_small" not in c:
            c["G_small"] = synth.randn((16, c["N"]), 1e-2, 7, dev, torch.bfloat16)
        so = torch.empty((c["G_small"].shape[0], c["K"]), dtype=torch.bfloat16, device=dev)
        f = lambda: bsq.linear_dgrad(c["G_small"], c["W"], out=so)
    else:
        do = torch.empty((c["W"].batch, c["W"].rows, c["W"].cols), dtype=torch.bfloat16, device=dev)
        f = lambda: bsq.dequant(c["W"], out=do)
    for _ in range(args.warmup):
        f()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        f()
    b.record()
    torch.cuda.synchronize()
    st, code = bsq.get_device_error()
    if st != 0:
        raise SystemExit(f"device error {code}")
    print(json.dumps({"profile": op, "workload": c["name"], "launches": args.warmup + args.steps,
                      "mean_ms": a.elapsed_time(b) / max(1, args.steps)}))
    return 0


# ---------------------------------------------------------------- work accounting
def packed_bytes(p):
    """Bytes of a packed operand including its scales (what the method must read)."""
    n = p.batch * p.rows * p.cols
    b = n * FMT_BYTES[p.fmt]
    if p.fmt == 1:
        b += 4 * p.batch * -(-p.rows // 128) * -(-p.cols // 128)
    elif p.fmt == 2:
        b += n / 32
    elif p.fmt == 3:
        b += n / 16 + 4 * p.batch
    return b


def step_plan(c):
    """(name, flops, algorithmic bytes) of the step's dominant launch when the step is one
    fused backward launch (grad_out read once for both products), else None."""
    if c["grouped"] or c["W"].fmt != c["X"].fmt:
        return None
    M, N, K = c["M"], c["N"], c["K"]
    return ("backward", 4.0 * M * N * K,
            packed_bytes(c["W"]) + packed_bytes(c["X"]) + 2 * M * N + 2 * M * K + 2 * N * K)


def plan(c):
    """List of (name, flops, algorithmic_bytes) for the ops of one step of config c."""
    M, N, K = c["M"], c["N"], c["K"]
    ops = []
    if not c["grouped"]:
        ops.append(("dgrad", 2.0 * M * N * K, packed_bytes(c["W"]) + 2 * M * N + 2 * M * K))
        ops.append(("wgrad", 2.0 * M * N * K, packed_bytes(c["X"]) + 2 * M * N + 2 * N * K))
    else:
        S = int(c["offsets"][-1])
        ops.append(("grouped_dgrad", 2.0 * S * N * K, packed_bytes(c["W"]) + 2 * S * N + 2 * S * K))
        if c["X"] is not None:
            ops.append(("grouped_wgrad", 2.0 * S * N * K, packed_bytes(c["X"]) + 2 * S * N + 2 * c["E"] * N * K))
    return ops


# ---------------------------------------------------------------- peaks and clocks
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))

        def find(keys):
            for k in keys:
                if k in d and isinstance(d[k], (int, float)):
                    return float(d[k])
            return None
        hbm = find(["hbm_gbs", "hbm_GBps"])
        bf16 = find(["bf16_tflops", "bf16_TFLOPs"])
        sus = find(["bf16_tflops_sustained"])
        if hbm and bf16:
            return {"hbm_gbs": hbm, "bf16_tflops": bf16, "bf16_tflops_sustained": sus or bf16, "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def op_roofline(flops, nbytes, ms, pk):
    """Roofline of one launch: the binding resource at the measured peaks, what was achieved
    against it (burst peak: each launch is timed on its own) and the sustained-peak fraction."""
    t = ms * 1e-3
    if flops / (pk["bf16_tflops"] * 1e12) >= nbytes / (pk["hbm_gbs"] * 1e9):
        a = flops / t / 1e12
        return {"bound": "tensor", "achieved": a, "unit": "TFLOP/s", "frac": a / pk["bf16_tflops"],
                "frac_sustained": a / pk["bf16_tflops_sustained"]}
    a = nbytes / t / 1e9
    return {"bound": "hbm", "achieved": a, "unit": "GB/s", "frac": a / pk["hbm_gbs"],
            "tflops": flops / t / 1e12}


# The GEMM kernel's sources: a traffic figure captured from an earlier build is reported
# only while these are unchanged.
KERNEL_SOURCES = ["bsq_gemm.cu", "bsq_decode.cuh", "bsq_ptx.cuh", "bsq_pipe.cuh", "bsq_internal.h"]


def kernel_source_sha1():
    h = hashlib.sha1()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "block_scaled_gemm_fp8_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(workload, op):
    """DRAM bytes (read + write) per launch of the GEMM kernel for `op` on `workload`, from
    the committed ncu summary profiles/bsq_gemm_kernel_<workload>.md (its `traffic:` lines),
    or None when there is no such capture or the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"bsq_gemm_kernel_{workload}.md")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha1()
    for line in open(path):
        m = re.match(r"\s*traffic:\s*op=(\w+)\s+bytes=(\d+)\s+source_sha1=([0-9a-f]+)", line)
        if m and m.group(1) == op and m.group(3) == sha:
            return int(m.group(2))
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], 0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- native arm
def fused(c):
    """A linear workload whose W and X share a format runs as one bsq_linear_backward launch."""
    return not c["grouped"] and c["W"].fmt == c["X"].fmt


def run_ops(c, ops_out, bsq, stream=None):
    """Launch one step (the backward of the layer); returns the number of library kernels launched."""
    if not c["grouped"]:
        bsq.linear_backward(c["G"], c["W"], c["X"], grad_x=ops_out["dgrad"], grad_w=ops_out["wgrad"], stream=stream)
        return 1 if fused(c) else 2
    bsq.grouped_dgrad(c["G"], c["W"], c["offsets_dev"], out=ops_out["grouped_dgrad"], stream=stream)
    n = 1
    if c["X"] is not None:
        bsq.grouped_wgrad(c["G"], c["X"], c["offsets_dev"], c["E"], out=ops_out["grouped_wgrad"], stream=stream)
        n += 1
    return n


def alloc_outputs(c, dev):
    M, N, K = c["M"], c["N"], c["K"]
    if not c["grouped"]:
        return {"dgrad": torch.empty((M, K), dtype=torch.bfloat16, device=dev),
                "wgrad": torch.empty((N, K), dtype=torch.bfloat16, device=dev)}
    o = {"grouped_dgrad": torch.empty((M, K), dtype=torch.bfloat16, device=dev)}
    if c["X"] is not None:
        o["grouped_wgrad"] = torch.empty((c["E"], N, K), dtype=torch.bfloat16, device=dev)
    return o


# Cycles of a device-side spin queued after the L2 flush and before the first event of a
# timed region: it keeps the GPU busy while the host enqueues the event and the calls,
# so that host-side launch work never shows up inside the events.
HOST_COVER_CYCLES = 400000


def time_step(c, outs, bsq, steps, flush):
    """CUDA-event time (ms) of each of `steps` L2-flushed steps, each one run_ops call."""
    stream = torch.cuda.current_stream()
    ts, launches = [], 0
    for _ in range(steps):
        flush.zero_()
        torch.cuda._sleep(HOST_COVER_CYCLES)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        launches += run_ops(c, outs, bsq)
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return ts, launches


def time_ops(c, outs, bsq, steps, warmup, flush):
    """Per-op CUDA-event times (ms) over `steps` L2-flushed steps, each op through its own
    single-product entry point, and the step times: those of the fused backward launch
    where the workload has one, else the sum of the ops.  Returns (per_op, step_ms, launches
    inside the timed steps)."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        run_ops(c, outs, bsq)
    torch.cuda.synchronize()
    names = list(outs.keys())
    per_op = {n: [] for n in names}
    step_ms = []
    launches = 0
    if fused(c):
        step_ms, launches = time_step(c, outs, bsq, steps, flush)
    for _ in range(steps):
        flush.zero_()
        torch.cuda._sleep(HOST_COVER_CYCLES)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
        evs[0].record(stream)
        for i, n in enumerate(names):
            if not c["grouped"]:
                (bsq.linear_dgrad(c["G"], c["W"], out=outs[n]) if n == "dgrad"
                 else bsq.linear_wgrad(c["G"], c["X"], out=outs[n]))
            elif n == "grouped_dgrad":
                bsq.grouped_dgrad(c["G"], c["W"], c["offsets_dev"], out=outs[n])
            else:
                bsq.grouped_wgrad(c["G"], c["X"], c["offsets_dev"], c["E"], out=outs[n])
            if not fused(c):
                launches += 1
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        for i, n in enumerate(names):
            per_op[n].append(evs[i].elapsed_time(evs[i + 1]))
        if not fused(c):
            step_ms.append(evs[0].elapsed_time(evs[-1]))
    return per_op, step_ms, launches


def time_small_m(c, bsq, steps, warmup, flush):
    """M = 16 dgrad through the same weight: (median ms, algorithmic bytes)."""
    G = c["G_small"]
    out = torch.empty((G.shape[0], c["K"]), dtype=torch.bfloat16, device=G.device)
    for _ in range(warmup):
        bsq.linear_dgrad(G, c["W"], out=out)
    torch.cuda.synchronize()
    ts = []
    stream = torch.cuda.current_stream()
    for _ in range(steps):
        flush.zero_()
        torch.cuda._sleep(HOST_COVER_CYCLES)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        bsq.linear_dgrad(G, c["W"], out=out)
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    nbytes = packed_bytes(c["W"]) + 2 * G.numel() + 2 * G.shape[0] * c["K"]
    return statistics.median(ts), nbytes


def time_small_m_rotated(c, bsq, reps=5):
    """M = 16 dgrad with inputs rotated over copies of the weight (and of grad_out and the
    output) that together exceed twice the L2, launched back to back: per-launch ms (median
    over `reps` passes of total time / launches) and the number of copies.  No flush kernel
    runs in between: every launch finds its weight outside L2 and follows a launch of its
    own kind, as in a decode loop over layers.  A device-side spin covers the host's
    enqueue of the whole pass, so host time never shows up inside the events."""
    import dataclasses
    W, G = c["W"], c["G_small"]
    l2 = getattr(torch.cuda.get_device_properties(G.device), "L2_cache_size", 0) or (129 << 20)
    wb = W.data.numel() * W.data.element_size() + W.scale.numel() * W.scale.element_size()
    n = int(-(-2 * l2 // wb)) + 1
    ws = [dataclasses.replace(W, data=W.data.clone(), scale=W.scale.clone(),
                              tensor_scale=None if W.tensor_scale is None else W.tensor_scale.clone())
          for _ in range(n)]
    gs = [G.clone() for _ in range(n)]
    outs = [torch.empty((G.shape[0], c["K"]), dtype=torch.bfloat16, device=G.device) for _ in range(n)]
    launches = 2 * n
    for i in range(n):
        bsq.linear_dgrad(gs[i], ws[i], out=outs[i])
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ts = []
    for _ in range(reps):
        torch.cuda._sleep(HOST_COVER_CYCLES * launches)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(launches):
            bsq.linear_dgrad(gs[i % n], ws[i % n], out=outs[i % n])
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) / launches)
    del ws, gs, outs
    return statistics.median(ts), n


def small_m_entry(c, bsq, steps, warmup, flush, pk):
    """The M = 16 dgrad's bench entry: L2 flushed before each single timed launch, and under
    "rotated" the same kernel over rotated weight copies (no flush in between)."""
    ms, nbytes = time_small_m(c, bsq, steps, warmup, flush)
    rms, copies = time_small_m_rotated(c, bsq)
    gbs = lambda t: nbytes / (t * 1e-3) / 1e9
    return {"M": int(c["G_small"].shape[0]), "ms": ms, "GB/s": gbs(ms), "frac_hbm": gbs(ms) / pk["hbm_gbs"],
            "algorithmic_bytes": nbytes,
            "rotated": {"ms": rms, "GB/s": gbs(rms), "frac_hbm": gbs(rms) / pk["hbm_gbs"], "weight_copies": copies,
                        "protocol": f"{2 * copies} launches back to back over {copies} copies of W, grad_out and "
                                    "grad_X (more than twice the L2); time per launch = total / launches"}}


def time_e2e(c, outs, bsq, steps, warmup):
    """Same ops through the ABI with every step's inputs copied from pinned host memory and
    its gradients copied back, pipelined the way a training loop prefetches: three streams
    (copy-in, compute, copy-out) and two device buffer sets, so that step i+1's inputs load
    while step i computes and step i-1's gradients drain.  Returns (ms per step, bytes in,
    bytes out per step)."""
    import dataclasses

    def pinned(t):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h

    def like(t):
        return None if t is None else torch.empty_like(t)

    # the step's inputs on the host
    host = {"G": pinned(c["G"])}
    for name in ("W", "X"):
        pk = c[name]
        if pk is not None:
            host[name] = {k: pinned(getattr(pk, k)) for k in ("data", "scale", "tensor_scale")
                          if getattr(pk, k) is not None}
    if c["grouped"]:
        host["offsets"] = pinned(c["offsets_dev"])
    slots = []
    for _ in range(2):
        d = {"G": like(c["G"])}
        for name in ("W", "X"):
            pk = c[name]
            if pk is not None:
                d[name] = dataclasses.replace(pk, data=like(pk.data), scale=like(pk.scale),
                                              tensor_scale=like(pk.tensor_scale))
        if c["grouped"]:
            d["offsets"] = like(c["offsets_dev"])
        d["out"] = {n: torch.empty_like(o) for n, o in outs.items()}
        d["host_out"] = {n: torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for n, o in outs.items()}
        slots.append(d)
    h2d = host["G"].numel() * host["G"].element_size()
    h2d += sum(t.numel() * t.element_size() for name in ("W", "X") if name in host for t in host[name].values())
    if c["grouped"]:
        h2d += host["offsets"].numel() * host["offsets"].element_size()
    d2h = sum(o.numel() * o.element_size() for o in outs.values())
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        k = i % 2
        d = slots[k]
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_comp[k])       # step i-2 has finished reading this buffer set
            d["G"].copy_(host["G"], non_blocking=True)
            for name in ("W", "X"):
                if name in host:
                    for f, h in host[name].items():
                        getattr(d[name], f).copy_(h, non_blocking=True)
            if c["grouped"]:
                d["offsets"].copy_(host["offsets"], non_blocking=True)
            ev_in[k].record(s_in)
        s_comp.wait_event(ev_in[k])
        s_comp.wait_event(ev_out[k])          # step i-2's gradients have been read back
        cc = dict(c)
        cc["G"] = d["G"]
        cc["W"] = d["W"]
        cc["X"] = d.get("X")
        if c["grouped"]:
            cc["offsets_dev"] = d["offsets"]
        run_ops(cc, d["out"], bsq, stream=s_comp)
        ev_comp[k].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[k])
            for n, o in d["out"].items():
                d["host_out"][n].copy_(o, non_blocking=True)
            ev_out[k].record(s_out)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(steps):
        step(warmup + i)
    b.record(s_out)                           # after the last step's read-back
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps, h2d, d2h


def measure_workload(n, bsq, synth, dev, steps, warmup, flush, pk):
    """Every op of workload n on freshly generated inputs: median ms, TFLOP/s and roofline
    per op, and the step's TFLOP/s with its fractions of the burst and sustained peaks."""
    c = synth.make_config(n, device=dev, seed=0)
    if c["grouped"]:
        c["offsets_dev"] = torch.from_numpy(c["offsets"]).to(dev)
    outs = alloc_outputs(c, dev)
    ops = plan(c)
    per_op, step_ms, launches = time_ops(c, outs, bsq, steps, warmup, flush)
    st, code = bsq.get_device_error()
    if st != 0:
        raise SystemExit(f"device error {code} during workload {n}")
    r = {"ops": {}, "launches": launches}
    for name, fl, nb in ops:
        ms = statistics.median(per_op[name])
        r["ops"][name] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12, "roofline": op_roofline(fl, nb, ms, pk)}
        r["ops"][name]["roofline"]["traffic"] = profiled_traffic(c["name"], name)
    ms = statistics.median(step_ms)
    fl = sum(o[1] for o in ops)
    sp = step_plan(c)
    if sp is not None:
        r["backward"] = {"ms": ms, "tflops": sp[1] / (ms * 1e-3) / 1e12,
                         "roofline": op_roofline(sp[1], sp[2], ms, pk)}
        r["backward"]["roofline"]["traffic"] = profiled_traffic(c["name"], "backward")
    r["step_ms"] = ms
    r["tflops"] = fl / (ms * 1e-3) / 1e12
    r["frac_burst"] = r["tflops"] / pk["bf16_tflops"]
    r["frac_sustained"] = r["tflops"] / pk["bf16_tflops_sustained"]
    if not c["grouped"] and c["X"].fmt != 0:
        r["forward"] = measure_forward(c, bsq, synth, steps, warmup, flush, pk)
    if n in SMALL_M_WORKLOADS:
        # M = 16 token rows against this workload's weight as well (the split-K kernel)
        if "G_small" not in c:
            c["G_small"] = synth.randn((16, c["N"]), 1e-2, 7, dev, torch.bfloat16)
        r["small_m_dgrad"] = small_m_entry(c, bsq, steps, warmup, flush, pk)
    if n == 4:
        r["grouped_decode_dgrad"] = measure_grouped_decode(c, bsq, synth, steps, warmup, flush, pk)
    deq = None
    if n in DEQUANT_WORKLOADS:
        deq = measure_dequant(c["W"], bsq, steps, warmup, flush, pk)
    del c, outs
    torch.cuda.empty_cache()
    return r, deq


def measure_forward(c, bsq, synth, steps, warmup, flush, pk):
    """bsq_linear_forward (Y = X W^T) on the workload's packed X and W, and with a BF16 X of
    the same shape (a layer whose weight alone is quantized) under "bf16_activation"."""
    y = torch.empty((c["M"], c["N"]), dtype=torch.bfloat16, device=c["G"].device)
    stream = torch.cuda.current_stream()
    M, N, K = c["M"], c["N"], c["K"]
    fl = 2.0 * M * N * K

    def timed(X):
        for _ in range(warmup):
            bsq.linear_forward(X, c["W"], out=y)
        torch.cuda.synchronize()
        ts = []
        for _ in range(steps):
            flush.zero_()
            torch.cuda._sleep(HOST_COVER_CYCLES)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            bsq.linear_forward(X, c["W"], out=y)
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ms = statistics.median(ts)
        nb = packed_bytes(X) + packed_bytes(c["W"]) + 2.0 * M * N
        return {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12, "roofline": op_roofline(fl, nb, ms, pk)}

    r = timed(c["X"])
    r["roofline"]["traffic"] = profiled_traffic(c["name"], "forward")
    xb = synth.make_packed(synth.FMT_BF16, 1, M, K, 1.0, 77, y.device)
    r["bf16_activation"] = timed(xb)
    r["bf16_activation"]["roofline"]["traffic"] = profiled_traffic(c["name"], "forward_bf16_activation")
    del xb
    return r


# The standalone dequant is timed on the packed weight of these workloads (one per format);
# the M = 16 dgrad on the headline weight and on these.
DEQUANT_WORKLOADS = (3, 4, 5)
SMALL_M_WORKLOADS = (3,)
DECODE_ROWS = 64   # a decode-sized grouped batch: routed rows over the grouped workload's experts


def _timed(f, steps, warmup, flush):
    """Median ms of f() with L2 flushed before each timed call (CUDA events, current stream)."""
    for _ in range(warmup):
        f()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ts = []
    for _ in range(steps):
        flush.zero_()
        torch.cuda._sleep(HOST_COVER_CYCLES)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        f()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def measure_grouped_decode(c, bsq, synth, steps, warmup, flush, pk, rows=DECODE_ROWS):
    """Grouped dgrad of a decode-sized batch (`rows` grad_out rows routed over the workload's
    experts by the same law) through bsq_grouped_dgrad: GB/s of algorithmic bytes -- the
    packed weights and scales of the experts that received rows, read once, plus grad_out
    and grad_x."""
    E, N, K, W = c["E"], c["N"], c["K"], c["W"]
    counts = synth.zipf_counts(rows, E, 1.1, 5, force_empty=[e for e in (0, 31, 63) if e < E])
    offs = torch.from_numpy(synth.offsets_from_counts(counts)).to(c["G"].device)
    G = synth.randn((rows, N), 1.0, 3, c["G"].device, torch.bfloat16)
    out = torch.empty((rows, K), dtype=torch.bfloat16, device=G.device)
    ms = _timed(lambda: bsq.grouped_dgrad(G, W, offs, out=out), steps, warmup, flush)
    active = int((counts > 0).sum())
    nbytes = packed_bytes(W) * active / E + 2.0 * rows * N + 2.0 * rows * K
    return {"rows": rows, "experts_routed": active, "ms": ms, "algorithmic_bytes": nbytes,
            "GB/s": nbytes / (ms * 1e-3) / 1e9, "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "kernel": "smallm_dgrad_cluster_kernel"}


def measure_e5m2(c, outs, bsq, steps, warmup, flush, pk):
    """The quantized-gradient backward on the workload: bsq_linear_backward_e5m2 whole (the
    gradient's E5M2 quantization, then both products), and bsq_quantize_e5m2 alone (GB/s of
    2 bytes read, 1 byte of codes and 2 of the dequantized copy written per element)."""
    G, M, N, K = c["G"], c["M"], c["N"], c["K"]
    codes = torch.empty((M, N), dtype=torch.uint8, device=G.device)
    deq = torch.empty((M, N), dtype=torch.bfloat16, device=G.device)
    q_ms = _timed(lambda: bsq.quantize_e5m2(G, codes=codes, deq=deq), steps, warmup, flush)
    b_ms = _timed(lambda: bsq.linear_backward_e5m2(G, c["W"], c["X"], grad_x=outs["dgrad"], grad_w=outs["wgrad"]),
                  steps, warmup, flush)
    qb = 5.0 * M * N
    fl = 4.0 * M * N * K
    return {"backward_ms": b_ms, "backward_tflops": fl / (b_ms * 1e-3) / 1e12,
            "quantize": {"ms": q_ms, "algorithmic_bytes": qb, "GB/s": qb / (q_ms * 1e-3) / 1e9,
                         "frac_hbm": qb / (q_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                         "kernels": "amax_bf16_kernel + quantize_e5m2_kernel"}}


def measure_dequant(p, bsq, steps, warmup, flush, pk):
    """bsq_dequant of a packed operand to BF16 in HBM: GB/s of algorithmic bytes (packed
    bytes and scales read once, 2 bytes per element written)."""
    out = torch.empty((p.batch, p.rows, p.cols), dtype=torch.bfloat16, device=p.data.device)
    for _ in range(warmup):
        bsq.dequant(p, out=out)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ts = []
    for _ in range(steps):
        flush.zero_()
        torch.cuda._sleep(HOST_COVER_CYCLES)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        bsq.dequant(p, out=out)
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    ms = statistics.median(ts)
    nbytes = packed_bytes(p) + 2.0 * p.batch * p.rows * p.cols
    del out
    return {"shape": [p.batch, p.rows, p.cols], "fmt": p.fmt, "ms": ms, "algorithmic_bytes": nbytes,
            "GB/s": nbytes / (ms * 1e-3) / 1e9, "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]}


# ---------------------------------------------------------------- the oracle as a baseline
def oracle_sample(c, ncols, seed=0):
    """Time the CPU oracle on ncols sampled output columns of every op of the step.

    Returns (seconds, flops computed).  Dequantizes only the sampled columns of the
    packed operand (as the oracle does for sampled parity checks) and runs the float64
    products for them.
    """
    from oracle import dequant as D
    from oracle import gemm as Gm
    from block_scaled_gemm_fp8_gb300 import synth
    names = {0: D.FMT_BF16, 1: D.FMT_FP8, 2: D.FMT_MXFP4, 3: D.FMT_NVFP4}
    rng = np.random.default_rng(seed)
    cols = np.sort(rng.choice(c["K"], size=min(ncols, c["K"]), replace=False))
    g_bits = c["G_host"]
    t0 = time.perf_counter()
    g = Gm.as_f64(g_bits)
    flops = 0.0
    if not c["grouped"]:
        for key, p in (("W", c["W"]), ("X", c["X"])):
            d, s, ts = c[key + "_host"]
            b = D.dequant_cols(names[p.fmt], d, s, ts, p.rows, p.cols, cols)
            r = g @ b if key == "W" else g.T @ b
            flops += 2.0 * r.shape[0] * g.shape[1 if key == "W" else 0] * len(cols)
    else:
        offs = c["offsets"]
        d, s, ts = c["W_host"]
        p = c["W"]
        for e in range(c["E"]):
            r0, r1 = Gm.expert_rows(offs, e)
            if r1 > r0:
                b = D.dequant_cols(names[p.fmt], d, s, ts, p.rows, p.cols, cols, e, p.batch)
                _ = g[r0:r1] @ b
                flops += 2.0 * (r1 - r0) * p.rows * len(cols)
    return time.perf_counter() - t0, flops


def host_copies(c):
    from block_scaled_gemm_fp8_gb300 import synth
    c["G_host"] = synth.bf16_numpy(c["G"])
    for key in ("W", "X"):
        if c.get(key) is not None:
            c[key + "_host"] = c[key].numpy()


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except ImportError:
        pass
    return os.cpu_count()


# ---------------------------------------------------------------- replicas
def max_over_ranks(value, device=None):
    """The largest value over the ranks of the initialised process group (the slowest
    replica sets the job's time), or `value` itself when there is no group of two or more."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() < 2:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def job_tflops(world, flops_per_step, steps, total_ms):
    """Whole-job throughput: every replica does flops_per_step per step; the job takes total_ms."""
    return world * flops_per_step * steps / (total_ms * 1e-3) / 1e12


# ---------------------------------------------------------------- main
def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from block_scaled_gemm_fp8_gb300 import synth

    if args.impl == "reference":
        if rank != 0:
            return 0
        c = synth.make_config(args.config, device="cpu")
        host_copies(c)
        ops = plan(c)
        ncols = 32
        for _ in range(args.warmup):
            oracle_sample(c, ncols, seed=1)
        secs, flops = 0.0, 0.0
        for k in range(args.steps):
            s, f = oracle_sample(c, ncols, seed=2 + k)
            secs += s
            flops += f
        value = flops / secs / 1e12
        line = {"impl": "reference", "metric": "dgrad+wgrad TFLOP/s", "value": value, "unit": "TFLOP/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": c["name"], "ops": [o[0] for o in ops]},
                "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                                 "sample": f"{ncols} sampled output columns of every op per step"},
                "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from block_scaled_gemm_fp8_gb300 import bsq
    bsq.lib()
    if args.profile:
        return profile_run(args, bsq, synth, dev)

    c = synth.make_config(args.config, device=dev, seed=0)
    if c["grouped"]:
        c["offsets_dev"] = torch.from_numpy(c["offsets"]).to(dev)
    outs = alloc_outputs(c, dev)
    ops = plan(c)
    flops_step = sum(o[1] for o in ops)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    sampler = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    per_op, step_ms, launches = time_ops(c, outs, bsq, args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    total_ms = max_over_ranks(sum(step_ms), device=dev)
    value = job_tflops(world, flops_step, args.steps, total_ms)
    st, code = bsq.get_device_error()
    if st != 0:
        raise SystemExit(f"device error {code} during the benchmark")

    pk = peaks()
    # dominant kernel: the fused backward launch where the step is one, else the op with
    # the largest share of the step
    sp = step_plan(c)
    if sp is not None:
        dom, dom_flops, dom_bytes = sp
        dom_ms = statistics.mean(step_ms)
    else:
        avg = {n: statistics.mean(v) for n, v in per_op.items()}
        dom = max(avg, key=avg.get)
        dom_flops, dom_bytes = [(o[1], o[2]) for o in ops if o[0] == dom][0]
        dom_ms = avg[dom]
    r = op_roofline(dom_flops, dom_bytes, dom_ms, pk)
    roof = {"bound": r["bound"], "achieved": r["achieved"],
            "peak": pk["bf16_tflops"] if r["bound"] == "tensor" else pk["hbm_gbs"], "unit": r["unit"],
            "frac": r["frac"]}
    roof["traffic"] = profiled_traffic(c["name"], dom)
    roof["kernel"] = f"bsq_gemm_kernel ({'dgrad+wgrad, one launch' if dom == 'backward' else dom})"
    roof["ms"] = dom_ms
    roof["peak_source"] = pk["source"]

    line = {"metric": "dgrad+wgrad TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": c["name"], "M": c["M"], "N": c["N"], "K": c["K"], "E": c["E"],
                       "ops": [o[0] for o in ops], "l2": "flushed by a 256 MiB memset before every timed step",
                       "parallelism": "replicas" if world > 1 else "single"},
            "per_op_ms": {n: statistics.median(v) for n, v in per_op.items()},
            "per_op_tflops": {o[0]: o[1] / (statistics.median(per_op[o[0]]) * 1e-3) / 1e12 for o in ops},
            "roofline": roof, "gpu_launches": launches, "clocks": clocks}

    if not c["grouped"] and c["X"].fmt != 0:
        line["forward"] = measure_forward(c, bsq, synth, args.steps, args.warmup, flush, pk)
    if args.config == 2:
        line["small_m_dgrad"] = small_m_entry(c, bsq, args.steps, args.warmup, flush, pk)
    if args.config == 2:
        line["e5m2_backward"] = measure_e5m2(c, outs, bsq, max(5, args.steps // 2), args.warmup, flush, pk)
    if not args.no_e2e:
        ms, h2d, d2h = time_e2e(c, outs, bsq, max(3, args.steps // 2), 2)
        line["e2e"] = {"value": world * flops_step / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms}
    if not args.no_extra:
        # the other workloads (parity-test shapes too) and the standalone dequant, each
        # timed the same way; the headline line above is unchanged by them
        extra, deq = {}, {}
        for n in (1, 2, 3, 4, 5):
            if n == args.config:
                continue
            r, d = measure_workload(n, bsq, synth, dev, max(5, args.steps // 2), args.warmup, flush, pk)
            extra[synth.CONFIG_NAMES[n]] = r
            if d is not None:
                deq[synth.CONFIG_NAMES[n]] = d
            line["gpu_launches_extra"] = line.get("gpu_launches_extra", 0) + r["launches"]
        line["other_workloads"] = extra
        line["dequant"] = deq
        line["peaks"] = pk
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host_copies(c)
        ncols = 4096   # every output column of the MXFP4 4096^3 workload: the whole step, a few seconds
        secs, fl = oracle_sample(c, ncols)
        line["cpu_baseline"] = {"value": fl / secs / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(),
                                "kind": "oracle", "seconds": secs,
                                "sample": f"{ncols} sampled output columns of every op (float64 oracle)"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
