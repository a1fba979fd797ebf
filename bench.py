"""Benchmark of the DCNv2 forward on one GB300 (or N independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

One step = the whole forward through the C ABI: x -> channels-last,
weight repack, sampling descriptors, fused kernel (four of the library's
kernels). Inputs are
resident in device memory; L2 is flushed (a 256 MiB write, outside the
timing events) before every timed step. Step time and the fused kernel's
time are taken with CUDA events on the launching stream; the JSON line
reports TFLOP/s of the contraction (2*N*Cout*Ho*Wo*Cin/group*kh*kw flops),
microseconds per call, the fused kernel's roofline fraction, an end-to-end
number through host buffers, and the CPU oracle timed on the host cores.

--impl reference times the CPU oracle (the only other implementation of
this operator available here) on the same workload; see the oracle package.
Under torchrun (N > 1) every rank runs its own full replica of the workload
(weak scaling, no collective on the data path); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from modulated_deformable_convolution_gb300.workloads import CONFIG_ORDER, CONFIGS, EXTRA_ORDER, make_inputs  # noqa: E402

METRIC = "modulated deform-conv fwd TFLOP/s & µs/call at 1 GB300; % of roofline"
UNIT = "TFLOP/s"
FLUSH_BYTES = 256 << 20
FUSED_SOURCES = ["mdcn_fused.cu", "mdcn_ptx.cuh", "mdcn_layout.cuh", "mdcn_plan.h"]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def describe(case) -> str:
    Ho, Wo = case.out_hw
    return (f"{case.name}: N={case.N} Cin={case.Cin} Cout={case.Cout} H={case.H} W={case.W} -> Ho={Ho} Wo={Wo} "
            f"{case.kh}x{case.kw} stride={case.stride[0]} pad={case.padding[0]} dil={case.dilation[0]} "
            f"group={case.group} dg={case.deformable_group} bias={'yes' if case.bias else 'no'} dtype={case.dtype}")


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, local):
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return dist
    return None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, v: float) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            return json.load(open(p)), "measured"
        except Exception:
            pass
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), reasons=parts[4:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["active_mask", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for name, val in zip(names[1:], r["reasons"][1:]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def fused_source_hash() -> str:
    h = hashlib.sha256()
    for f in FUSED_SOURCES:
        h.update(open(os.path.join(ROOT, "modulated_deformable_convolution_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the fused kernel from a committed ncu summary,
    or None when there is none or the kernel changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        t = json.load(open(p))
        e = t.get(workload)
        if e and e.get("fused_source_hash") == fused_source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def measure_fp32_peaks(dev, n: int = 8192, reps: int = 10):
    """Dense fp32-input rates on this GPU, measured in this run with cuBLAS
    through torch.matmul (n^3 GEMM, 2*n^3 flops, best of `reps`, CUDA events):
    TF32 tensor cores allowed, and strict fp32. Returns TFLOP/s of each."""
    a = torch.randn(n, n, device=dev)
    b = torch.randn(n, n, device=dev)
    out = {}
    prev = torch.backends.cuda.matmul.allow_tf32
    try:
        for name, tf32 in (("tf32", True), ("fp32_strict", False)):
            torch.backends.cuda.matmul.allow_tf32 = tf32
            torch.matmul(a, b)
            torch.cuda.synchronize()
            best = float("inf")
            for _ in range(reps if tf32 else 3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                torch.matmul(a, b)
                e1.record()
                torch.cuda.synchronize()
                best = min(best, e0.elapsed_time(e1) * 1e-3)
            out[name] = 2.0 * n ** 3 / best / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    del a, b
    torch.cuda.empty_cache()
    return out


def peak_for(case, peaks, peak_src, fp32_peaks):
    """(peak TFLOP/s of the case's contraction, note). fp16/bf16: the measured
    bf16 burst (fp16 has the same dense rate). fp32: the split-TF32 contraction
    runs three TF32 MMAs per k-step, so a third of the TF32 rate measured in
    this run."""
    if case.dtype == "f32":
        if fp32_peaks and fp32_peaks.get("tf32"):
            return fp32_peaks["tf32"] / 3.0, "measured in this run: cuBLAS TF32 8192^3 / 3 passes (split-TF32)"
        return peaks["bf16_tflops"] * (1.1 / 2.25) / 3.0, f"{peak_src} bf16 burst x nominal tf32/bf16 ratio / 3"
    return peaks["bf16_tflops"], f"{peak_src} bf16 burst (fp16 has the same dense rate)"


def time_forward(mdcn, case, dev, steps, warmup, flush):
    """Device times of `steps` mdcn_forward calls (L2 flushed before each) and
    of the fused kernel alone after the step-wise prep calls, on one workload.
    Returns (step ms list, fused ms list, plan, status)."""
    d = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(case).items()}
    x, off, m, w, b = d["x"], d["offset"], d["mask"], d["weight"], d["bias"]
    h = mdcn.Handle(**case.attrs())
    ws = torch.empty(mdcn.mdcn_workspace_size(h, x, off, m, w, b), dtype=torch.uint8, device=dev)
    out = torch.empty(mdcn.mdcn_output_dims(h, x, off, m, w, b), dtype=x.dtype, device=dev)
    st = torch.cuda.current_stream(dev)
    plan = mdcn.mdcn_query_plan(h, x, off, m, w, b)
    for _ in range(warmup):
        flush.zero_()
        mdcn.mdcn_forward(h, x, off, m, w, b, out, ws, st)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda._sleep(int(2e5) * steps)
    for i in range(steps):
        flush.zero_()
        evs[i][0].record(st)
        mdcn.mdcn_forward(h, x, off, m, w, b, out, ws, st)
        evs[i][1].record(st)
    torch.cuda._sleep(int(2e5) * steps)
    for i in range(steps):
        flush.zero_()
        if plan["path"] == 2:
            # a direct plan is one kernel: mdcn_forward is that kernel alone
            fev[i][0].record(st)
            mdcn.mdcn_forward(h, x, off, m, w, b, out, ws, st)
            fev[i][1].record(st)
            continue
        mdcn.mdcn_prepare_input(h, x, off, m, w, b, ws, st)
        mdcn.mdcn_pack_weight(h, x, off, m, w, b, ws, st)
        fev[i][0].record(st)
        mdcn.mdcn_forward_prepared(h, x, off, m, w, b, out, ws, st)
        fev[i][1].record(st)
    torch.cuda.synchronize()
    s, bits = mdcn.mdcn_query_status(ws)
    return ([a.elapsed_time(c) for a, c in evs], [a.elapsed_time(c) for a, c in fev], plan,
            "ok" if s == mdcn.MDCN_OK else f"device status {bits:#x}")


def per_config_table(mdcn, dev, flush, peaks, peak_src, fp32_peaks, steps=20, warmup=5):
    """Every named workload through mdcn_forward: µs per call, contraction
    TFLOP/s, the fused kernel's time, and the roofline fractions of the step
    and of the fused kernel. Roofline time = max(flops / tensor peak, bytes /
    HBM bandwidth), bytes = x + offset + mask + weight + bias + output once."""
    table = {}
    for name in CONFIG_ORDER + EXTRA_ORDER:
        case = CONFIGS[name]
        step_ms, fused_ms, plan, status = time_forward(mdcn, case, dev, steps, warmup, flush)
        peak, note = peak_for(case, peaks, peak_src, fp32_peaks)
        t_mma = case.flops / (peak * 1e12)
        t_hbm = case.io_bytes / (peaks["hbm_gbs"] * 1e9)
        roof_s = max(t_mma, t_hbm)
        us = statistics.mean(step_ms) * 1e3
        kus = statistics.mean(fused_ms) * 1e3
        table[name] = {
            "workload": describe(case), "us_per_call": us, "tflops": case.flops / (us * 1e-6) / 1e12,
            "kernel_us": kus, "kernel_tflops": case.flops / (kus * 1e-6) / 1e12,
            "roofline_us": roof_s * 1e6, "bound": "tensor" if t_mma >= t_hbm else "hbm",
            "frac_step": roof_s / (us * 1e-6), "frac_kernel": roof_s / (kus * 1e-6),
            "peak_tflops": peak, "peak_source": note, "ctas": plan["ctas"], "split": plan["split"],
            "launches": plan["launches"], "path": "direct" if plan["path"] == 2 else "fused", "status": status,
        }
        log(f"[per_config] {name}: {us:.1f} us/call, kernel {kus:.1f} us, frac kernel "
            f"{table[name]['frac_kernel']:.3f}, {status}")
    return table


def cpu_oracle_time(case, inp, budget_s: float = 20.0):
    """Times the oracle as it stands on a bounded slice (whole output rows of
    every image and channel). Returns (flops of the slice, seconds, rows, threads)."""
    import oracle

    oracle.build()
    import numpy as np

    np64 = lambda t: None if t is None else t.detach().to("cpu", torch.float64).numpy()
    args = [np64(inp[k]) for k in ("x", "offset", "mask", "weight", "bias")]
    Ho, _ = case.out_hw
    flops_row = case.flops / Ho
    # one probe row to size the slice
    t0 = time.perf_counter()
    oracle.forward(*args, ho_range=(0, 1), **case.attrs())
    per_row = max(time.perf_counter() - t0, 1e-6)
    rows = int(max(1, min(Ho, budget_s / per_row)))
    t0 = time.perf_counter()
    oracle.forward(*args, ho_range=(0, rows), **case.attrs())
    dt = time.perf_counter() - t0
    return flops_row * rows, dt, rows, oracle.num_threads()


def run_reference(args, case, world, rank, dist):
    """The CPU oracle arm: K timed steps of a bounded slice of the workload."""
    barrier(dist)
    if rank != 0:
        return
    import oracle

    oracle.build()
    inp = make_inputs(case)
    np64 = lambda t: None if t is None else t.detach().to("cpu", torch.float64).numpy()
    a = [np64(inp[k]) for k in ("x", "offset", "mask", "weight", "bias")]
    Ho, _ = case.out_hw
    t0 = time.perf_counter()
    oracle.forward(*a, ho_range=(0, 1), **case.attrs())
    per_row = max(time.perf_counter() - t0, 1e-6)
    budget = 150.0 / max(1, args.steps + args.warmup)  # whole run within a few minutes
    rows = int(max(1, min(Ho, budget / per_row)))
    flops = case.flops / Ho * rows
    for _ in range(args.warmup):
        oracle.forward(*a, ho_range=(0, rows), **case.attrs())
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.forward(*a, ho_range=(0, rows), **case.attrs())
        times.append(time.perf_counter() - t0)
    sec = statistics.mean(times)
    value = flops / sec / 1e12
    sample = f"output rows 0..{rows - 1} of {Ho} (all images, all channels) of {case.name}"
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": describe(case)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, case, world, rank, local, dist):
    import modulated_deformable_convolution_gb300 as mdcn

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp_cpu = make_inputs(case)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp_cpu.items()}
    h = mdcn.Handle(**case.attrs())
    x, off, m, w, b = d["x"], d["offset"], d["mask"], d["weight"], d["bias"]
    ws = torch.empty(mdcn.mdcn_workspace_size(h, x, off, m, w, b), dtype=torch.uint8, device=dev)
    out = torch.empty(mdcn.mdcn_output_dims(h, x, off, m, w, b), dtype=x.dtype, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    plan = mdcn.mdcn_query_plan(h, x, off, m, w, b)

    def step():
        # the public call: prep launch(es), the fused kernel
        mdcn.mdcn_forward(h, x, off, m, w, b, out, ws, stream)

    def fused_step(ev):
        # the same work through the step-wise calls, to time the fused kernel
        # alone (a direct plan is one kernel: mdcn_forward is that kernel)
        if plan["path"] == 2:
            ev[0].record(stream)
            step()
            ev[1].record(stream)
            return
        mdcn.mdcn_prepare_input(h, x, off, m, w, b, ws, stream)
        mdcn.mdcn_pack_weight(h, x, off, m, w, b, ws, stream)
        ev[0].record(stream)
        mdcn.mdcn_forward_prepared(h, x, off, m, w, b, out, ws, stream)
        ev[1].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    s, bits = mdcn.mdcn_query_status(ws)
    if s != mdcn.MDCN_OK:
        raise RuntimeError(f"device status after warm-up: {bits:#x}")

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(dist)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    # The GPU first spins for ~0.1 ms per step, so the host has enqueued every
    # timed step before the first one runs: the events then time the device,
    # not the Python launch path. L2 is flushed before every step.
    torch.cuda._sleep(int(2e5) * args.steps)
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    clk = clocks.stop()
    torch.cuda._sleep(int(2e5) * args.steps)
    for i in range(args.steps):
        flush.zero_()
        fused_step(fev[i])
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(c) for a, c in evs]
    fused_ms = [a.elapsed_time(c) for a, c in fev]
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(dist, ms)
    s, bits = mdcn.mdcn_query_status(ws)
    if s != mdcn.MDCN_OK:
        raise RuntimeError(f"device status after the timed steps: {bits:#x}")

    # end to end through the C ABI with host buffers (mdcn_forward_host): each
    # step copies its inputs from pinned host memory, runs the forward and
    # copies the output back. Steps rotate over three streams, each with its own
    # device buffer, so one step's copies overlap the others' kernels (a caller
    # streaming batches; a fourth stream measured no faster); the single-stream
    # figure is reported beside it.
    pinned = {k: (None if v is None else v.contiguous().pin_memory()) for k, v in inp_cpu.items()}
    E2E_STREAMS = 3
    out_hosts = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(E2E_STREAMS)]
    h2d = sum(v.numel() * v.element_size() for v in pinned.values() if v is not None)
    d2h = out_hosts[0].numel() * out_hosts[0].element_size()
    e2e_steps = max(4, min(args.steps, 20))
    hb = mdcn.mdcn_host_buffer_size(h, pinned["x"], pinned["offset"], pinned["mask"], pinned["weight"],
                                    pinned["bias"])
    hbufs = [torch.empty(hb, dtype=torch.uint8, device=dev) for _ in range(E2E_STREAMS)]
    hstreams = [torch.cuda.Stream(dev) for _ in range(E2E_STREAMS)]

    def e2e_step(k, nstreams):
        i = k % nstreams
        mdcn.mdcn_forward_host(h, pinned["x"], pinned["offset"], pinned["mask"], pinned["weight"], pinned["bias"],
                               out_hosts[i], hbufs[i], hstreams[i])

    def e2e_time(nstreams):
        for k in range(2):
            e2e_step(k, nstreams)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dist)
        e0.record(stream)
        for hs in hstreams:
            hs.wait_event(e0)
        for k in range(e2e_steps):
            e2e_step(k, nstreams)
        for hs in hstreams:
            ev = torch.cuda.Event()
            ev.record(hs)
            stream.wait_event(ev)
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(dist, e0.elapsed_time(e1) / e2e_steps)

    e2e_ms = e2e_time(E2E_STREAMS)
    e2e_serial_ms = e2e_time(1)

    # ablation (two-stage im2col + cuBLAS design) for context, same flush rule
    abl_ms = None
    try:
        aws = torch.empty(mdcn.mdcn_im2col_gemm_workspace_size(h, x, off, m, w, b), dtype=torch.uint8, device=dev)
        a_out = torch.empty_like(out)
        for _ in range(2):
            mdcn.mdcn_forward_im2col_gemm(h, x, off, m, w, b, a_out, aws, stream)
        at = []
        for _ in range(min(args.steps, 10)):
            flush.zero_()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            mdcn.mdcn_forward_im2col_gemm(h, x, off, m, w, b, a_out, aws, stream)
            a1.record(stream)
            at.append((a0, a1))
        torch.cuda.synchronize()
        abl_ms = statistics.mean(a.elapsed_time(c) for a, c in at)
        del aws, a_out
    except Exception as e:  # the ablation is context only
        log("ablation skipped:", e)

    # the pack form (offset and mask from an ordinary convolution of x in front
    # of the deformable one), random front-end weights of the layer's shape,
    # same flush rule; its flops count both convolutions
    pack = None
    try:
        gp = torch.Generator().manual_seed(11)
        kh, kw = w.shape[2], w.shape[3]
        K = kh * kw
        dg = case.attrs()["deformable_group"]
        Cin = x.shape[1]
        w_om = (torch.randn(3 * dg * K, Cin, kh, kw, generator=gp) / (Cin * K) ** 0.5).to(x.dtype).to(dev)
        b_om = (0.5 * torch.randn(3 * dg * K, generator=gp)).to(x.dtype).to(dev)
        poff, pmsk = torch.empty_like(off), torch.empty_like(m)
        p_out = torch.empty_like(out)
        pws = torch.empty(mdcn.mdcn_pack_workspace_size(h, x, poff, pmsk, w, b), dtype=torch.uint8, device=dev)
        for _ in range(2):
            mdcn.mdcn_forward_pack(h, x, w_om, b_om, w, b, poff, pmsk, p_out, pws, stream)
        pt = []
        for _ in range(min(args.steps, 20)):
            flush.zero_()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            mdcn.mdcn_forward_pack(h, x, w_om, b_om, w, b, poff, pmsk, p_out, pws, stream)
            a1.record(stream)
            pt.append((a0, a1))
        torch.cuda.synchronize()
        if mdcn.mdcn_query_status(pws)[0] != mdcn.MDCN_OK:
            raise RuntimeError("pack form: device status set")
        pack_ms = statistics.mean(a.elapsed_time(c) for a, c in pt)
        fe_flops = 2 * x.shape[0] * 3 * dg * K * off.shape[2] * off.shape[3] * Cin * K
        pack = {"ms_per_call": pack_ms, "tflops": (case.flops + fe_flops) / (pack_ms * 1e-3) / 1e12,
                "front_end_flops": fe_flops, "launches": 5,
                "call": "mdcn_forward_pack: front-end conv (prep + fused kernel, plain), split into offset and "
                        "sigmoid(mask), then the deformable convolution (prep or weight pack + fused kernel)"}
        del pws, p_out, poff, pmsk
    except Exception as e:  # context only
        log("pack form skipped:", e)

    # the backward pass (gradients of sum(grad_out * y) for x, offset, mask,
    # weight and bias), same flush rule; its flops are the two contractions
    # (column gradients and weight gradient), twice the forward's
    bwd = None
    try:
        from modulated_deformable_convolution_gb300.workloads import make_grad_out
        go = make_grad_out(case).to(dev)
        gb = torch.empty_like(b) if b is not None else None
        grads = [torch.empty_like(t) for t in (x, off, m, w)]
        bws = torch.empty(mdcn.mdcn_backward_workspace_size(h, x, off, m, w, gb), dtype=torch.uint8, device=dev)
        for _ in range(2):
            mdcn.mdcn_backward(h, x, off, m, w, go, *grads, gb, bws, stream)
        bt = []
        for _ in range(min(args.steps, 20)):
            flush.zero_()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            mdcn.mdcn_backward(h, x, off, m, w, go, *grads, gb, bws, stream)
            a1.record(stream)
            bt.append((a0, a1))
        torch.cuda.synchronize()
        bwd_ms = statistics.mean(a.elapsed_time(c) for a, c in bt)
        bwd = {"ms_per_call": bwd_ms, "tflops": 2 * case.flops / (bwd_ms * 1e-3) / 1e12,
               "launches": mdcn.mdcn_backward_launches(h, x, off, m, w, gb),
               "call": "mdcn_backward: weight pack; per image chunk: channels-last x, column gradients "
                       "(tcgen05 GEMM for 16-bit I/O, cuBLAS for fp32), sampling backward (grad_offset, grad_mask, "
                       "grad_x reductions, columns), weight gradient (tcgen05 GEMM split over CTAs + ordered sum; "
                       "cuBLAS for fp32), grad_x to NCHW; weight gradient layout, bias reduction"}
        del bws, grads
    except Exception as e:  # context only
        log("backward skipped:", e)

    # every named workload (rank 0 of a single-GPU run), and the fp32 tensor
    # peaks measured on this GPU for the fp32 workloads' denominators
    peaks, peak_src = measured_peaks()
    fp32_peaks = None
    per_config = None
    if world == 1 and not args.no_per_config:
        try:
            fp32_peaks = measure_fp32_peaks(dev)
        except Exception as e:  # context only
            log("fp32 peak measurement skipped:", e)
        per_config = per_config_table(mdcn, dev, flush, peaks, peak_src, fp32_peaks)

    if rank != 0:
        return
    flops = case.flops
    value = world * flops / (ms_max * 1e-3) / 1e12
    fused_mean_s = statistics.mean(fused_ms) * 1e-3
    achieved = flops / fused_mean_s / 1e12
    peak, peak_note = peak_for(case, peaks, peak_src, fp32_peaks)
    kernel = "fused_kernel"
    if plan["path"] == 2:
        kernel = "direct_kernel" if plan["launches"] == 1 else "direct_kernel (channels-last form)"
    if case.io_bytes / (peaks["hbm_gbs"] * 1e9) > flops / (peak * 1e12):
        # little contraction per byte (depthwise): the algorithmic bytes against the measured HBM copy rate
        achieved_gbs = case.io_bytes / fused_mean_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved_gbs / peaks["hbm_gbs"], "traffic": profiled_traffic(case.name), "kernel": kernel,
                "peak_source": ("measured" if peak_src == "measured" else "fallback") + " HBM copy rate",
                "kernel_us": fused_mean_s * 1e6}
    else:
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": profiled_traffic(case.name), "kernel": kernel, "peak_source": peak_note,
                "kernel_us": fused_mean_s * 1e6}
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        f, sec, rows, thr = cpu_oracle_time(case, inp_cpu)
        Ho, _ = case.out_hw
        cpu = {"value": f / sec / 1e12, "unit": UNIT, "cores": thr, "kind": "oracle",
               "sample": f"output rows 0..{rows - 1} of {Ho} (all images, all channels), {sec:.1f} s"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "us_per_call": ms_max * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": case.dtype,
        "data": "synthetic",
        "config": {"workload": describe(case), "global_batch": case.N * world,
                   "l2": "flushed before every timed step (256 MiB write outside the events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "step": "mdcn_forward: channels-last x + weight pack, fused kernel (sampling in-kernel)"
                           + (", stream-K split tiles summed in-kernel" if plan["split"] else "")
                           + f" ({plan['launches']} launches)",
                   "plan": plan},
        "step_ms": {"mean": ms, "p10": sorted(step_ms)[len(step_ms) // 10],
                    "p90": sorted(step_ms)[(len(step_ms) * 9) // 10]},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "call": "mdcn_forward_host (C ABI, pinned host buffers), steps rotating over 3 streams x 3 device buffers",
                "single_stream": {"value": world * flops / (e2e_serial_ms * 1e-3) / 1e12,
                                  "ms_per_step": e2e_serial_ms}},
        "pack_form": pack,
        "backward": bwd,
        "ablation_im2col_gemm": None if abl_ms is None else {"ms_per_call": abl_ms,
                                                             "tflops": flops / (abl_ms * 1e-3) / 1e12},
        "gpu_launches": plan["launches"] * args.steps,
        "clocks": clk,
        "fp32_peaks_tflops": fp32_peaks,
        "per_config": per_config,
    }
    print(json.dumps(line), flush=True)


def run_fused_only(args, case):
    """Profiling aid: prepares the workspace once, then launches only the fused
    kernel args.fused_only times (after one untimed launch), each after an L2
    flush, and prints the median CUDA-event time. Used for ncu captures of the
    fused kernel (`-k regex:fused_kernel -s 1 -c 1`)."""
    import modulated_deformable_convolution_gb300 as mdcn

    dev = torch.device("cuda", 0)
    d = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(case).items()}
    x, off, m, w, b = d["x"], d["offset"], d["mask"], d["weight"], d["bias"]
    h = mdcn.Handle(**case.attrs())
    ws = torch.empty(mdcn.mdcn_workspace_size(h, x, off, m, w, b), dtype=torch.uint8, device=dev)
    out = torch.empty(mdcn.mdcn_output_dims(h, x, off, m, w, b), dtype=x.dtype, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream(dev)
    mdcn.mdcn_prepare_input(h, x, off, m, w, b, ws, st)
    mdcn.mdcn_pack_weight(h, x, off, m, w, b, ws, st)
    mdcn.mdcn_forward_prepared(h, x, off, m, w, b, out, ws, st)
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e5) * args.fused_only)
    evs = []
    for _ in range(args.fused_only):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        mdcn.mdcn_forward_prepared(h, x, off, m, w, b, out, ws, st)
        e1.record(st)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    s, bits = mdcn.mdcn_query_status(ws)
    us = statistics.median(a.elapsed_time(c) for a, c in evs) * 1e3
    print(json.dumps({"workload": case.name, "fused_kernel_us": us, "tflops": case.flops / (us * 1e-6) / 1e12,
                      "status": s}), flush=True)


def run_prep_vs_copy(args, case):
    """Profiling aid: args.prep_vs_copy rounds of, each after an L2 flush, a
    plain elementwise copy of x (PyTorch), the channels-last transpose alone,
    the weight pack alone and one mdcn_forward (prep + fused kernel); prints
    the mean CUDA-event time of each. Used for the ncu launch list that puts
    the prep beside a copy of the same bytes."""
    import modulated_deformable_convolution_gb300 as mdcn

    dev = torch.device("cuda", 0)
    d = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(case).items()}
    a = (d["x"], d["offset"], d["mask"], d["weight"], d["bias"])
    h = mdcn.Handle(**case.attrs())
    ws = torch.empty(mdcn.mdcn_workspace_size(h, *a), dtype=torch.uint8, device=dev)
    out = torch.empty(mdcn.mdcn_output_dims(h, *a), dtype=a[0].dtype, device=dev)
    y = torch.empty_like(d["x"])
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream(dev)
    steps = {
        "copy_x": lambda: torch.add(d["x"], 0, out=y),
        "prepare_input": lambda: mdcn.mdcn_prepare_input(h, *a, ws, st),
        "pack_weight": lambda: mdcn.mdcn_pack_weight(h, *a, ws, st),
        "forward": lambda: mdcn.mdcn_forward(h, *a, out, ws),
    }
    evs = {k: [] for k in steps}
    for _ in range(args.prep_vs_copy):
        for k, fn in steps.items():
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            fn()
            e1.record(st)
            evs[k].append((e0, e1))
    torch.cuda.synchronize()
    print(json.dumps({"workload": case.name, **{k + "_us": statistics.mean(x.elapsed_time(y) for x, y in v) * 1e3
                                               for k, v in evs.items()}}), flush=True)


def run_backward_only(args, case):
    """Profiling aid: runs mdcn_backward args.backward_only times (after one
    untimed call), each after an L2 flush, and prints the median CUDA-event
    time per call. Used for the launch list of the backward's kernels."""
    import modulated_deformable_convolution_gb300 as mdcn
    from modulated_deformable_convolution_gb300.workloads import make_grad_out

    dev = torch.device("cuda", 0)
    d = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(case).items()}
    x, off, m, w, b = d["x"], d["offset"], d["mask"], d["weight"], d["bias"]
    go = make_grad_out(case).to(dev)
    h = mdcn.Handle(**case.attrs())
    gb = torch.empty_like(b) if b is not None else None
    grads = [torch.empty_like(t) for t in (x, off, m, w)]
    ws = torch.empty(mdcn.mdcn_backward_workspace_size(h, x, off, m, w, gb), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream(dev)
    mdcn.mdcn_backward(h, x, off, m, w, go, *grads, gb, ws, st)
    torch.cuda.synchronize()
    evs = []
    for _ in range(args.backward_only):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        mdcn.mdcn_backward(h, x, off, m, w, go, *grads, gb, ws, st)
        e1.record(st)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    us = statistics.median(a.elapsed_time(c) for a, c in evs) * 1e3
    print(json.dumps({"workload": case.name, "backward_us": us, "tflops": 2 * case.flops / (us * 1e-6) / 1e12,
                      "launches": mdcn.mdcn_backward_launches(h, x, off, m, w, gb)}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="neck_f16", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the table of every named workload (and the fp32 peak measurement)")
    ap.add_argument("--fused-only", type=int, default=0, metavar="N",
                    help="profiling aid: time N launches of the fused kernel alone")
    ap.add_argument("--backward-only", type=int, default=0, metavar="N",
                    help="profiling aid: time N calls of mdcn_backward alone")
    ap.add_argument("--prep-vs-copy", type=int, default=0, metavar="N",
                    help="profiling aid: N rounds of a plain copy of x, the prep kernels and one forward")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_info()
    dist = init_dist(world, local)
    case = CONFIGS[args.config]
    try:
        if args.impl == "reference":
            run_reference(args, case, world, rank, dist)
        elif args.fused_only:
            from modulated_deformable_convolution_gb300 import build

            build.build()
            run_fused_only(args, case)
        elif args.backward_only:
            from modulated_deformable_convolution_gb300 import build

            build.build()
            run_backward_only(args, case)
        elif args.prep_vs_copy:
            from modulated_deformable_convolution_gb300 import build

            build.build()
            run_prep_vs_copy(args, case)
        else:
            from modulated_deformable_convolution_gb300 import build

            if not os.path.exists(os.path.join(ROOT, "modulated_deformable_convolution_gb300", "libmdcn.so")):
                build.build()
            run_ours(args, case, world, rank, local, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
