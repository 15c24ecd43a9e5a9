#!/usr/bin/env python
"""Throughput of the INT8 NCxHWx<32> Conv2d fprop path on GB300.

One step = one i8c_plan_run (fp16 filter staging kernel + the tcgen05
implicit-GEMM kernel) over one batch of the synthetic workload, inputs
resident in HBM.  The default workload is the largest of the five, the
dilated 5x9 layer of the kernel-benchmark trace (N=8 C=32 512x512 K=64).
Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--all]
  python bench.py --impl reference ...   # the CPU oracle, timed on the host

With N > 1 (torchrun) every rank runs an independent replica on its own
GPU (the convolution has no exchange step): value = work of all ranks /
max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "INT8 conv fprop TOPS (1 GB300) and % of dense INT8 tensor-core roofline"
DEFAULT_WORKLOAD = "n8c32h512k64r5x9d2x3"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_TENSOR_TFLOPS = 1900.0


def ops_of(wl) -> int:
    # 2*N*K*P*Q*C*R*S with P, Q from the library (not the oracle)
    import int8_implicit_gemm_gb300 as ext
    P, Q = ext.i8c_output_size(wl.shape_tuple())
    return 2 * wl.N * wl.K * P * Q * wl.C * wl.R * wl.S


def tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        # kind::f16 (fp16 operands) runs at the bf16 rate: nominal ratio 1.
        return float(d["bf16_tflops"]), "of measured (bf16 burst cuBLAS; fp16 kind::f16 at the same nominal rate)"
    except Exception:
        return FALLBACK_TENSOR_TFLOPS, "of fallback (1.9 PFLOP/s bf16; fp16 at the same nominal rate)"


F32_SOURCES = ("direct_f32.cu",)  # the fp32 direct convolution's kernel source


def kernel_source_digest(workload: str | None = None) -> str:
    """Digest of the kernel sources a workload's traffic figure depends on:
    the fp32 direct convolution's own file for the fp32 workload, every other
    source for the int8 workloads."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "int8_implicit_gemm_gb300", "csrc")
    f32 = workload == synth.F32_WORKLOAD.name
    for name in sorted(os.listdir(csrc)):
        if not name.endswith((".cu", ".cuh", ".h")) or (name in F32_SOURCES) != f32:
            continue
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def max_over_ranks(ms: float, world: int, device: str = "cuda") -> float:
    """The job's time: every rank times the same K steps between barriers,
    and the slowest rank sets the pace (all-reduce MAX; gloo on CPU tensors
    works the same way as NCCL on device tensors)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: the units all replicas processed per second."""
    return world * units_per_rank / (ms_per_step * 1e-3)


def ncu_counters(workload: str):
    """The workload's kernel counters from the committed ncu summary (DRAM
    bytes per launch, tensor-pipe and DRAM throughput percentages), if they
    were taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "conv_fprop_dram_traffic.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
    except Exception:
        return None
    entry = d.get("workloads", {}).get(workload)
    if entry is None or entry.get("source_digest") != kernel_source_digest(workload):
        return None
    return entry


def dram_traffic(workload: str):
    """Per-launch DRAM bytes of the workload's kernel from the committed ncu
    summary, if it was taken on the current kernel sources."""
    entry = ncu_counters(workload)
    return None if entry is None else entry.get("bytes_per_launch")


# The tensor-core engine the int8 path runs on (tcgen05 kind::f16): the engine
# probe measured 128 SM cycles per M = 128, N = 256, K = 16 MMA, that is
# 128*256*16 / 128 = 4096 multiply-adds, or 8192 ops, per SM cycle.
ENGINE_OPS_PER_SM_CLOCK = 2 * 128 * 256 * 16 / 128


def engine_peak(sms: int):
    """Peak of the engine actually used: ops per SM clock x SMs x the maximum
    SM clock (MEASURED_PEAKS.json's sm_max_mhz, else 2070 MHz)."""
    mhz = 2070.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            mhz = float(json.load(fh)["sm_max_mhz"])
    except Exception:
        pass
    return ENGINE_OPS_PER_SM_CLOCK * sms * mhz * 1e6 / 1e12, (
        f"tcgen05 kind::f16 at 8192 ops per SM cycle (engine probe: 128 cycles per 128x256x16 MMA) x {sms} SMs "
        f"x {mhz:.0f} MHz")


class ClockSampler:
    """nvidia-smi clocks, utilisation and throttle reasons sampled every 20 ms;
    the summary keeps the samples taken while the GPU was busy."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.2)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.strip()]
        os.unlink(self.out.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                if float(r[9]) < 50:  # idle sample (before or after the load)
                    continue
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                for name, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(name)
            except Exception:
                continue
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "note": "samples at >= 50% utilisation, 20 ms apart, over the timed "
                                             "steps and the kernel-timing steps that follow them"}


def cpu_oracle_rate(wl, budget_s: float, max_images: int | None = None):
    """Time the CPU oracle (as it stands) on the first images of the workload
    until about budget_s seconds of work are done.  Returns (TOPS, cores, sample)."""
    import oracle
    x = wl.activations_nchw()
    f = wl.filters_kcrs()
    shape = list(wl.shape_tuple())
    orc = oracle.Oracle()
    P, Q = orc.out_size(wl.shape_tuple())
    cores = os.cpu_count() or 1
    n_img, done_ops, elapsed = 1, 0, 0.0
    limit = wl.N if max_images is None else min(wl.N, max_images)
    while True:
        shape[0] = n_img
        t0 = time.perf_counter()
        orc.conv2d_fprop(x[:n_img], f, tuple(shape), wl.alpha, threads=cores)
        dt = time.perf_counter() - t0
        done_ops = 2 * n_img * wl.K * P * Q * wl.C * wl.R * wl.S
        elapsed = dt
        if dt >= budget_s / 4 or n_img >= limit:
            break
        n_img = min(limit, n_img * 4 if dt < budget_s / 16 else n_img * 2)
    sample = f"{n_img} of {wl.N} images, all {wl.K} output channels ({done_ops / 2:.3g} multiply-adds)"
    return done_ops / elapsed / 1e12, cores, sample, elapsed


def run_ours(args, wl, rank, world):
    import torch
    import int8_implicit_gemm_gb300 as ext
    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    shape = wl.shape_tuple()
    P, Q = ext.i8c_output_size(shape)
    ops = ops_of(wl)
    x_bytes = wl.N * wl.C * wl.H * wl.W
    f_bytes = wl.K * wl.C * wl.R * wl.S
    y_bytes = wl.N * wl.K * P * Q

    # seeded inputs, packed on the device by the library's layout kernels
    x_nchw = torch.from_numpy(wl.activations_nchw()).cuda()
    f_kcrs = torch.from_numpy(wl.filters_kcrs()).cuda()
    x0 = torch.empty(x_bytes, dtype=torch.int8, device="cuda")
    f0 = torch.empty(f_bytes, dtype=torch.int8, device="cuda")
    ext.i8c_pack_nchw_to_ncxhwx32(x_nchw, x0, wl.N, wl.C, wl.H, wl.W)
    ext.i8c_pack_kcrs_to_cxrskx32(f_kcrs, f0, wl.K, wl.C, wl.R, wl.S)
    del x_nchw, f_kcrs
    # rotate distinct buffer sets so that the sets together exceed L2
    set_bytes = x_bytes + f_bytes + y_bytes
    nsets = max(1, min(64, math.ceil(2 * L2_BYTES / set_bytes)))
    sets = []
    for i in range(nsets):
        xi = x0 if i == 0 else x0.clone()
        fi = f0 if i == 0 else f0.clone()
        sets.append((xi, fi, torch.empty(y_bytes, dtype=torch.int8, device="cuda")))
    # The timed steps run an uninstrumented plan; a second plan of the same
    # shape brackets each convolution kernel with CUDA events (which keep the
    # kernel from overlapping the filter conversion) for the roofline figure.
    plan = ext.Plan(shape)
    plan_k = ext.Plan(shape, timing_events=max(1, args.steps))
    stream = torch.cuda.current_stream()

    def step(i, pl=plan):
        xi, fi, yi = sets[i % nsets]
        pl.run(xi, fi, yi, wl.alpha, stream)

    for i in range(args.warmup):
        step(i)
        step(i, plan_k)
    torch.cuda.synchronize()
    assert plan.status(stream) == 0 and plan_k.status(stream) == 0
    plan_k.kernel_time()  # discard warm-up launches

    # The K timed steps are captured once into a CUDA graph (the library's
    # launches are capturable) and replayed in the timed region; --no-graph
    # launches them one by one instead.  Both are timed; `value` is the graph.
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    stream_ms = ev0.elapsed_time(ev1)
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        gstream = torch.cuda.Stream()
        launches0 = ext.launch_count()
        with torch.cuda.graph(graph, stream=gstream):
            cs = torch.cuda.current_stream()
            for i in range(args.steps):
                xi, fi, yi = sets[i % nsets]
                plan.run(xi, fi, yi, wl.alpha, cs)
        graph_launches = ext.launch_count() - launches0
        graph.replay()  # untimed warm replay
        torch.cuda.synchronize()
        assert plan.status(stream) == 0

    clocks = ClockSampler(dev) if (rank == 0 and not args.no_clocks) else None
    if clocks:
        clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = ext.launch_count()
    t_wall0 = time.perf_counter()
    ev0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_wall = time.perf_counter() - t_wall0
    launches = graph_launches if graph is not None else ext.launch_count() - launches0
    total_ms = ev0.elapsed_time(ev1)
    # kernel timing (event-bracketed plan), repeated for at least ~0.5 s so
    # that the clock sampler sees the GPU under this load
    t_k0 = time.perf_counter()
    kern_ms, kern_n = 0.0, 0
    while True:
        for i in range(args.steps):
            step(i, plan_k)
        torch.cuda.synchronize()
        ms_, n_ = plan_k.kernel_time()
        kern_ms += ms_
        kern_n += n_
        if time.perf_counter() - t_k0 > 0.5 or clocks is None:
            break
    clock_rec = clocks.stop() if clocks else None
    st = plan.status(stream) or plan_k.status(stream)
    if st != 0:
        raise RuntimeError(f"device status {ext.status_string(st)}")

    total_ms = max_over_ranks(total_ms, world)
    ms_per_step = total_ms / args.steps
    value = job_rate(ops, world, ms_per_step) / 1e12

    # End to end through the C-ABI on pinned host buffers: every step copies
    # x and f in, runs and copies y out.  i8c_plan_run_host_pipelined
    # overlaps step i's run with step i+1's input copy and step i-1's output
    # copy (the plan's two staging sets and copy streams); the serial form
    # (i8c_plan_run_host: copy in, run, copy out on one stream) is reported
    # beside it.
    plan_h = ext.Plan(shape, host_staging=2)
    xh = x0.cpu().pin_memory()
    fh = f0.cpu().pin_memory()
    yh = torch.empty(y_bytes, dtype=torch.int8).pin_memory()
    e2e_steps = max(3, min(args.steps, 50))
    for _ in range(2):
        plan_h.run_host(xh, fh, yh, wl.alpha, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        plan_h.run_host(xh, fh, yh, wl.alpha, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    assert plan_h.status(stream) == 0
    e2e_serial_ms = e0.elapsed_time(e1) / e2e_steps
    plan_h.run_host_pipelined([xh] * 4, [fh] * 4, [yh] * 4, [wl.alpha] * 4, stream)  # warm-up
    torch.cuda.synchronize()
    e0.record(stream)
    plan_h.run_host_pipelined([xh] * e2e_steps, [fh] * e2e_steps, [yh] * e2e_steps, [wl.alpha] * e2e_steps, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    assert plan_h.status(stream) == 0
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    plan_h.destroy()

    peak, peak_note = tensor_peak()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    epeak, epeak_note = engine_peak(sms)
    kernel_name = {1: "conv_fprop_tc_kernel", 4: "conv_fprop_tr_kernel", 5: "conv_fprop_tr_kernel"}.get(
        plan.info["kernel_variant"], "conv_fprop_halo_kernel")
    bracketed_ms = kern_ms / max(1, kern_n)
    prepacked_ms = None
    if plan.info["kernels_per_run"] != 1:
        prepacked_ms = prepacked_burst(shape, sets, wl.alpha, args.steps, stream)
    kern_avg_ms, kern_how = kernel_duration(plan.info, ms_per_step, bracketed_ms, prepacked_ms)
    achieved = ops / (kern_avg_ms * 1e-3) / 1e12
    counters = ncu_counters(wl.name)
    traffic = None if counters is None else counters.get("bytes_per_launch")
    result = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "s8 in/out; s8 x s8 products on fp16 tensor-core operands, fp32 chunks flushed to exact s32",
        "data": "synthetic (seeded xoshiro256**, uniform/normal int8 per workload)",
        "config": {"workload": wl.name, "shape": dict(zip(
            ["N", "C", "H", "W", "K", "R", "S", "pad_h", "pad_w", "stride_h", "stride_w", "dil_h", "dil_w"], shape)),
            "P": P, "Q": Q, "alpha": wl.alpha,
            "l2": f"{nsets} rotating input/output sets, {nsets * set_bytes / 2**20:.0f} MiB total > 129 MiB L2",
            "plan": {k: plan.info[k] for k in ("kernel_variant", "block_m", "block_n", "num_tiles", "num_ctas",
                                              "num_chunks", "chunk_slices", "acc_buffers", "smem_bytes",
                                              "filter_run", "filter_stages", "tail_split", "work_units")},
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": kernel_name, "kernel_ms": round(kern_avg_ms, 6), "kernel_ms_how": kern_how,
                     "kernel_ms_bracketed": round(bracketed_ms, 6),
                     "algorithmic_bytes": x_bytes + f_bytes + y_bytes,
                     "engine_peak": round(epeak, 1), "frac_engine": round(achieved / epeak, 4),
                     "ncu": None if counters is None else {
                         k: counters.get(k) for k in ("tensor_pipe_active_pct", "dram_gbs", "duration_us", "source")},
                     "note": f"int8 ops (2*N*K*P*Q*C*R*S) per launch / kernel_ms; peak {peak_note}; engine_peak "
                             f"{epeak_note}"},
        "e2e": {"value": round(ops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TOPS", "ms_per_step": round(e2e_ms, 6),
                "h2d_bytes_per_step": x_bytes + f_bytes, "d2h_bytes_per_step": y_bytes,
                "path": "i8c_plan_run_host_pipelined (C-ABI): H2D of x and f from pinned host memory and D2H of y "
                        "on the plan's copy streams with two device staging sets, overlapped across steps",
                "serial_ms_per_step": round(e2e_serial_ms, 6),
                "serial_path": "i8c_plan_run_host (copy in, run, copy out on one stream)"},
        "gpu_launches": launches,
        "launch": {"mode": "cuda graph of the K steps, replayed once" if graph is not None else "stream",
                   "ms_per_step_stream_launches": round(stream_ms / args.steps, 6)},
        "wall_s_timed_region": round(t_wall, 4),
    }
    if clock_rec is not None:
        result["clocks"] = clock_rec
    graph = None  # release the captured launches before the plan's memory
    plan.destroy()
    plan_k.destroy()
    if rank == 0 and not args.no_all:
        # every workload's conv-kernel time and roofline fraction, quickly
        # (device-resident random inputs; the bench line's own numbers above
        # are the headline)
        result["all_workloads"] = {w.name: bench_one_quick(w) for w in synth.WORKLOADS}
    if rank == 0 and world == 1 and not args.no_cpu:
        v, cores, sample, el = cpu_oracle_rate(wl, args.cpu_budget)
        result["cpu_baseline"] = {"value": round(v, 6), "unit": "TOPS", "cores": cores, "kind": "oracle",
                                  "sample": sample, "seconds": round(el, 2)}
    return result


F32_METRIC = "fp32 direct conv TFLOP/s (kernel-benchmark trace layer, 1 GB300) and % of the fp32 SIMT roofline"


def simt_fp32_peak(sms: int):
    """fp32 FMA peak of the SIMT cores: SMs x 128 FMA lanes x 2 flops x the
    maximum SM clock (MEASURED_PEAKS.json's sm_max_mhz, else 2070 MHz)."""
    mhz, note = 2070.0, "nominal maximum SM clock 2070 MHz"
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            mhz = float(json.load(fh)["sm_max_mhz"])
            note = f"measured maximum SM clock {mhz:.0f} MHz"
    except Exception:
        pass
    return sms * 128 * 2 * mhz * 1e6 / 1e12, f"{sms} SMs x 128 fp32 FMA lanes x 2 flops x {note}"


def run_f32(args, rank, world):
    """The fp32 direct convolution (i8c_conv2d_fprop_f32) on the trace's layer."""
    import torch
    import int8_implicit_gemm_gb300 as ext
    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    wl = synth.F32_WORKLOAD
    shape = wl.shape_tuple()
    P, Q = ext.i8c_output_size(shape)
    ops = 2 * wl.N * wl.K * P * Q * wl.C * wl.R * wl.S
    xh = torch.from_numpy(wl.inputs_nchw())
    wh = torch.from_numpy(wl.weights_kcrs())
    bh = torch.from_numpy(wl.bias())
    x, w, b = xh.cuda(), wh.cuda(), bh.cuda()
    y = torch.empty((wl.N, wl.K, P, Q), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        ext.i8c_conv2d_fprop_f32(x, w, b, y, shape, stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(dev) if (rank == 0 and not args.no_clocks) else None
    if clocks:
        clocks.start()
    if world > 1:
        torch.distributed.barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    launches0 = ext.launch_count()
    ev0.record(stream)
    for _ in range(args.steps):
        ext.i8c_conv2d_fprop_f32(x, w, b, y, shape, stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    launches = ext.launch_count() - launches0
    total_ms = ev0.elapsed_time(ev1)
    clock_rec = clocks.stop() if clocks else None
    total_ms = max_over_ranks(total_ms, world)
    ms = total_ms / args.steps
    value = job_rate(ops, world, ms) / 1e12
    # end to end: pinned host inputs copied in, the call, the output copied back
    xp, wp, bp = xh.pin_memory(), wh.pin_memory(), bh.pin_memory()
    yp = torch.empty(y.shape, dtype=torch.float32).pin_memory()
    e2e_steps = max(2, min(args.steps, 5))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        x.copy_(xp, non_blocking=True)
        w.copy_(wp, non_blocking=True)
        b.copy_(bp, non_blocking=True)
        ext.i8c_conv2d_fprop_f32(x, w, b, y, shape, stream)
        yp.copy_(y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak, peak_note = simt_fp32_peak(sms)
    result = {
        "metric": F32_METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded xoshiro256**: x uniform [0,1), w and "
                                                    "bias uniform [-1/sqrt(C*R*S), 1/sqrt(C*R*S)))",
        "config": {"workload": wl.name, "shape": dict(zip(
            ["N", "C", "H", "W", "K", "R", "S", "pad_h", "pad_w", "stride_h", "stride_w", "dil_h", "dil_w"], shape)),
            "P": P, "Q": Q, "l2": "inputs 268 MB and outputs 516 MB, both larger than the 129 MiB L2",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "alu", "achieved": round(ops / (ms * 1e-3) / 1e12, 2), "peak": round(peak, 1),
                     "unit": "TFLOP/s", "frac": round(ops / (ms * 1e-3) / 1e12 / peak, 4),
                     "traffic": dram_traffic(wl.name), "kernel": "conv_f32_direct_kernel",
                     "note": f"2*N*K*P*Q*C*R*S flops per call / CUDA-event time per call (weight transpose + "
                             f"convolution); peak {peak_note}"},
        "e2e": {"value": round(ops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s", "ms_per_step": round(e2e_ms, 6),
                "h2d_bytes_per_step": 4 * (xh.numel() + wh.numel() + bh.numel()),
                "d2h_bytes_per_step": 4 * y.numel(), "path": "pinned host copies + i8c_conv2d_fprop_f32"},
        "gpu_launches": launches,
    }
    if clock_rec is not None:
        result["clocks"] = clock_rec
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        orc = oracle.Oracle()
        xs, ws, bs = xh.numpy()[:1], wh.numpy(), bh.numpy()
        cores = os.cpu_count() or 1
        k = 1
        while True:
            sshape = (1,) + tuple(shape[1:4]) + (k,) + tuple(shape[5:])
            t0 = time.perf_counter()
            orc.conv_f64(xs, ws[:k], sshape, bias=bs[:k], threads=cores)
            dt = time.perf_counter() - t0
            if dt >= args.cpu_budget / 4 or k >= wl.K:
                break
            k = min(wl.K, k * 4 if dt < args.cpu_budget / 16 else k * 2)
        s_ops = 2 * k * P * Q * wl.C * wl.R * wl.S
        result["cpu_baseline"] = {"value": round(s_ops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
                                  "kind": "oracle", "sample": f"1 of {wl.N} images, {k} of {wl.K} output channels "
                                                              f"(double precision)", "seconds": round(dt, 2)}
    return result


def run_f32_reference(args, rank, world):
    """The double-precision oracle of the fp32 direct convolution as the
    reference arm: each step is a bounded sample (the first 64 input rows of
    one image, 16 of the 64 output channels), timed on the host cores."""
    if rank != 0:
        return None
    import oracle
    wl = synth.F32_WORKLOAD
    shape = wl.shape_tuple()
    orc = oracle.Oracle()
    k, rows = 16, 64
    x, w, b = wl.inputs_nchw()[:1, :, :rows], wl.weights_kcrs()[:k], wl.bias()[:k]
    sshape = (1, shape[1], rows, shape[3], k) + tuple(shape[5:])
    P, Q = orc.out_size(sshape)
    cores = os.cpu_count() or 1
    for _ in range(args.warmup):
        orc.conv_f64(x, w, sshape, bias=b, threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.conv_f64(x, w, sshape, bias=b, threads=cores)
    dt = time.perf_counter() - t0
    v = 2 * k * P * Q * wl.C * wl.R * wl.S * args.steps / dt / 1e12
    sample = f"first {rows} input rows of 1 of {wl.N} images, {k} of {wl.K} output channels per step (double precision)"
    return {"impl": "reference", "metric": F32_METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def kernel_duration(info, step_ms, bracketed_ms, prepacked_ms=None):
    """The convolution kernel's average launch duration.  When a run is that
    one kernel (the filter converted inside it), the K timed steps are K
    back-to-back launches of it, so the CUDA events around the timed region
    measure it directly (launch gaps included).  Otherwise (a conversion
    kernel first) the kernel alone runs back to back in prepacked runs (the
    filter converted once, i8c_plan_set_filter), timed the same way; without
    those, the plan's own events around each convolution launch, which keep
    it from overlapping the conversion and so include its launch latency."""
    if info["kernels_per_run"] == 1:
        return step_ms, "CUDA events around the timed region / steps: one launch of the kernel per step"
    if prepacked_ms is not None:
        return prepacked_ms, ("CUDA events around back-to-back prepacked runs / runs: one launch of the kernel per "
                              "run, the filter converted once beforehand")
    return bracketed_ms, "CUDA events around each launch of the kernel (plan timing events)"


def prepacked_burst(shape, sets, alpha, steps, stream):
    """ms per run of back-to-back prepacked runs (the convolution kernel
    alone) over the rotating input sets, the filter set once."""
    import torch
    import int8_implicit_gemm_gb300 as ext
    plan = ext.Plan(shape)
    plan.set_filter(sets[0][1], stream)
    n = len(sets)
    for i in range(3):
        plan.run_prepacked(sets[i % n][0], sets[i % n][2], alpha, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        plan.run_prepacked(sets[i % n][0], sets[i % n][2], alpha, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    st = plan.status(stream)
    plan.destroy()
    if st != 0:
        raise RuntimeError(f"device status {ext.status_string(st)} in prepacked runs")
    return e0.elapsed_time(e1) / steps


def bench_one_quick(wl, steps=30, warmup=5):
    """Device time per step and conv-kernel roofline fraction for one workload."""
    import torch
    import int8_implicit_gemm_gb300 as ext
    shape = wl.shape_tuple()
    P, Q = ext.i8c_output_size(shape)
    ops = ops_of(wl)
    xb, fb, yb = wl.N * wl.C * wl.H * wl.W, wl.K * wl.C * wl.R * wl.S, wl.N * wl.K * P * Q
    nsets = max(1, min(64, math.ceil(2 * L2_BYTES / (xb + fb + yb))))
    g = torch.Generator(device="cuda").manual_seed(wl.x_seed)
    sets = [(torch.randint(-128, 128, (xb,), dtype=torch.int8, device="cuda", generator=g),
             torch.randint(-128, 128, (fb,), dtype=torch.int8, device="cuda", generator=g),
             torch.empty(yb, dtype=torch.int8, device="cuda")) for _ in range(nsets)]
    plan = ext.Plan(shape)
    plan_k = ext.Plan(shape, timing_events=steps)
    s = torch.cuda.current_stream()
    for i in range(warmup):
        plan.run(*sets[i % nsets], wl.alpha, s)
        plan_k.run(*sets[i % nsets], wl.alpha, s)
    torch.cuda.synchronize()
    plan_k.kernel_time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for i in range(steps):
        plan.run(*sets[i % nsets], wl.alpha, s)
    e1.record(s)
    for i in range(steps):
        plan_k.run(*sets[i % nsets], wl.alpha, s)
    torch.cuda.synchronize()
    assert plan.status(s) == 0 and plan_k.status(s) == 0
    kms, kn = plan_k.kernel_time()
    peak, _ = tensor_peak()
    step_ms = e0.elapsed_time(e1) / steps
    pre = prepacked_burst(shape, sets, wl.alpha, steps, s) if plan.info["kernels_per_run"] != 1 else None
    kern, _ = kernel_duration(plan.info, step_ms, kms / max(1, kn), pre)
    plan.destroy()
    plan_k.destroy()
    return {"ms_per_step": round(step_ms, 6), "TOPS": round(ops / (step_ms * 1e-3) / 1e12, 2),
            "kernel_ms": round(kern, 6), "kernel_ms_bracketed": round(kms / max(1, kn), 6),
            "kernel_TOPS": round(ops / (kern * 1e-3) / 1e12, 2),
            "frac": round(ops / (kern * 1e-3) / 1e12 / peak, 4), "block_n": plan.info["block_n"],
            "kernel_variant": plan.info["kernel_variant"]}


def run_reference(args, wl, rank, world):
    """The CPU oracle as the reference arm: each step is a bounded sample
    (the first image of the workload), timed on the host cores."""
    if rank != 0:
        return None
    import oracle
    x = wl.activations_nchw()
    f = wl.filters_kcrs()
    orc = oracle.Oracle()
    P, Q = orc.out_size(wl.shape_tuple())
    shape = list(wl.shape_tuple())
    shape[0] = 1
    cores = os.cpu_count() or 1
    step_ops = 2 * wl.K * P * Q * wl.C * wl.R * wl.S
    for _ in range(args.warmup):
        orc.conv2d_fprop(x[:1], f, tuple(shape), wl.alpha, threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.conv2d_fprop(x[:1], f, tuple(shape), wl.alpha, threads=cores)
    dt = time.perf_counter() - t0
    v = step_ops * args.steps / dt / 1e12
    sample = f"1 of {wl.N} images per step, all {wl.K} output channels"
    return {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "s8 (int64 accumulation)",
            "data": "synthetic", "config": {"workload": wl.name, "shape": dict(zip(
                ["N", "C", "H", "W", "K", "R", "S", "pad_h", "pad_w", "stride_h", "stride_w", "dil_h", "dil_w"],
                wl.shape_tuple())), "P": P, "Q": Q, "alpha": wl.alpha},
            "cpu_baseline": {"value": round(v, 6), "unit": "TOPS", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 6), "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(synth.WORKLOADS_BY_NAME) + [synth.F32_WORKLOAD.name])
    ap.add_argument("--all", action="store_true", help="(default) also time every workload, device time only")
    ap.add_argument("--no-all", action="store_true", help="skip the per-workload device-time lines")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch the timed steps one by one")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of CPU oracle work for cpu_baseline")
    args = ap.parse_args()
    args.steps = max(1, args.steps)
    args.warmup = max(3, args.warmup)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.workload == synth.F32_WORKLOAD.name:
        if args.impl == "reference":
            res = run_f32_reference(args, rank, world)
            if res is not None:
                print(json.dumps(res), flush=True)
            return
        if world > 1:
            import torch
            torch.distributed.init_process_group("nccl")
        res = run_f32(args, rank, world)
        if rank == 0:
            print(json.dumps(res), flush=True)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
        return
    wl = synth.WORKLOADS_BY_NAME[args.workload]
    if args.impl == "reference":
        res = run_reference(args, wl, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, wl, rank, world)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
