"""Benchmark of the fused dequantization GEMM library on one GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-breakdown]

A step is one pass over the workload's calls with inputs resident in HBM.
The default workload is the INT8 weight-only decode sweep
(M in {1, 4, 16} x K = 4096 x N in {4096, 14336}); its value is the whole-job
HBM throughput on algorithmic bytes (packed weights + scales + activations +
outputs) in GB/s.  Every step reads a different replica of all inputs, and one
step's inputs are larger than the 129 MB L2, so no step starts with its
weights in L2.  Rank 0 prints one JSON line.

The `breakdown` key carries the other workloads (INT4 Llama-7B linears, the
MXFP4 quantize + GEMM and the FP8 GEMM) measured in the same run, each with
its own roofline.  `--impl reference` times the CPU oracle on a bounded
sample of the same workload instead (the oracle is the only place this
script runs oracle code besides the cpu_baseline leg).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

L2_BYTES = 129 * 1024 * 1024


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# Nominal dense tensor rates relative to bf16 (2.25 PF): fp8 4.5 PF, fp4 13.5 PF.
NOMINAL_RATIO = {"bf16": 1.0, "fp16": 1.0, "fp8": 2.0, "fp4": 6.0}


# ----------------------------------------------------------------- workloads
# Each workload builds its inputs on the device (R replicas) and returns a
# list of calls; a call is (name, fn(replica), alg_bytes, flops, dtype_for_peak).


def _wo_bytes(bits, M, K, N):
    wbytes = K * N // 2 if bits == 4 else K * N
    return wbytes + 2 * N + 2 * M * K + 2 * M * N


class WeightOnly:
    def __init__(self, wq, torch, bits, shapes, replicas, seed=0):
        self.wq, self.torch, self.bits, self.shapes = wq, torch, bits, shapes
        self.cases = []
        for (M, K, N) in shapes:
            c = workloads.w4a16_case(M, K, N, seed) if bits == 4 else workloads.w8a16_case(M, K, N, seed)
            self.cases.append(c)
        self.dev = []
        for _ in range(replicas):
            reps = []
            for c in self.cases:
                x = torch.from_numpy(c.x).cuda()
                w = torch.from_numpy(c.w).cuda()
                s = torch.from_numpy(c.scales).cuda()
                y = torch.empty((c.x.shape[0], c.w.shape[1]), dtype=torch.float16, device="cuda")
                reps.append((x, w, s, y))
            self.dev.append(reps)
        self.fn = wq.wq_gemm_w4a16 if bits == 4 else wq.wq_gemm_w8a16
        tag = "w4a16" if bits == 4 else "w8a16"
        self.calls = []
        for i, (M, K, N) in enumerate(shapes):
            self.calls.append((f"{tag}_{M}x{K}x{N}", i, _wo_bytes(bits, M, K, N), 2 * M * N * K))

    def run(self, r, i):
        x, w, s, y = self.dev[r][i]
        self.fn(x, w, s, y=y)

    def host_inputs(self):
        t = self.torch
        out = []
        for c in self.cases:
            out.append(tuple(t.from_numpy(a).pin_memory() for a in (c.x, c.w, c.scales)))
        return out

    def e2e_step(self, host, i, stream):
        t = self.torch
        hx, hw, hs = host[i]
        x = hx.to("cuda", non_blocking=True)
        w = hw.to("cuda", non_blocking=True)
        s = hs.to("cuda", non_blocking=True)
        y = self.fn(x, w, s)
        return y.to("cpu", non_blocking=True), sum(a.numel() * a.element_size() for a in (hx, hw, hs)), \
            y.numel() * y.element_size()

    def oracle_call(self, i):
        from oracle import wq_oracle as O

        c = self.cases[i]
        return (O.gemm_w4a16 if self.bits == 4 else O.gemm_w8a16)(c.x, c.w, c.scales)


def _sample_clocks():
    """Start nvidia-smi sampling clocks and throttle reasons every 200 ms."""
    try:
        q = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        return subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "200"],
                                stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
    except (OSError, ValueError):
        return None


def _pci_bus_id(torch, dev):
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


def _finish_clocks(proc, pci):
    if proc is None:
        return None
    proc.terminate()
    try:
        out, err = proc.communicate(timeout=5)
    except subprocess.TimeoutExpired:
        proc.kill()
        out, err = proc.communicate()
    rows = [[x.strip() for x in line.split(",")] for line in out.splitlines()]
    rows = [r for r in rows if len(r) >= 9]
    ids = {r[0] for r in rows}
    if pci is not None and any(i.upper().endswith(pci[-12:].upper()) for i in ids):
        rows = [r for r in rows if r[0].upper().endswith(pci[-12:].upper())]
    elif len(ids) > 1:
        return {"error": f"could not match the GPU among {sorted(ids)}"}
    sm, mx, reasons = [], None, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for f in rows:
        try:
            sm.append(float(f[1]))
            mx = float(f[2])
        except ValueError:
            continue
        for n, v in zip(names, f[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return {"error": (err or "no samples").strip()[:200]}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier_max(torch, value, ws):
    if ws == 1:
        return value
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _hold_stream(torch, seconds):
    """Keep the stream busy for about `seconds` (a device-side spin) so that the
    host can enqueue the whole timed region before the GPU reaches it: the
    events then measure device time only, not Python / launch latency."""
    torch.cuda._sleep(int(seconds * 2.2e9))  # cycles at or above the maximum SM clock


def time_workload(torch, wl, steps, warmup, replicas, ws):
    """Time `steps` passes over wl.calls; per-launch CUDA events on the launching stream."""
    stream = torch.cuda.current_stream()
    n_calls = len(wl.calls)
    t_host = time.perf_counter()
    for s in range(warmup):
        for (_, i, _, _) in wl.calls:
            wl.run(s % replicas, i)
    host_per_step = (time.perf_counter() - t_host) / max(1, warmup)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_calls)]
          for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    _hold_stream(torch, 2.0 * host_per_step * steps + 2e-3)
    t0.record(stream)
    for s in range(steps):
        for j, (_, i, _, _) in enumerate(wl.calls):
            ev[s][j][0].record(stream)
            wl.run(s % replicas, i)
            ev[s][j][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    total_ms = _barrier_max(torch, t0.elapsed_time(t1), ws)
    per_call = []
    for j, (name, _, nbytes, flops) in enumerate(wl.calls):
        ms = [ev[s][j][0].elapsed_time(ev[s][j][1]) for s in range(steps)]
        per_call.append({"call": name, "ms": statistics.mean(ms), "bytes": nbytes, "flops": flops})
    return total_ms, per_call


def roofline_for(call, peaks, bound, dtype="fp16", traffic=None):
    if bound == "hbm":
        achieved = call["bytes"] / (call["ms"] * 1e-3) / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
    else:
        achieved = call["flops"] / (call["ms"] * 1e-3) / 1e12
        peak, unit = peaks["bf16_tflops"] * NOMINAL_RATIO[dtype], "TFLOP/s"
    return {"bound": bound, "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic, "kernel_call": call["call"],
            "peak_source": peaks["source"] + (f" (bf16 x {NOMINAL_RATIO[dtype]} nominal ratio)" if bound == "tensor"
                                              and dtype != "bf16" else "")}


def run_ours(args):
    import torch

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    import bit_quantized_gemm_dequant_gb300 as wq

    peaks = load_peaks()
    replicas = 3
    spec = workloads.WORKLOADS[args.workload]
    bits = 4 if spec["op"] == "w4a16" else 8
    wl = WeightOnly(wq, torch, bits, spec["shapes"], replicas)
    step_bytes = sum(c[2] for c in wl.calls)

    clock_proc = _sample_clocks() if rank == 0 else None
    total_ms, per_call = time_workload(torch, wl, args.steps, args.warmup, replicas, ws)
    clocks = _finish_clocks(clock_proc, _pci_bus_id(torch, local)) if rank == 0 else None

    value = ws * step_bytes * args.steps / (total_ms * 1e-3) / 1e9
    dominant = max(per_call, key=lambda c: c["ms"])
    roof = roofline_for(dominant, peaks, "hbm", traffic=args.traffic)

    # End to end through the public API with pinned host buffers: H2D of the
    # step's inputs, the call, D2H of the result, every step.
    host = wl.host_inputs()
    stream = torch.cuda.current_stream()
    for _ in range(2):
        for (_, i, _, _) in wl.calls:
            wl.e2e_step(host, i, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, min(args.steps, 10))
    h2d = d2h = 0
    e0.record(stream)
    for _ in range(e2e_steps):
        h2d = d2h = 0
        for (_, i, _, _) in wl.calls:
            _, bi, bo = wl.e2e_step(host, i, stream)
            h2d += bi
            d2h += bo
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = _barrier_max(torch, e0.elapsed_time(e1), ws)
    e2e_val = ws * step_bytes * e2e_steps / (e2e_ms * 1e-3) / 1e9

    breakdown = []
    if not args.no_breakdown and rank == 0:
        breakdown = run_breakdown(torch, wq, peaks, args)

    cpu = cpu_baseline(wl, step_bytes, budget_s=args.cpu_budget) if (rank == 0 and ws == 1) else None

    if rank == 0:
        line = {
            "metric": "W4A16/W8A16 GEMV HBM GB/s (% peak); MXFP4/FP8 GEMM TFLOPS (% peak)",
            "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8/int4 weights x fp16 activations, fp32 accumulate", "data": "synthetic",
            "config": {"workload": f"{args.workload}: " + ", ".join(f"{m}x{k}x{n}" for (m, k, n) in spec["shapes"]),
                       "shapes_MxKxN": spec["shapes"], "seed": 0, "replicas": replicas,
                       "l2": f"inputs rotate over {replicas} replicas; one step reads "
                             f"{step_bytes / 1e6:.0f} MB (> {L2_BYTES / 1e6:.0f} MB L2)",
                       "parallelism": f"replicas x{ws}"},
            "roofline": roof,
            "per_call": [{**c, "GBps": round(c["bytes"] / (c["ms"] * 1e-3) / 1e9, 1)} for c in per_call],
            "e2e": {"value": round(e2e_val, 3), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": len(wl.calls) * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "breakdown": breakdown,
        }
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()


def time_calls(torch, calls, steps, warmup, flush_bytes=2 * L2_BYTES):
    """Per-call CUDA-event times (ms) on the launching stream.  Before every
    call an L2-sized buffer is overwritten (outside the events), so no call
    starts with its operands in L2."""
    stream = torch.cuda.current_stream()
    scratch = torch.empty(flush_bytes // 4, dtype=torch.float32, device="cuda")
    for _ in range(warmup):
        for c in calls:
            c["run"]()
    torch.cuda.synchronize()
    ev = {c["call"]: [] for c in calls}
    _hold_stream(torch, 60e-6 * steps * len(calls) + 2e-3)
    for _ in range(steps):
        for c in calls:
            scratch.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            c["run"]()
            e1.record(stream)
            ev[c["call"]].append((e0, e1))
    torch.cuda.synchronize()
    out = []
    for c in calls:
        ms = statistics.median(a.elapsed_time(b) for a, b in ev[c["call"]])
        out.append({"call": c["call"], "ms": ms, "bytes": c["bytes"], "flops": c["flops"]})
    del scratch
    return out


def run_breakdown(torch, wq, peaks, args):
    """Other workloads, each timed over a few steps with its own roofline."""
    out = []
    steps, warm = 5, 3

    spec = workloads.WORKLOADS["w4a16_llama7b"]
    wl = WeightOnly(wq, torch, 4, spec["shapes"], 1)
    calls = [{"call": name, "run": (lambda i=i: wl.run(0, i)), "bytes": nb, "flops": fl}
             for (name, i, nb, fl) in wl.calls]
    for c in time_calls(torch, calls, steps, warm):
        M = int(c["call"].split("_")[1].split("x")[0])
        bound = "hbm" if M <= 64 else "tensor"
        out.append({"workload": "w4a16_llama7b", **c, "roofline": roofline_for(c, peaks, bound, "fp16")})
    del wl, calls
    torch.cuda.empty_cache()

    # MXFP4: quantize both fp32 operands on the device, then the GEMM.
    K = N = 8192
    w_src = torch.from_numpy(workloads.mx_source(N, K, seed=0, stream=1)).cuda()
    wd, ws = wq.mx_quantize_fp4(w_src)
    calls = [{"call": f"mx_quantize_{N}x{K}", "run": (lambda: wq.mx_quantize_fp4(w_src, wd, ws)),
              "bytes": N * K * 4 + N * K // 2 + N * K // 32, "flops": 0, "bound": "hbm"}]
    keep = []
    for M in (128, 2048, 8192):
        a_src = torch.from_numpy(workloads.mx_source(M, K, seed=0, stream=0)).cuda()
        ad, asc = wq.mx_quantize_fp4(a_src)
        c_out = torch.empty((M, N), dtype=torch.float32, device="cuda")
        keep.append((a_src, ad, asc, c_out))
        calls.append({"call": f"mx_gemm_{M}x{K}x{N}",
                      "run": (lambda ad=ad, asc=asc, c_out=c_out: wq.mx_gemm_fp4(ad, asc, wd, ws, c=c_out)),
                      "bytes": (M + N) * (K // 2 + K // 32) + 4 * M * N, "flops": 2 * M * N * K,
                      "bound": "hbm" if M <= 128 else "tensor"})
    for c, spec_c in zip(time_calls(torch, calls, steps, warm), calls):
        out.append({"workload": "mxfp4", **c, "roofline": roofline_for(c, peaks, spec_c["bound"], "fp4")})
    del keep, calls, w_src, wd, ws
    torch.cuda.empty_cache()

    calls, keep = [], []
    for (M, K, N) in workloads.WORKLOADS["fp8"]["shapes"]:
        case = workloads.fp8_case(M, K, N, seed=0)
        a = torch.from_numpy(case.a8).cuda()
        b = torch.from_numpy(case.b8).cuda()
        cc = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        keep.append((a, b, cc))
        calls.append({"call": f"fp8_{M}x{K}x{N}",
                      "run": (lambda a=a, b=b, cc=cc, sa=case.scale_a, sb=case.scale_b: wq.fp8_gemm(a, b, sa, sb, c=cc)),
                      "bytes": M * K + K * N + 2 * M * N, "flops": 2 * M * N * K,
                      "bound": "hbm" if M <= 16 else "tensor"})
    for c, spec_c in zip(time_calls(torch, calls, steps, warm), calls):
        out.append({"workload": "fp8", **c, "roofline": roofline_for(c, peaks, spec_c["bound"], "fp8")})
    del keep, calls
    torch.cuda.empty_cache()
    return out


def cpu_baseline(wl, step_bytes, budget_s=15.0):
    """The oracle as it stands on this host, over whole steps until ~budget_s."""
    t0 = time.perf_counter()
    n = 0
    while True:
        for (_, i, _, _) in wl.calls:
            wl.oracle_call(i)
        n += 1
        if time.perf_counter() - t0 >= budget_s or n >= 20:
            break
    dt = time.perf_counter() - t0
    return {"value": round(step_bytes * n / dt / 1e9, 4), "unit": "GB/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{n} full step(s) of the workload on the CPU oracle (numpy float64, BLAS threads = cores)"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    spec = workloads.WORKLOADS[args.workload]
    from oracle import wq_oracle as O

    bits = 4 if spec["op"] == "w4a16" else 8
    cases = [(workloads.w4a16_case if bits == 4 else workloads.w8a16_case)(M, K, N, 0) for (M, K, N) in spec["shapes"]]
    fn = O.gemm_w4a16 if bits == 4 else O.gemm_w8a16
    # A bounded sample of the workload per step: the first `per_step` calls.
    per_step = 2 if args.steps + args.warmup > 4 else len(cases)
    sample_bytes = sum(_wo_bytes(bits, *spec["shapes"][i]) for i in range(per_step))
    for _ in range(args.warmup):
        for c in cases[:per_step]:
            fn(c.x, c.w, c.scales)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for c in cases[:per_step]:
            fn(c.x, c.w, c.scales)
    dt = time.perf_counter() - t0
    value = sample_bytes * args.steps / dt / 1e9
    sample = f"first {per_step} call(s) of the workload per step: " + ", ".join(
        f"{m}x{k}x{n}" for (m, k, n) in spec["shapes"][:per_step])
    print(json.dumps({
        "impl": "reference", "metric": "W4A16/W8A16 GEMV HBM GB/s (% peak); MXFP4/FP8 GEMM TFLOPS (% peak)",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: " + ", ".join(f"{m}x{k}x{n}" for (m, k, n) in spec["shapes"]),
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="w8a16_decode", choices=["w8a16_decode", "w4a16_llama7b", "w4a16_tiny"])
    ap.add_argument("--no-breakdown", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch of the dominant kernel from an ncu capture of this build")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
