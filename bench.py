"""Benchmark of the fused dequantization GEMM library on one GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--only SUBSTRING] [--no-breakdown] [--no-e2e]

A step is one pass over the workload's calls with inputs resident in HBM.
The default workload is the INT8 weight-only decode sweep
(M in {1, 4, 16} x K = 4096 x N in {4096, 14336}); its value is the whole-job
HBM throughput on algorithmic bytes (packed weights + scales + activations +
outputs) in GB/s.  Steps rotate over replicas of all inputs and one step reads
more than the 129 MB L2, so no call starts with its weights in L2.

Before the timed region the stream is held by a device-side spin long enough
for the host to enqueue every timed launch, so CUDA events measure device time
and not Python / launch latency.  The K steps run back to back between two
events, with nothing recorded between calls, so consecutive kernels overlap as
they do in a real call sequence (the skinny kernels are launched as
programmatic dependents).  Per-call kernel times, and the roofline of the
dominant kernel, come from a second pass in which each call sits between its
own pair of events.  Rank 0 prints one JSON line.

`breakdown` carries the other workloads (INT4 Llama-7B linears, MXFP4 quantize
+ GEMM, FP8 GEMM), each call timed after an L2 flush, with its own roofline.
`--impl reference` times the CPU oracle on a bounded sample of the workload;
the oracle runs nowhere else in this script except the cpu_baseline leg.
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
METRIC = "W4A16/W8A16 GEMV HBM GB/s (% peak); MXFP4/FP8 GEMM TFLOPS (% peak)"
# Nominal dense tensor rates relative to bf16 (2.25 PF): fp8 4.5 PF, fp4 13.5 PF.
NOMINAL_RATIO = {"bf16": 1.0, "fp16": 1.0, "fp8": 2.0, "fp4": 6.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------- workloads
# A workload owns device inputs (several replicas) and a list of calls.  Each
# call is a dict: name, index, bytes, flops, bound ("hbm"/"tensor"), dtype
# (for the tensor peak).  The main line's unit is GB/s when every call is
# HBM-bound, TFLOP/s otherwise.


def _wo_bytes(bits, M, K, N, group_n=1, asym=False):
    groups = -(-N // group_n)
    return (K * N // 2 if bits == 4 else K * N) + 2 * groups + (groups if asym else 0) + 2 * M * K + 2 * M * N


def _wo_tag(bits, group_n=None, asym=False):
    """Call-name prefix of a weight-only workload, shared by both bench arms."""
    return ("w4a16" if bits == 4 else "w8a16") + (f"_g{group_n}" + ("zp" if asym else "") if group_n else "")


class WeightOnly:
    """Weight-only GEMMs; with ``group_n`` the column-grouped entry points
    (one scale, and with ``asym`` one zero point, per group of columns)."""

    def __init__(self, torch, wq, bits, shapes, replicas, seed=0, group_n=None, asym=False, batched=False):
        self.torch, self.bits, self.group_n, self.asym, self.batched = torch, bits, group_n, asym, batched
        self.shapes = shapes
        if group_n:
            self.cases = [workloads.grouped_case(bits, M, K, N, group_n, asym, seed) for (M, K, N) in shapes]
            self.fn = None if wq is None else (wq.wq_gemm_w4a16_grouped if bits == 4 else wq.wq_gemm_w8a16_grouped)
        else:
            self.cases = [(workloads.w4a16_case if bits == 4 else workloads.w8a16_case)(M, K, N, seed)
                          for (M, K, N) in shapes]
            self.fn = None if wq is None else (wq.wq_gemm_w4a16 if bits == 4 else wq.wq_gemm_w8a16)
        self.dev = []
        for _ in range(replicas if wq is not None else 0):  # wq None: host-side cases only (oracle arm)
            reps = []
            for c in self.cases:
                z = getattr(c, "zeros", None)
                reps.append((torch.from_numpy(c.x).cuda(), torch.from_numpy(c.w).cuda(),
                             torch.from_numpy(c.scales).cuda(),
                             torch.empty((c.x.shape[0], c.w.shape[1]), dtype=torch.float16, device="cuda"),
                             torch.from_numpy(z).cuda() if z is not None else None))
            self.dev.append(reps)
        # One zero-filled workspace serves every call: they run one after the
        # other on one stream and each leaves it zero-filled.
        tag = _wo_tag(bits, group_n, asym)
        self.calls = []
        need = 0
        if wq is not None:
            op = wq.WQ_OP_W4A16 if bits == 4 else wq.WQ_OP_W8A16
            need = max(wq.wq_workspace_size(op, M, N, K) for (M, K, N) in shapes)
        if batched:
            if wq is not None:
                self.batch_fn = wq.wq_gemm_w4a16_batched if bits == 4 else wq.wq_gemm_w8a16_batched
                probs = (wq.WqProblem * len(shapes))(*[
                    wq.WqProblem(M, N, K, 16, K, 16, N, 16, 1, 16, N) for (M, K, N) in shapes])
                need = max(need, int(wq.lib.wq_batched_workspace_size(op, len(shapes), probs)))
            self.calls.append({"call": f"{tag}_batched_" + "+".join(f"{M}x{K}x{N}" for (M, K, N) in shapes),
                               "index": -1, "bytes": sum(_wo_bytes(bits, M, K, N) for (M, K, N) in shapes),
                               "flops": sum(2 * M * N * K for (M, K, N) in shapes), "bound": "hbm",
                               "dtype": "fp16", "problems": len(shapes)})
        else:
            for i, (M, K, N) in enumerate(shapes):
                self.calls.append({"call": f"{tag}_{M}x{K}x{N}", "index": i,
                                   "bytes": _wo_bytes(bits, M, K, N, group_n or 1, asym),
                                   "flops": 2 * M * N * K, "bound": "hbm" if M <= 64 else "tensor",
                                   "dtype": "fp16"})
        if wq is not None:
            self.ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")

    def _call(self, x, w, s, z, y=None):
        if self.group_n:
            return self.fn(x, w, s, z, self.group_n, y=y, workspace=self.ws)
        return self.fn(x, w, s, y=y, workspace=self.ws)

    def run(self, r, i):
        if i < 0:  # the whole batch in one call
            reps = self.dev[r]
            self.batch_fn([d[0] for d in reps], [d[1] for d in reps], [d[2] for d in reps],
                          ys=[d[3] for d in reps], workspace=self.ws)
            return
        x, w, s, y, z = self.dev[r][i]
        self._call(x, w, s, z, y)

    def host_inputs(self):
        out = []
        for c in self.cases:
            arrs = [c.x, c.w, c.scales] + ([c.zeros] if getattr(c, "zeros", None) is not None else [])
            out.append(tuple(self.torch.from_numpy(a).pin_memory() for a in arrs))
        return out

    def e2e_call(self, host, i):
        if i < 0:  # the whole batch: every problem's inputs in, every output out
            devs = [[a.to("cuda", non_blocking=True) for a in h] for h in host]
            ys = self.batch_fn([d[0] for d in devs], [d[1] for d in devs], [d[2] for d in devs], workspace=self.ws)
            for y in ys:
                y.to("cpu", non_blocking=True)
            return (sum(a.numel() * a.element_size() for h in host for a in h),
                    sum(y.numel() * y.element_size() for y in ys))
        dev = [a.to("cuda", non_blocking=True) for a in host[i]]
        y = self._call(dev[0], dev[1], dev[2], dev[3] if len(dev) > 3 else None)
        y.to("cpu", non_blocking=True)
        return sum(a.numel() * a.element_size() for a in host[i]), y.numel() * y.element_size()

    def oracle_call(self, i, cols=None):
        """Run the oracle on call i (or, i < 0, on every problem of the batch);
        with `cols`, on the first `cols` output columns of each call only.
        Returns the bytes and flops of the work done and what the sample was."""
        from oracle import wq_oracle as O

        if i < 0:  # the whole batch
            b = f = 0
            for j in range(len(self.cases)):
                bj, fj, _ = self.oracle_call(j, cols)
                b, f = b + bj, f + fj
            return b, f, "every problem of the batch" + (f", first {cols} columns of each" if cols else "")
        c = self.cases[i]
        M, K, N = self.shapes[i]
        n = N if cols is None else min(cols, N)
        w = c.w[:, :n]
        if self.group_n:
            g = -(-n // c.group_n)
            z = c.zeros[:g] if c.zeros is not None else None
            (O.gemm_w4a16_grouped if self.bits == 4 else O.gemm_w8a16_grouped)(c.x, w, c.scales[:g], z, c.group_n)
        else:
            (O.gemm_w4a16 if self.bits == 4 else O.gemm_w8a16)(c.x, w, c.scales[:n])
        desc = "whole call" if n == N else f"first {n} of {N} columns (extrapolated)"
        return _wo_bytes(self.bits, M, K, n, self.group_n or 1, self.asym), 2 * M * n * K, desc


class MxFp4:
    """Per M: quantize A [M, K] and W [N, K] on the device, then C = A W^T.
    W's block scales go into the tensor cores' layout once per step, as part
    of preparing W (the quantize-W call); each GEMM call rearranges A's
    scales, then runs mx_gemm_fp4_tc.  fused_a: A is quantized inside the
    GEMM launch instead (mx_gemm_fp4_qa), one call per M."""

    def __init__(self, torch, wq, shapes, replicas, seed=0, fused_a=False):
        self.torch, self.wq = torch, wq
        self.fused_a = fused_a
        K, N = shapes[0][1], shapes[0][2]
        self.K, self.N = K, N
        self.w_src = workloads.mx_source(N, K, seed=seed, stream=1)
        self.a_srcs = [workloads.mx_source(M, K, seed=seed, stream=0) for (M, _, _) in shapes]
        self._oracle_ops = None
        self.dev = []
        for _ in range(replicas if wq is not None else 0):  # wq None: host-side sources only (oracle arm)
            w = torch.from_numpy(self.w_src).cuda()
            wd, wsc = wq.mx_quantize_fp4(w)
            reps = {"w": (w, wd, wsc, wq.fp4_scales_tc(wsc, K)), "a": []}
            for a_src in self.a_srcs:
                a = torch.from_numpy(a_src).cuda()
                ad, asc = wq.mx_quantize_fp4(a)
                c = torch.empty((a.shape[0], N), dtype=torch.float32, device="cuda")
                reps["a"].append((a, ad, asc, wq.fp4_scales_tc(asc, K), c))
            self.dev.append(reps)
        self.calls = [{"call": f"mx_quantize_{N}x{K}", "index": ("qw", 0), "launches": 2,
                       "bytes": N * K * 4 + N * K // 2 + N * K // 32, "flops": 0, "bound": "hbm", "dtype": "fp4"}]
        for i, (M, _, _) in enumerate(shapes):
            if fused_a:  # one launch: A read as FP32, W, C written
                self.calls.append({"call": f"mx_gemm_qa_{M}x{K}x{N}", "index": ("gq", i),
                                   "bytes": M * K * 4 + N * (K // 2 + K // 32) + 4 * M * N, "flops": 2 * M * N * K,
                                   "bound": "hbm" if M <= 128 else "tensor", "dtype": "fp4"})
                continue
            self.calls.append({"call": f"mx_quantize_{M}x{K}", "index": ("qa", i),
                               "bytes": M * K * 4 + M * K // 2 + M * K // 32, "flops": 0, "bound": "hbm",
                               "dtype": "fp4"})
            self.calls.append({"call": f"mx_gemm_{M}x{K}x{N}", "index": ("g", i), "launches": 2,
                               "bytes": (M + N) * (K // 2 + K // 32) + 4 * M * N, "flops": 2 * M * N * K,
                               "bound": "hbm" if M <= 128 else "tensor", "dtype": "fp4"})

    # Oracle samples: quantize 64 rows; GEMM 4 rows of A against 256 rows of W.
    Q_ROWS, G_ROWS_A, G_ROWS_W = 64, 4, 256

    def oracle_call(self, idx):
        from oracle import wq_oracle as O

        kind, i = idx
        K, N = self.K, self.N
        if kind in ("qw", "qa"):
            src = self.w_src if kind == "qw" else self.a_srcs[i]
            r = min(self.Q_ROWS, src.shape[0])
            O.mx_quantize_fp4(src[:r])
            return r * K * 4 + r * K // 2 + r * K // 32, 0, f"first {r} of {src.shape[0]} rows (extrapolated)"
        if self._oracle_ops is None:  # quantized row subsets, made once (outside the timed sample)
            self._oracle_ops = (O.mx_quantize_fp4(self.w_src[:self.G_ROWS_W]),
                                [O.mx_quantize_fp4(a[:self.G_ROWS_A]) for a in self.a_srcs])
        (wd, ws), a_ops = self._oracle_ops
        M = self.a_srcs[i].shape[0]
        if kind == "gq":  # A's rows quantized inside the timed sample, as the fused call does
            ad, asc = O.mx_quantize_fp4(self.a_srcs[i][:self.G_ROWS_A])
            O.mx_gemm_fp4(ad, asc, wd, ws)
            m, n = ad.shape[0], wd.shape[0]
            return (m * K * 4 + n * (K // 2 + K // 32) + 4 * m * n, 2 * m * n * K,
                    f"{m} of {M} rows of A (quantized) x {n} of {N} rows of W (extrapolated)")
        ad, asc = a_ops[i]
        O.mx_gemm_fp4(ad, asc, wd, ws)
        m, n = ad.shape[0], wd.shape[0]
        return ((m + n) * (K // 2 + K // 32) + 4 * m * n, 2 * m * n * K,
                f"{m} of {M} rows of A x {n} of {N} rows of W (extrapolated)")

    def run(self, r, idx):
        kind, i = idx
        d = self.dev[r]
        w, wd, wsc, wsc_tc = d["w"]
        if kind == "qw":
            self.wq.mx_quantize_fp4(w, wd, wsc)
            self.wq.fp4_scales_tc(wsc, self.K, out=wsc_tc)
            return
        a, ad, asc, asc_tc, c = d["a"][i]
        if kind == "gq":
            self.wq.mx_gemm_fp4_qa(a, wd, wsc_tc, c=c)
        elif kind == "qa":
            self.wq.mx_quantize_fp4(a, ad, asc)
        else:
            self.wq.fp4_scales_tc(asc, self.K, out=asc_tc)
            self.wq.mx_gemm_fp4_tc(ad, asc_tc, wd, wsc_tc, c=c)


class NvFp4:
    """Per M: quantize A [M, K] and W [N, K] to NVFP4 on the device, then C = A W^T
    (block scales rearranged as in MxFp4)."""

    def __init__(self, torch, wq, shapes, replicas, seed=0):
        self.torch, self.wq = torch, wq
        K, N = shapes[0][1], shapes[0][2]
        self.K, self.N = K, N
        self.w_src = workloads.mx_source(N, K, seed=seed, stream=1)
        self.a_srcs = [workloads.mx_source(M, K, seed=seed, stream=0) for (M, _, _) in shapes]
        self._oracle_ops = None
        self.dev = []
        for _ in range(replicas if wq is not None else 0):  # wq None: host-side sources only (oracle arm)
            w = torch.from_numpy(self.w_src).cuda()
            wd, wsc, gw = wq.nv_quantize_fp4(w)
            nv = wq.WQ_FP4_NV
            reps = {"w": (w, wd, wsc, gw, wq.fp4_scales_tc(wsc, K, nv)), "a": []}
            for a_src in self.a_srcs:
                a = torch.from_numpy(a_src).cuda()
                ad, asc, ga = wq.nv_quantize_fp4(a)
                c = torch.empty((a.shape[0], N), dtype=torch.float32, device="cuda")
                reps["a"].append((a, ad, asc, ga, wq.fp4_scales_tc(asc, K, nv), c))
            self.dev.append(reps)

        def qbytes(r):  # the source twice (amax, then codes), codes and E4M3 scales out
            return r * K * 8 + r * K // 2 + r * K // 16

        self.calls = [{"call": f"nv_quantize_{N}x{K}", "index": ("qw", 0), "launches": 4, "bytes": qbytes(N),
                       "flops": 0, "bound": "hbm", "dtype": "fp4"}]
        for i, (M, _, _) in enumerate(shapes):
            self.calls.append({"call": f"nv_quantize_{M}x{K}", "index": ("qa", i), "launches": 3,
                               "bytes": qbytes(M), "flops": 0, "bound": "hbm", "dtype": "fp4"})
            self.calls.append({"call": f"nv_gemm_{M}x{K}x{N}", "index": ("g", i), "launches": 2,
                               "bytes": (M + N) * (K // 2 + K // 16) + 4 * M * N, "flops": 2 * M * N * K,
                               "bound": "hbm" if M <= 128 else "tensor", "dtype": "fp4"})

    Q_ROWS, G_ROWS_A, G_ROWS_W = 64, 4, 256

    def oracle_call(self, idx):
        from oracle import wq_oracle as O

        kind, i = idx
        K, N = self.K, self.N
        if kind in ("qw", "qa"):
            src = self.w_src if kind == "qw" else self.a_srcs[i]
            r = min(self.Q_ROWS, src.shape[0])
            O.nv_quantize_fp4(src[:r])
            return r * K * 8 + r * K // 2 + r * K // 16, 0, f"first {r} of {src.shape[0]} rows (extrapolated)"
        if self._oracle_ops is None:
            self._oracle_ops = (O.nv_quantize_fp4(self.w_src[:self.G_ROWS_W]),
                                [O.nv_quantize_fp4(a[:self.G_ROWS_A]) for a in self.a_srcs])
        (wd, ws, gw), a_ops = self._oracle_ops
        ad, asc, ga = a_ops[i]
        O.nv_gemm_fp4(ad, asc, ga, wd, ws, gw)
        m, n = ad.shape[0], wd.shape[0]
        M = self.a_srcs[i].shape[0]
        return ((m + n) * (K // 2 + K // 16) + 4 * m * n, 2 * m * n * K,
                f"{m} of {M} rows of A x {n} of {N} rows of W (extrapolated)")

    def run(self, r, idx):
        kind, i = idx
        d = self.dev[r]
        w, wd, wsc, gw, wsc_tc = d["w"]
        nv = self.wq.WQ_FP4_NV
        if kind == "qw":
            self.wq.nv_quantize_fp4(w, wd, wsc, gw)
            self.wq.fp4_scales_tc(wsc, self.K, nv, out=wsc_tc)
            return
        a, ad, asc, ga, asc_tc, c = d["a"][i]
        if kind == "qa":
            self.wq.nv_quantize_fp4(a, ad, asc, ga)
        else:
            self.wq.fp4_scales_tc(asc, self.K, nv, out=asc_tc)
            self.wq.nv_gemm_fp4_tc(ad, asc_tc, ga, wd, wsc_tc, gw, c=c)


class Fp8:
    def __init__(self, torch, wq, shapes, replicas, seed=0):
        self.torch, self.wq = torch, wq
        self.cases = [workloads.fp8_case(M, K, N, seed) for (M, K, N) in shapes]
        self.shapes = shapes
        self.dev = []
        for _ in range(replicas if wq is not None else 0):  # wq None: host-side cases only (oracle arm)
            self.dev.append([(torch.from_numpy(c.a8).cuda(), torch.from_numpy(c.b8).cuda(),
                              torch.empty((c.a8.shape[0], c.b8.shape[1]), dtype=torch.bfloat16, device="cuda"))
                             for c in self.cases])
        self.calls = [{"call": f"fp8_{M}x{K}x{N}", "index": i, "bytes": M * K + K * N + 2 * M * N,
                       "flops": 2 * M * N * K, "bound": "hbm" if M <= 16 else "tensor", "dtype": "fp8"}
                      for i, (M, K, N) in enumerate(shapes)]

    # Oracle sample: 8 rows of A against the first 1024 columns of B.
    ROWS, COLS = 8, 1024

    def oracle_call(self, i):
        from oracle import wq_oracle as O

        c = self.cases[i]
        M, K, N = self.shapes[i]
        m, n = min(self.ROWS, M), min(self.COLS, N)
        O.fp8_gemm(c.a8[:m], c.b8[:, :n], c.scale_a, c.scale_b)
        return m * K + K * n + 2 * m * n, 2 * m * n * K, f"{m} of {M} rows x {n} of {N} columns (extrapolated)"

    def run(self, r, i):
        a, b, c = self.dev[r][i]
        self.wq.fp8_gemm(a, b, self.cases[i].scale_a, self.cases[i].scale_b, c=c)


def make_workload(torch, wq, name, replicas, only=None):
    spec = workloads.WORKLOADS[name]
    shapes = spec["shapes"]
    if spec["op"] in ("w4a16", "w8a16"):
        wl = WeightOnly(torch, wq, 4 if spec["op"] == "w4a16" else 8, shapes, replicas,
                        group_n=spec.get("group_n"), asym=spec.get("asym", False),
                        batched=spec.get("batched", False))
    elif spec["op"] == "mxfp4":
        wl = MxFp4(torch, wq, shapes, replicas, fused_a=spec.get("fused_a", False))
    elif spec["op"] == "nvfp4":
        wl = NvFp4(torch, wq, shapes, replicas)
    else:
        wl = Fp8(torch, wq, shapes, replicas)
    if only:
        wl.calls = [c for c in wl.calls if only in c["call"]]
        if not wl.calls:
            raise SystemExit(f"--only {only!r} matches no call of {name}")
    return wl


# Workloads reported in `breakdown` besides the headline one.  mxfp4_qa (A
# quantized inside the GEMM's cooperative launch) is timed on request only
# (--workload mxfp4_qa): the default command is also the one whose launches
# are listed under a profiler, and that kernel is kept out of profiler runs.
BREAKDOWN = ("w8a16_decode_batched", "w4a16_decode", "w4a16_decode_batched", "w4a16_llama7b",
             "w8a16_grouped_decode", "mxfp4", "nvfp4", "fp8")


def replicas_for(step_bytes):
    """Enough replicas that the inputs touched between two uses of one replica exceed 2x L2."""
    return max(2, min(8, int(np.ceil(2 * L2_BYTES / max(1, step_bytes))) + 1))


# ------------------------------------------------------------------- timing


def _hold_stream(torch, seconds):
    """Keep the stream busy for about `seconds` with a device-side spin, so that
    the host enqueues the whole timed region before the GPU reaches it: the
    events then measure device time, not Python / launch latency."""
    seconds = min(seconds, 0.05)  # under a profiler host launches are slow: cap the hold
    torch.cuda._sleep(int(seconds * 2.2e9))  # cycles at (or above) the maximum SM clock


def _barrier_max(torch, value, ws):
    """The largest of the ranks' values (the slowest rank's time); every rank
    gets it.  The reduction tensor lives where the process group's backend
    wants it: on the GPU for NCCL, on the host for gloo."""
    if ws == 1:
        return value
    import torch.distributed as dist

    device = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _summary(c, ms):
    return {k: c[k] for k in ("call", "bytes", "flops", "bound", "dtype")} | {"ms": ms}


def time_steps(torch, wl, steps, warmup, replicas, ws):
    """K steps over wl.calls, back to back on one stream, between two CUDA
    events (nothing recorded between the calls, so consecutive kernels may
    overlap the way they do in a real sequence of calls)."""
    stream = torch.cuda.current_stream()
    t_host = time.perf_counter()
    for s in range(warmup):
        for c in wl.calls:
            wl.run(s % replicas, c["index"])
    host_per_step = (time.perf_counter() - t_host) / max(1, warmup)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    _hold_stream(torch, 2.0 * host_per_step * steps + 2e-3)
    t0.record(stream)
    for s in range(steps):
        for c in wl.calls:
            wl.run(s % replicas, c["index"])
    t1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    return _barrier_max(torch, t0.elapsed_time(t1), ws)


def time_each_call(torch, wl, steps, replicas):
    """Per-call device time: the same K steps again, each call between its own
    pair of CUDA events on the launching stream (the events serialise the
    calls, so this is each kernel's duration alone)."""
    stream = torch.cuda.current_stream()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in wl.calls]
          for _ in range(steps)]
    torch.cuda.synchronize()
    t_host = time.perf_counter()
    for c in wl.calls:
        wl.run(0, c["index"])
    host_per_step = time.perf_counter() - t_host
    torch.cuda.synchronize()
    _hold_stream(torch, 2.0 * host_per_step * steps + 2e-3)
    for s in range(steps):
        for j, c in enumerate(wl.calls):
            ev[s][j][0].record(stream)
            wl.run(s % replicas, c["index"])
            ev[s][j][1].record(stream)
    torch.cuda.synchronize()
    return [_summary(c, statistics.mean(ev[s][j][0].elapsed_time(ev[s][j][1]) for s in range(steps)))
            for j, c in enumerate(wl.calls)]


def time_calls_flushed(torch, wl, steps, warmup):
    """Per-call device times (median ms), each call preceded by an L2 flush
    (a 2 x L2 buffer overwritten outside the events)."""
    stream = torch.cuda.current_stream()
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    for _ in range(warmup):
        for c in wl.calls:
            wl.run(0, c["index"])
    torch.cuda.synchronize()
    ev = {c["call"]: [] for c in wl.calls}
    _hold_stream(torch, 80e-6 * steps * len(wl.calls) + 2e-3)
    for _ in range(steps):
        for c in wl.calls:
            scratch.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            wl.run(0, c["index"])
            e1.record(stream)
            ev[c["call"]].append((e0, e1))
    torch.cuda.synchronize()
    out = [_summary(c, statistics.median(a.elapsed_time(b) for a, b in ev[c["call"]])) for c in wl.calls]
    del scratch
    return out


# DRAM bytes (read + write) of one launch, from one ncu capture of the call's
# kernel (the profile named beside it).  A figure is used only while the
# kernel's code is the code it was taken on (same SHA-256 of the source with
# comments removed, code_sha256); else the roofline reports traffic null.
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# a call, from an ncu capture of that call, with the SHA-256 of the code of
# every source its kernel is compiled from (code_sha256 of each, in order).
# A figure is reported only while those sources still hold that code.
SKINNY_SOURCES = ("bit_quantized_gemm_dequant_gb300/csrc/wo_skinny.cu",
                  "bit_quantized_gemm_dequant_gb300/csrc/skinny_common.cuh",
                  "bit_quantized_gemm_dequant_gb300/csrc/tc_common.cuh",
                  "bit_quantized_gemm_dequant_gb300/csrc/wq_internal.h")
BATCHED_SOURCES = ("bit_quantized_gemm_dequant_gb300/csrc/wo_batched.cu",
                   "bit_quantized_gemm_dequant_gb300/csrc/skinny_common.cuh",
                   "bit_quantized_gemm_dequant_gb300/csrc/tc_common.cuh",
                   "bit_quantized_gemm_dequant_gb300/csrc/wq_internal.h")
WO_GEMM_SOURCES = ("bit_quantized_gemm_dequant_gb300/csrc/wo_gemm.cu",
                   "bit_quantized_gemm_dequant_gb300/csrc/tc_common.cuh",
                   "bit_quantized_gemm_dequant_gb300/csrc/wq_internal.h")
FP4_GEMM_SOURCES = ("bit_quantized_gemm_dequant_gb300/csrc/gemm_mxf4.cu",
                    "bit_quantized_gemm_dequant_gb300/csrc/mx_block.cuh",
                    "bit_quantized_gemm_dequant_gb300/csrc/tc_common.cuh",
                    "bit_quantized_gemm_dequant_gb300/csrc/wq_internal.h")
FP8_SOURCES = ("bit_quantized_gemm_dequant_gb300/csrc/gemm_fp8.cu",
               "bit_quantized_gemm_dequant_gb300/csrc/tc_common.cuh",
               "bit_quantized_gemm_dequant_gb300/csrc/wq_internal.h")
CAPTURED_TRAFFIC = {
    "w8a16_16x4096x14336":
        {"bytes": 58_932_224 + 81_920, "sources": SKINNY_SOURCES, "sha256": "dd7eac26bf5a279150b6c656275224f6bb697d7a1366c5dff68949f92c906d52"},
    "w8a16_batched_1x4096x4096+4x4096x4096+16x4096x4096+1x4096x14336+4x4096x14336+16x4096x14336":
        {"bytes": 227_881_216 + 5_397_248, "sources": BATCHED_SOURCES, "sha256": "d2feb37b479c0b3921272d36160bed0a59aaf9ff653ecd9cf3bb821d99568f9e"},
    "w4a16_64x4096x11008":
        {"bytes": 23_121_664 + 0, "sources": WO_GEMM_SOURCES, "sha256": "017da18f0fc221b5ab0d5beb4f93f8975fb361416a83d6b69797023eac01d3ef"},
    "mx_gemm_128x8192x8192":
        {"bytes": 36_239_872 + 2_304, "sources": FP4_GEMM_SOURCES, "sha256": "7e31aaba2391f37b7b6b2c8d9220cc160d19db187ac3d68f7a87b7dd6c5d45be"},
    "mx_gemm_2048x8192x8192":
        {"bytes": 44_658_176 + 16_946_944, "sources": FP4_GEMM_SOURCES, "sha256": "7e31aaba2391f37b7b6b2c8d9220cc160d19db187ac3d68f7a87b7dd6c5d45be"},
    "nv_gemm_2048x8192x8192":
        {"bytes": 47_368_192 + 19_126_272, "sources": FP4_GEMM_SOURCES, "sha256": "7e31aaba2391f37b7b6b2c8d9220cc160d19db187ac3d68f7a87b7dd6c5d45be"},
    "mx_gemm_8192x8192x8192":
        {"bytes": 123_218_432 + 229_491_456, "sources": FP4_GEMM_SOURCES, "sha256": "7e31aaba2391f37b7b6b2c8d9220cc160d19db187ac3d68f7a87b7dd6c5d45be"},
    "nv_gemm_8192x8192x8192":
        {"bytes": 151_796_992 + 231_795_200, "sources": FP4_GEMM_SOURCES, "sha256": "7e31aaba2391f37b7b6b2c8d9220cc160d19db187ac3d68f7a87b7dd6c5d45be"},
    "fp8_8192x8192x8192":
        {"bytes": 214_076_672 + 110_690_816, "sources": FP8_SOURCES, "sha256": "cc4cfe24612f25dd3ab2a6bae7fbdc0ed6040fa71727478b9752671a18d37d5d"},
    "fp8_4096x4096x4096":
        {"bytes": 33_620_992 + 288_000, "sources": FP8_SOURCES, "sha256": "cc4cfe24612f25dd3ab2a6bae7fbdc0ed6040fa71727478b9752671a18d37d5d"},
}


def code_sha256(text):
    """SHA-256 of a C++/CUDA source with its comments, indentation and blank
    lines removed, so that such edits do not invalidate a capture of
    unchanged code."""
    import hashlib
    import re

    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = [re.sub(r"//.*$", "", ln).strip() for ln in text.splitlines()]
    return hashlib.sha256("\n".join(ln for ln in lines if ln).encode()).hexdigest()


def sources_sha256(paths):
    """One SHA-256 over the code_sha256 of each source, in order."""
    import hashlib

    parts = []
    for rel in paths:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            parts.append(code_sha256(f.read()))
    return hashlib.sha256("\n".join(parts).encode()).hexdigest()


def captured_traffic(call_name):
    """DRAM bytes of one launch from an ncu capture, while the kernel's
    sources (comments aside) still hold the code that was captured; else None."""
    t = CAPTURED_TRAFFIC.get(call_name)
    if t is None:
        return None
    try:
        if sources_sha256(t["sources"]) != t["sha256"]:
            return None
    except OSError:
        return None
    return t["bytes"]


def roofline_for(call, peaks, traffic=None):
    if call["bound"] == "hbm":
        achieved = call["bytes"] / (call["ms"] * 1e-3) / 1e9
        peak, unit, src = peaks["hbm_gbs"], "GB/s", peaks["source"] + " HBM copy"
    else:
        ratio = NOMINAL_RATIO[call["dtype"]]
        achieved = call["flops"] / (call["ms"] * 1e-3) / 1e12
        peak, unit = peaks["bf16_tflops"] * ratio, "TFLOP/s"
        src = peaks["source"] + (f" bf16 burst x {ratio:g} (nominal {call['dtype']}/bf16 ratio)" if ratio != 1
                                 else " bf16 burst")
    return {"bound": call["bound"], "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic, "kernel_call": call["call"], "peak_source": src}


# ------------------------------------------------------------------- clocks


class _NvmlClocks:
    """Samples the SM clock and the clock-event (throttle) reasons through NVML,
    called with ctypes on the driver's library, from a background thread about
    every 0.5 ms: a timed region of well under a millisecond still gets
    samples.  Only reads; changes no setting."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, pci):
        import ctypes
        import threading

        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        if pci is None or self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci.encode(), ctypes.byref(self.dev)) != 0:
            raise OSError("no NVML handle for the GPU")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx)) == 0 else None
        self.samples, self.seen = [], set()
        self.stop = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _run(self):
        ct = self.ct
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while not self.stop.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ct.byref(clk)) == 0:  # NVML_CLOCK_SM
                self.samples.append(float(clk.value))
            if self.reasons_fn(self.dev, ct.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.seen.add(name)
            time.sleep(0.0005)

    def finish(self):
        self.stop.set()
        self.thread.join(timeout=5)
        try:
            self.lib.nvmlShutdown()
        except Exception:
            pass
        if not self.samples:
            return {"error": "no samples"}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz, "reasons": sorted(self.seen),
                "samples": len(self.samples), "source": "NVML, ~0.5 ms period"}


def _sample_clocks(pci=None):
    """Start sampling clocks and throttle reasons: NVML at ~0.5 ms when the
    driver library loads, else nvidia-smi every 200 ms."""
    try:
        return _NvmlClocks(pci)
    except Exception:
        pass
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
    if isinstance(proc, _NvmlClocks):
        return proc.finish()
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


# ----------------------------------------------------------------- the arms


def _dist():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def _unit_of(calls):
    return "GB/s" if all(c["bound"] == "hbm" for c in calls) else "TFLOP/s"


def _throughput(calls, unit, seconds, factor=1):
    if unit == "GB/s":
        return factor * sum(c["bytes"] for c in calls) / seconds / 1e9
    return factor * sum(c["flops"] for c in calls) / seconds / 1e12


DTYPES = {"w8a16": "int8 weights x fp16 activations, fp32 accumulate",
          "w4a16": "int4 weights x fp16 activations, fp32 accumulate",
          "mxfp4": "e2m1 x e2m1 with e8m0 block scales, fp32 accumulate",
          "nvfp4": "e2m1 x e2m1 with e4m3 block scales and fp32 tensor scales, fp32 accumulate",
          "fp8": "e4m3 x e4m3, fp32 accumulate, bf16 out"}


def run_ours(args):
    import torch

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    import bit_quantized_gemm_dequant_gb300 as wq

    wq.set_static_weights(args.static_weights)
    peaks = load_peaks()
    probe = make_workload(torch, wq, args.workload, 1, args.only)
    step_bytes = sum(c["bytes"] for c in probe.calls)
    del probe
    torch.cuda.empty_cache()
    replicas = replicas_for(step_bytes)
    wl = make_workload(torch, wq, args.workload, replicas, args.only)
    unit = _unit_of(wl.calls)

    clock_proc = _sample_clocks(_pci_bus_id(torch, local)) if rank == 0 else None
    total_ms = time_steps(torch, wl, args.steps, args.warmup, replicas, ws)
    clocks = _finish_clocks(clock_proc, _pci_bus_id(torch, local)) if rank == 0 else None
    per_call = time_each_call(torch, wl, args.steps, replicas)

    value = _throughput(wl.calls, unit, total_ms * 1e-3 / args.steps, factor=ws)
    dominant = max(per_call, key=lambda c: c["ms"])
    roof = roofline_for(dominant, peaks,
                        traffic=args.traffic if args.traffic is not None else captured_traffic(dominant["call"]))

    e2e = None
    if not args.no_e2e and hasattr(wl, "e2e_call"):
        host = wl.host_inputs()
        for c in wl.calls:
            wl.e2e_call(host, c["index"])
        torch.cuda.synchronize()
        n = max(1, min(args.steps, 10))
        h2d = d2h = 0
        t0 = time.perf_counter()
        for _ in range(n):
            h2d = d2h = 0
            for c in wl.calls:
                bi, bo = wl.e2e_call(host, c["index"])
                h2d += bi
                d2h += bo
        torch.cuda.synchronize()
        e2e_s = _barrier_max(torch, time.perf_counter() - t0, ws)
        e2e = {"value": round(_throughput(wl.calls, unit, e2e_s / n, factor=ws), 3), "unit": unit,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "how": "wall clock over steps of: pinned-host -> device copies of X, W and scales, the C-ABI call, "
                      "device -> pinned-host copy of Y; one synchronize at the end"}

    breakdown = []
    if not args.no_breakdown and rank == 0:
        for name in BREAKDOWN:
            if name == args.workload:
                continue
            decode = workloads.WORKLOADS[name].get("batched") or name.endswith("_decode")
            reps = 1
            if decode:  # inputs rotate over replicas, as for the headline
                reps = replicas_for(sum(_wo_bytes(4 if workloads.WORKLOADS[name]["op"] == "w4a16" else 8, *sh)
                                        for sh in workloads.WORKLOADS[name]["shapes"]))
            other = make_workload(torch, wq, name, reps)
            if decode:
                # decode sweeps: back to back, as the headline is measured
                steps_ms = time_steps(torch, other, 20, 5, reps, 1)
                unit_o = _unit_of(other.calls)
                row = {"workload": name, "call": "back-to-back step of " + ", ".join(c["call"] for c in other.calls),
                       "bytes": sum(c["bytes"] for c in other.calls), "flops": sum(c["flops"] for c in other.calls),
                       "bound": "hbm", "dtype": "fp16", "ms": steps_ms / 20}
                row["roofline"] = roofline_for(row, peaks)
                if args.cpu_budget > 0:
                    row["cpu_baseline"] = oracle_rate(other, other.calls, unit_o, 1.5)
                breakdown.append(row)
            else:
                for c in time_calls_flushed(torch, other, 5, 3):
                    row = {"workload": name, **c, "roofline": roofline_for(c, peaks, captured_traffic(c["call"]))}
                    if args.cpu_budget > 0:
                        row["cpu_baseline"] = oracle_rate(other, [next(x for x in other.calls if x["call"] == c["call"])],
                                                          row["roofline"]["unit"], 0.7)
                    breakdown.append(row)
            del other
            torch.cuda.empty_cache()

    cpu = cpu_baseline(wl, unit, args.cpu_budget) if (rank == 0 and ws == 1 and args.cpu_budget > 0) else None

    if rank == 0:
        op = workloads.WORKLOADS[args.workload]["op"]
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": DTYPES[op],
            "data": "synthetic (seeded numpy; shapes and distributions of the workload)",
            "config": {"workload": f"{args.workload}: " + ", ".join(c["call"] for c in wl.calls), "seed": 0,
                       "replicas": replicas,
                       "l2": f"inputs rotate over {replicas} replicas of {step_bytes / 1e6:.0f} MB per step "
                             f"(> 2 x {L2_BYTES / 1e6:.0f} MB L2 between reuses)",
                       "parallelism": f"replicas x{ws}",
                       "static_weights": bool(args.static_weights)},
            "roofline": roof,
            "per_call": [{**c, "achieved": roofline_for(c, peaks)["achieved"]} for c in per_call],
            "e2e": e2e,
            "gpu_launches": sum(c.get("launches", 1) for c in wl.calls) * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "breakdown": breakdown,
        }
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()


def cpu_baseline(wl, unit, budget_s):
    """The oracle as it stands on this host: whole calls of the workload, in
    order, until about budget_s seconds have passed."""
    if not hasattr(wl, "oracle_call"):
        return None
    t0 = time.perf_counter()
    nbytes = nflops = ncalls = 0
    desc = set()
    while time.perf_counter() - t0 < budget_s and ncalls < 200:
        c = wl.calls[ncalls % len(wl.calls)]
        b, f, d = wl.oracle_call(c["index"])
        nbytes += b
        nflops += f
        ncalls += 1
        desc.add(d)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9 if unit == "GB/s" else nflops / dt / 1e12
    return {"value": round(value, 5), "unit": unit, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{ncalls} oracle call(s) of the workload in order ({dt:.1f} s; {'; '.join(sorted(desc))}; "
                      f"numpy float64, BLAS threads = cores)"}


def oracle_rate(wl, calls, unit, budget_s):
    """The oracle's throughput on the given calls, in `unit`, from a bounded
    sample (each call's own oracle sample, repeated for about budget_s)."""
    nbytes = nflops = n = 0
    desc = set()
    t0 = time.perf_counter()
    while n == 0 or time.perf_counter() - t0 < budget_s:
        for c in calls:
            b, f, d = wl.oracle_call(c["index"])
            nbytes, nflops = nbytes + b, nflops + f
            desc.add(d)
        n += 1
        if n >= 50:
            break
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9 if unit == "GB/s" else nflops / dt / 1e12
    return {"value": round(value, 6), "unit": unit, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} pass(es), {dt:.2f} s: " + "; ".join(sorted(desc))}


# Column subset per weight-only call in the reference arm (the oracle's cost
# is dequantizing W in float64, proportional to the columns).
REF_COLS = 2048


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    spec = workloads.WORKLOADS[args.workload]
    wl = make_workload(None, None, args.workload, 0, args.only)  # host-side inputs only
    unit = _unit_of(wl.calls)
    op = spec["op"]

    def one_step():
        b = f = 0
        desc = set()
        for c in wl.calls:
            if op in ("w4a16", "w8a16"):
                bi, fi, d = wl.oracle_call(c["index"], cols=REF_COLS)
            else:
                bi, fi, d = wl.oracle_call(c["index"])
            b, f = b + bi, f + fi
            desc.add(d)
        return b, f, desc

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    nbytes = nflops = 0
    desc = set()
    for _ in range(args.steps):
        b, f, d = one_step()
        nbytes, nflops = nbytes + b, nflops + f
        desc |= d
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9 if unit == "GB/s" else nflops / dt / 1e12
    sample = "every call of the workload per step, each on the oracle's sample: " + "; ".join(sorted(desc))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: " + ", ".join(c["call"] for c in wl.calls),
                   "seed": 0, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="w8a16_decode", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--only", default=None, help="keep only the calls whose name contains this string")
    ap.add_argument("--no-breakdown", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--static-weights", action="store_true",
                    help="wq_set_static_weights(1): the weights are only read during the run, so the decode "
                         "kernels may load their first weight boxes while the previous call finishes")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the dominant kernel from an ncu capture of this build")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world = os.environ.get("WORLD_SIZE")
    if world is None and args.gpus > 1:
        # No launcher around this process: start one rank per GPU under the
        # torch launcher (127.0.0.1 rendezvous) and pass its status on.
        import socket

        with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(args.gpus),
               "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
        sys.exit(subprocess.call(cmd))
    if world is not None and int(world) != args.gpus:
        sys.exit(f"bench.py: --gpus {args.gpus} but the launcher started {world} rank(s)")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
