"""Seeded synthetic inputs for the fused dequantization GEMM library.

This module serves both the CUDA path (tests, benchmark, smoke check) and the
CPU oracle, and holds none of the method's arithmetic: it only draws random
codes, activations, scales and float sources with the shapes and value
distributions of the workloads below.  The one non-random step, turning the
FP8 source into e4m3 bytes, is input preparation done by PyTorch's own
``float8_e4m3fn`` cast (the FP8 page's GEMM consumes e4m3 inputs that were
scaled so that the tensor's amax maps to 448).

Every generator takes a seed; weights, activations and sources draw from
separate streams (``numpy.random.default_rng((seed, stream_id, ...))``) so
that a weight matrix is the same for every M that multiplies it.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# Stream ids keep the draws of different tensors independent.
_W_STREAM, _X_STREAM, _S_STREAM, _SRC_STREAM = 1, 2, 3, 4


def _rng(seed: int, *tags: int) -> np.random.Generator:
    return np.random.default_rng((int(seed),) + tuple(int(t) for t in tags))


# ---------------------------------------------------------------- weight-only


def activations_fp16(m: int, k: int, seed: int = 0) -> np.ndarray:
    """X fp16 [m, k], entries N(0, 1) drawn in float32 and rounded to fp16."""
    return _rng(seed, _X_STREAM, m, k).standard_normal((m, k), dtype=np.float32).astype(np.float16)


def activations_fp16_shifted(m: int, k: int, kind: str, seed: int = 0) -> np.ndarray:
    """X fp16 [m, k] with a non-zero mean: "normal_mean2" draws N(2, 1),
    "uniform01" draws U(0, 1) (both in float32, rounded to fp16)."""
    g = _rng(seed, _X_STREAM, 7, m, k)
    if kind == "normal_mean2":
        v = g.standard_normal((m, k), dtype=np.float32) + np.float32(2.0)
    elif kind == "uniform01":
        v = g.random((m, k), dtype=np.float32)
    else:
        raise ValueError(kind)
    return v.astype(np.float16)


def int4_codes_packed(k: int, n: int, seed: int = 0) -> np.ndarray:
    """Packed INT4 weights uint8 [k/2, n]: codes uniform on 0..15, the code for
    even k in the low nibble and odd k in the high nibble."""
    if k % 2:
        raise ValueError("k must be even")
    # Two independent uniform nibbles per byte are one uniform byte.
    return _rng(seed, _W_STREAM, k, n).integers(0, 256, size=(k // 2, n), dtype=np.uint8)


def int8_codes(k: int, n: int, seed: int = 0, lo: int = -127, hi: int = 127) -> np.ndarray:
    """INT8 weights [k, n], uniform on lo..hi inclusive."""
    return _rng(seed, _W_STREAM, k, n).integers(lo, hi + 1, size=(k, n), dtype=np.int16).astype(np.int8)


def column_scales_fp16(n: int, lo: float, hi: float, seed: int = 0) -> np.ndarray:
    """Per-column fp16 scales [n], uniform on [lo, hi) drawn in float32."""
    return _rng(seed, _S_STREAM, n).uniform(lo, hi, size=n).astype(np.float32).astype(np.float16)


@dataclass
class WeightOnlyCase:
    x: np.ndarray        # fp16 [M, K]
    w: np.ndarray        # uint8 [K/2, N] (INT4) or int8 [K, N] (INT8)
    scales: np.ndarray   # fp16 [N]
    bits: int


def w4a16_case(m: int, k: int, n: int, seed: int = 0) -> WeightOnlyCase:
    """INT4 weight-only case: X ~ N(0,1), codes U{0..15}, scales ~ U(0.005, 0.02)."""
    return WeightOnlyCase(activations_fp16(m, k, seed), int4_codes_packed(k, n, seed),
                          column_scales_fp16(n, 0.005, 0.02, seed), 4)


def w8a16_case(m: int, k: int, n: int, seed: int = 0) -> WeightOnlyCase:
    """INT8 weight-only case: X ~ N(0,1), q U{-127..127}, scales ~ U(0.001, 0.01)."""
    return WeightOnlyCase(activations_fp16(m, k, seed), int8_codes(k, n, seed),
                          column_scales_fp16(n, 0.001, 0.01, seed), 8)


_Z_STREAM = 5


@dataclass
class GroupedCase:
    x: np.ndarray        # fp16 [M, K]
    w: np.ndarray        # uint8 [K/2, N] (INT4) or int8 [K, N] (INT8)
    scales: np.ndarray   # fp16 [ceil(N / group_n)]
    zeros: object        # uint8 (INT4) / int8 (INT8) [ceil(N / group_n)], or None
    group_n: int
    bits: int


def grouped_case(bits: int, m: int, k: int, n: int, group_n: int, asym: bool, seed: int = 0) -> GroupedCase:
    """Weight-only case with column-grouped scales and optional zero points.
    Codes and activations as in ``w4a16_case`` / ``w8a16_case``; one scale per
    group of ``group_n`` columns (same ranges); zero points U{0..15} (INT4) or
    U{-32..32} (INT8)."""
    groups = -(-n // group_n)
    base = w4a16_case(m, k, n, seed) if bits == 4 else w8a16_case(m, k, n, seed)
    lo, hi = (0.005, 0.02) if bits == 4 else (0.001, 0.01)
    scales = column_scales_fp16(groups, lo, hi, seed + 1000 * group_n)
    zeros = None
    if asym:
        g = _rng(seed, _Z_STREAM, groups, group_n)
        zeros = (g.integers(0, 16, groups).astype(np.uint8) if bits == 4
                 else g.integers(-32, 33, groups).astype(np.int8))
    return GroupedCase(base.x, base.w, scales, zeros, group_n, bits)


# ---------------------------------------------------------------------- MXFP4


def mx_source(rows: int, cols: int, seed: int = 0, sigma: float = 0.5, stream: int = 0) -> np.ndarray:
    """float32 [rows, cols] ~ N(0, sigma^2): the MXFP4 operands before quantization."""
    g = _rng(seed, _SRC_STREAM, stream, rows, cols)
    return (g.standard_normal((rows, cols), dtype=np.float32) * np.float32(sigma)).astype(np.float32)


# ------------------------------------------------------------------------ FP8


@dataclass
class Fp8Case:
    a8: np.ndarray   # uint8 e4m3fn bytes [M, K]
    b8: np.ndarray   # uint8 e4m3fn bytes [K, N]
    scale_a: float   # float32 per-tensor scale: amax_A / 448
    scale_b: float


def _to_e4m3_bytes(src: np.ndarray):
    import torch  # only for its float8_e4m3fn cast (input preparation)

    amax = float(np.abs(src).max())
    scale = np.float32(amax / 448.0) if amax > 0 else np.float32(1.0)
    scaled = (src * np.float32(448.0 / amax)).astype(np.float32) if amax > 0 else src
    t = torch.from_numpy(np.ascontiguousarray(scaled)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy(), float(scale)


def fp8_case(m: int, k: int, n: int, seed: int = 0) -> Fp8Case:
    """Sources ~ N(0, 1), scaled so that each tensor's amax maps to 448, cast to
    e4m3fn; the per-tensor scale is amax / 448."""
    src_a = _rng(seed, _SRC_STREAM, 10, m, k).standard_normal((m, k), dtype=np.float32)
    src_b = _rng(seed, _SRC_STREAM, 11, k, n).standard_normal((k, n), dtype=np.float32)
    a8, sa = _to_e4m3_bytes(src_a)
    b8, sb = _to_e4m3_bytes(src_b)
    return Fp8Case(a8, b8, sa, sb)


# ---------------------------------------------------------------- workloads

#: The workloads the library is measured on, named by what they are.
WORKLOADS = {
    "w4a16_tiny": {"op": "w4a16", "shapes": [(16, 512, 512)]},
    "w8a16_decode": {"op": "w8a16", "shapes": [(m, 4096, n) for n in (4096, 14336) for m in (1, 4, 16)]},
    # The decode sweep with one scale and one zero point per 128 columns.
    "w8a16_grouped_decode": {"op": "w8a16", "group_n": 128, "asym": True,
                             "shapes": [(m, 4096, n) for n in (4096, 14336) for m in (1, 16)]},
    # The decode (M <= 16) calls of the Llama-7B-shaped INT4 linears.
    "w4a16_decode": {"op": "w4a16", "shapes": [(m, k, n) for (k, n) in ((4096, 4096), (4096, 11008), (11008, 4096))
                                               for m in (1, 8)]},
    # The same two decode sweeps as one batched call per step (all problems of
    # the sweep in one launch).
    "w8a16_decode_batched": {"op": "w8a16", "batched": True,
                             "shapes": [(m, 4096, n) for n in (4096, 14336) for m in (1, 4, 16)]},
    "w4a16_decode_batched": {"op": "w4a16", "batched": True,
                             "shapes": [(m, k, n) for (k, n) in ((4096, 4096), (4096, 11008), (11008, 4096))
                                        for m in (1, 8)]},
    "w4a16_llama7b": {"op": "w4a16", "shapes": [(m, k, n) for (k, n) in ((4096, 4096), (4096, 11008), (11008, 4096))
                                                for m in (1, 8, 64, 512, 4096)]},
    "mxfp4": {"op": "mxfp4", "shapes": [(m, 8192, 8192) for m in (128, 2048, 8192)]},
    # The same, with A quantized inside the GEMM launch (one call per M).
    "mxfp4_qa": {"op": "mxfp4", "fused_a": True, "shapes": [(m, 8192, 8192) for m in (128, 2048, 8192)]},
    # The same operands in NVFP4 (16-element blocks, E4M3 block scales, FP32
    # tensor scale), quantized on the device, then C = A W^T.
    "nvfp4": {"op": "nvfp4", "shapes": [(m, 8192, 8192) for m in (128, 2048, 8192)]},
    "fp8": {"op": "fp8", "shapes": [(4096, 4096, 4096), (8192, 8192, 8192), (16, 8192, 8192)]},
}
