"""CPU oracle for the fused dequantization GEMM library — TEST INFRASTRUCTURE ONLY.

This module is a plain, slow, obviously-correct restatement of what the four
source pages define.  It exists so that tests, the smoke check and the CPU
baseline leg of the benchmark can check the CUDA path against something
written independently of it.  Nothing in the product (the package, its C ABI
or its kernels) may import or call it; the product fails loudly instead when
its CUDA library is missing.

It shares no code with the CUDA path.  Inputs come from the seeded generators
in ``workloads.py`` (which hold none of the method's arithmetic).

Pages cited (title, then the short name used below):

* "Triton 工业级融合微算子编写：W4A16 极速切片矩阵乘与 Blackwell NVFP4 硬件指令实装"
  (dreamvfia.cn) — the *W4A16 page*.
* "量化推理引擎中的微缩放格式前瞻：MXFP4 矩阵乘法 Kernel 原理" (pwwt.cn) —
  the *MXFP4 page*.
* "Triton Quantization | Triton 量化算子：W8A16 权重量化融合矩阵乘法
  (Quantization GEMM)" (datawhalechina llm-algo-leetcode) — the *W8A16 page*.
* "通过 CUTLASS 命名约定在 Triton 中实现 FP8 GEMM 内核" (blog.hotdry.top) —
  the *FP8 page*.

Precision: every contraction accumulates in float64.  The one place where
floating point decides an integer (the MXFP4 code choice) is taken in
float32, the precision the MXFP4 page's simulator computes in.

Every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` against closed forms, brute force with exact
rational arithmetic, hand-derived worked examples and library routines.
"""
from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------
# Weight-only INT4 (W4A16 page, §二 "Triton 工业级 W4A16 融合矩阵乘算子实装")
# --------------------------------------------------------------------------

INT4_ZERO_POINT = 8  # W4A16 page §二: dequantize as (q - 8) * scale


def unpack_int4(wq: np.ndarray) -> np.ndarray:
    """Unpack INT4 codes from bytes laid out ``[K/2, N]``.

    W4A16 page §二: byte row ``k // 2`` holds two K-consecutive codes; the
    code for ``k`` sits at bit offset ``(k % 2) * 4``, so the even k is the
    low nibble and the odd k the high nibble.  Returns int codes ``[K, N]``
    in ``0..15``.
    """
    wq = np.asarray(wq, dtype=np.uint8)
    half_k, n = wq.shape
    q = np.empty((2 * half_k, n), dtype=np.int64)
    q[0::2, :] = wq & 0x0F
    q[1::2, :] = wq >> 4
    return q


def dequant_w4(wq: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """W = (q - 8) * s[n] in float64 (W4A16 page §二, per-column scale)."""
    q = unpack_int4(wq).astype(np.float64)
    s = np.asarray(scales).astype(np.float64)
    return (q - INT4_ZERO_POINT) * s[None, :]


def gemm_w4a16(x: np.ndarray, wq: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Y[m, n] = sum_k x[m, k] * (q[k, n] - 8) * s[n], accumulated in float64.

    W4A16 page §二: activations fp16 ``[M, K]``, packed INT4 ``[K/2, N]``,
    fp16 scales ``[N]``.  The page rounds the dequantized weight to fp16
    inside its loop; the plain definition it approximates is the exact
    product, which is what this returns (float64, no output rounding).
    """
    xf = np.asarray(x).astype(np.float64)
    return xf @ dequant_w4(wq, scales)


# --------------------------------------------------------------------------
# Weight-only INT8 (W8A16 page, Step 1 formula and the reference solution)
# --------------------------------------------------------------------------


def dequant_w8(w: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """W = q * s[n] in float64 (W8A16 page, Step 1: Y = X x (W_int8 x S))."""
    q = np.asarray(w, dtype=np.int8).astype(np.float64)
    s = np.asarray(scales).astype(np.float64)
    return q * s[None, :]


def gemm_w8a16(x: np.ndarray, w: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Y = X @ (W_int8 * S) with per-column S, accumulated in float64.

    W8A16 page, Step 1 and Step 3: X fp16 ``[M, K]``, W int8 ``[K, N]``,
    S fp16 ``[N]``, symmetric (no zero point).
    """
    xf = np.asarray(x).astype(np.float64)
    return xf @ dequant_w8(w, scales)


# --------------------------------------------------------------------------
# Column-grouped scales and zero points (W8A16 page, "扩展说明": when N is
# large several columns may share one scale, and a zero_point turns the
# symmetric scheme asymmetric; W4A16 page §一, the naive dequantization
# w = (w_int4 - zero_point) * scale)
# --------------------------------------------------------------------------


def dequant_grouped(q: np.ndarray, scales: np.ndarray, zeros, group_n: int, default_zero: int) -> np.ndarray:
    """W[k, n] = (q[k, n] - z[n // group_n]) * s[n // group_n] in float64.

    ``q`` are the integer codes ``[K, N]``.  Columns ``g*group_n ..
    (g+1)*group_n - 1`` share scale ``s[g]`` and zero point ``z[g]``; the
    last group may be short.  ``zeros=None`` is the symmetric scheme, with
    the fixed zero point ``default_zero``.
    """
    q = np.asarray(q, dtype=np.int64)
    n = q.shape[1]
    g = np.arange(n) // int(group_n)
    s = np.asarray(scales).astype(np.float64)[g]
    z = np.full(n, default_zero, np.int64) if zeros is None else np.asarray(zeros).astype(np.int64)[g]
    return (q - z[None, :]).astype(np.float64) * s[None, :]


def gemm_w4a16_grouped(x: np.ndarray, wq: np.ndarray, scales: np.ndarray, zeros=None, group_n: int = 1) -> np.ndarray:
    """Y[m, n] = sum_k x[m, k] * (q[k, n] - z[n // G]) * s[n // G], float64.

    Packed INT4 codes as in ``unpack_int4``; ``zeros`` are integers (one per
    column group) or None for the W4A16 page's fixed zero point 8.  With
    ``group_n = 1`` and ``zeros=None`` this is ``gemm_w4a16``.
    """
    xf = np.asarray(x).astype(np.float64)
    return xf @ dequant_grouped(unpack_int4(wq), scales, zeros, group_n, INT4_ZERO_POINT)


def gemm_w8a16_grouped(x: np.ndarray, w: np.ndarray, scales: np.ndarray, zeros=None, group_n: int = 1) -> np.ndarray:
    """Y[m, n] = sum_k x[m, k] * (q[k, n] - z[n // G]) * s[n // G], float64.

    INT8 codes ``[K, N]``; ``zeros`` are integers (one per column group) or
    None for the W8A16 page's symmetric scheme (zero point 0).  With
    ``group_n = 1`` and ``zeros=None`` this is ``gemm_w8a16``.
    """
    xf = np.asarray(x).astype(np.float64)
    q = np.asarray(w, dtype=np.int8).astype(np.int64)
    return xf @ dequant_grouped(q, scales, zeros, group_n, 0)


# --------------------------------------------------------------------------
# MXFP4 (MXFP4 page: micro-block format, §二 equations, §三 simulator)
# --------------------------------------------------------------------------

MX_BLOCK = 32  # MXFP4 page: 32 four-bit elements share one E8M0 exponent
E8M0_BIAS = 127  # MXFP4 page §二.2: S = 2^(E - 127)
# MXFP4 page §三: the E2M1 magnitude grid the simulator rounds onto.
E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
E2M1_MAX = 6.0
AMAX_FLOOR = np.float32(1e-8)  # MXFP4 page §三: amax.clamp(min=1e-8)


def ceil_log2_f32(q: np.ndarray) -> np.ndarray:
    """Exact ceil(log2(q)) for positive normal float32 ``q``.

    The MXFP4 page §三 takes ``ceil(log2(amax / 6))``.  Read as the exact
    mathematical value: write q = f * 2^x with f in [0.5, 1); log2(q) is an
    integer only when f == 0.5 (then it is x - 1), otherwise its ceiling is x.
    """
    f, x = np.frexp(np.asarray(q, dtype=np.float32))
    return np.where(f == np.float32(0.5), x - 1, x).astype(np.int64)


def mx_quantize_fp4(src: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Quantize float32 ``[R, C]`` (C % 32 == 0) to MXFP4.

    Steps in the MXFP4 page's order (§三, ``pack_tensor_to_mxfp4_layout``),
    all on float32 values:

    1. split every row into 32-element blocks;
    2. amax = max |x| over the block, clamped below at 1e-8;
    3. e = ceil(log2(amax / 6)) (exact, see ``ceil_log2_f32``); E = e + 127;
    4. normalise v = x / 2^e (exact: a power-of-two division);
    5. code magnitude j = argmin_j | |v| - grid[j] |, the first index on a tie
       (numpy's argmin, like the page's torch.argmin, returns the first);
    6. sign bit = (x < 0); the 4-bit code is sign << 3 | j.

    Returns ``(data, scales)``: data uint8 ``[R, C/2]`` with element 2t in the
    low nibble and 2t+1 in the high nibble of byte t (the same nibble order as
    the W4A16 page's INT4 packing), and E8M0 bytes uint8 ``[R, C/32]``.
    Data and scale segments are separate arrays, as the MXFP4 page §一 lays
    them out.
    """
    x = np.asarray(src, dtype=np.float32)
    rows, cols = x.shape
    if cols % MX_BLOCK:
        raise ValueError("cols must be a multiple of 32")
    nb = cols // MX_BLOCK
    blocks = x.reshape(rows, nb, MX_BLOCK)
    amax = np.abs(blocks).max(axis=-1) if nb else np.zeros((rows, 0), np.float32)
    amax = np.maximum(amax, AMAX_FLOOR)
    q = (amax / np.float32(E2M1_MAX)).astype(np.float32)
    e = ceil_log2_f32(q)
    pow2 = np.ldexp(np.float32(1.0), e).astype(np.float32)
    v = (blocks / pow2[..., None]).astype(np.float32)
    grid = np.asarray(E2M1_GRID, dtype=np.float32)
    dist = np.abs(np.abs(v)[..., None] - grid).astype(np.float32)
    j = np.argmin(dist, axis=-1).astype(np.uint8)
    sign = (blocks < 0).astype(np.uint8)
    codes = ((sign << 3) | j).reshape(rows, cols)
    data = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    scales = (e + E8M0_BIAS).astype(np.uint8)
    return data, scales


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """Value of 4-bit E2M1 codes: (-1)^s * grid[code & 7] (MXFP4 page §三)."""
    c = np.asarray(codes, dtype=np.int64)
    mag = np.asarray(E2M1_GRID, dtype=np.float64)[c & 7]
    return np.where(c & 8, -mag, mag)


def mx_unpack_codes(data: np.ndarray) -> np.ndarray:
    """Split MXFP4 data bytes ``[R, C/2]`` into codes ``[R, C]`` (low nibble first)."""
    d = np.asarray(data, dtype=np.uint8)
    rows, half = d.shape
    codes = np.empty((rows, 2 * half), dtype=np.int64)
    codes[:, 0::2] = d & 0x0F
    codes[:, 1::2] = d >> 4
    return codes


def mx_dequantize(data: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """x_hat = decode(code) * 2^(E - 127), float64 ``[R, C]`` (MXFP4 page §二.2)."""
    vals = e2m1_decode(mx_unpack_codes(data))
    rows, cols = vals.shape
    e = np.asarray(scales, dtype=np.int64) - E8M0_BIAS
    vals = vals.reshape(rows, cols // MX_BLOCK, MX_BLOCK)
    return np.ldexp(vals, e[..., None]).reshape(rows, cols)


def mx_gemm_fp4(a_data, a_scales, w_data, w_scales, rows=None) -> np.ndarray:
    """C = A @ W^T for MXFP4 operands, float64.

    MXFP4 page §二.1 (block dot-product equation) and §二.2 (exponent
    addition): for every output (m, n) and every 32-element K block k,

        dC = 2^(E_A[m,k] + E_W[n,k] - 254) * sum_{i<32} a[m,k,i] * w[n,k,i]

    and C is the sum of dC over the blocks, in the simulator's order (§三):
    block dot first, then the combined power-of-two scale, then the running
    sum.  A ``[M, K/2]`` + ``[M, K/32]`` and W ``[N, K/2]`` + ``[N, K/32]``
    are both K-contiguous.  ``rows`` optionally restricts the output to a
    subset of A's rows (used for sampled parity at large sizes).
    """
    ca = e2m1_decode(mx_unpack_codes(a_data))
    cw = e2m1_decode(mx_unpack_codes(w_data))
    ea = np.asarray(a_scales, dtype=np.int64)
    ew = np.asarray(w_scales, dtype=np.int64)
    if rows is not None:
        ca, ea = ca[rows], ea[rows]
    m, k = ca.shape
    n = cw.shape[0]
    nb = k // MX_BLOCK
    out = np.zeros((m, n), dtype=np.float64)
    for b in range(nb):
        sl = slice(b * MX_BLOCK, (b + 1) * MX_BLOCK)
        block_dot = ca[:, sl] @ cw[:, sl].T  # exact: small dyadic rationals
        combined = ea[:, b][:, None] + ew[:, b][None, :] - 2 * E8M0_BIAS
        out += np.ldexp(block_dot, combined)
    return out


# --------------------------------------------------------------------------
# FP8 e4m3 (FP8 page: kernel listing and the 精度管理 / 风险考虑 bullets)
# --------------------------------------------------------------------------

E4M3_MAX = 448.0  # FP8 page, 精度管理: scale_max = 448 (E4M3 range)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Value of e4m3fn bytes as float64.

    Sign bit 7, exponent bits 6..3 with bias 7, mantissa bits 2..0.
    Exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is no
    infinity, so the largest finite value is 1.75 * 2^8 = 448, the E4M3 range
    the FP8 page states.
    """
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    man = (c & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + man / 8.0, ex - 7)
    sub = np.ldexp(man / 8.0, -6)
    val = sign * np.where(ex == 0, sub, normal)
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def fp8_gemm(a8: np.ndarray, b8: np.ndarray, scale_a: float, scale_b: float,
             rows=None) -> np.ndarray:
    """C = (sum_k dec(A[m,k]) * dec(B[k,n])) * scale_a * scale_b, float64.

    FP8 page kernel listing and its 精度管理 bullet: e4m3 inputs, FP32 (here
    float64) accumulation, the per-tensor scales applied once to the
    accumulator.  A ``[M, K]``, B ``[K, N]`` e4m3 bytes.  ``rows`` optionally
    restricts the output to a subset of A's rows.
    """
    a = e4m3_decode(a8 if rows is None else np.asarray(a8)[rows])
    b = e4m3_decode(b8)
    return (a @ b) * (float(np.float32(scale_a)) * float(np.float32(scale_b)))


# --------------------------------------------------------------------------
# NVFP4 (W4A16 page, §三 "Blackwell 第五代 Tensor Core NVFP4 指令实操": E2M1
# elements under a two-level block scaling, an FP8 local scale per block of
# elements inside a tensor-wide scale, executed natively by the tensor cores).
# The page gives no block size or scale encoding; the reading taken here is:
# 16-element blocks along the contiguous dimension, an unsigned E4M3 scale per
# block, and a float32 scale per tensor that maps the tensor's amax onto the
# largest block scale times the largest element (448 x 6).  Elements are
# chosen exactly as the MXFP4 page's simulator chooses them (nearest E2M1 grid
# point, the smaller magnitude on a tie, sign bit = x < 0).
# --------------------------------------------------------------------------

NV_BLOCK = 16
NV_SCALE_RANGE = np.float32(E2M1_MAX * E4M3_MAX)  # 6 * 448 = 2688


def e4m3_encode(values) -> np.ndarray:
    """Non-negative values -> e4m3fn bytes: round to the nearest finite e4m3
    value, ties to the even code, saturating at 448 (0x7E).

    The 127 non-negative finite codes 0x00..0x7E decode to increasing values,
    so the result is a search over that table (exact in float64)."""
    v = np.asarray(values, dtype=np.float64)
    if (v < 0).any() or np.isnan(v).any():
        raise ValueError("e4m3_encode takes non-negative numbers")
    table = e4m3_decode(np.arange(0x7F))
    hi = np.clip(np.searchsorted(table, v, side="left"), 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_lo, d_hi = np.abs(v - table[lo]), np.abs(table[hi] - v)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    return np.where(v >= E4M3_MAX, 0x7E, code).astype(np.uint8)


def nv_tensor_scale(src: np.ndarray) -> np.float32:
    """The tensor-wide scale g = amax / (6 * 448) in float32 (1 for an all-zero
    tensor): the largest block then gets the largest block scale, 448."""
    amax = np.float32(np.abs(np.asarray(src, dtype=np.float32)).max()) if np.size(src) else np.float32(0)
    return np.float32(1.0) if amax == 0 else np.float32(amax / NV_SCALE_RANGE)


def nv_quantize_fp4(src: np.ndarray, g=None):
    """Quantize float32 ``[R, C]`` (C % 16 == 0) to NVFP4, in float32 steps:

    1. g = nv_tensor_scale(src) unless given;
    2. per 16-element block: amax = max |x|; the block scale
       s = e4m3(amax / (6 g)) (the division in float32, 6 g rounded to
       float32 first; round to nearest even, saturating at 448);
    3. d = s * g in float32; a block whose scale is 0 gets code 0 everywhere;
    4. v = x / d in float32; code magnitude = the nearest E2M1 grid point to
       |v|, the first (smaller) one on a tie; sign bit = x < 0.

    Returns ``(data, scales, g)``: data uint8 ``[R, C/2]`` (element 2t in the
    low nibble of byte t, as for MXFP4), e4m3 block scales uint8 ``[R, C/16]``
    and g (float32)."""
    x = np.asarray(src, dtype=np.float32)
    rows, cols = x.shape
    if cols % NV_BLOCK:
        raise ValueError("cols must be a multiple of 16")
    g = nv_tensor_scale(x) if g is None else np.float32(g)
    blocks = x.reshape(rows, cols // NV_BLOCK, NV_BLOCK)
    amax = np.abs(blocks).max(axis=-1) if cols else np.zeros((rows, 0), np.float32)
    sb_f = (amax / np.float32(np.float32(6.0) * g)).astype(np.float32)
    sb = e4m3_encode(sb_f)
    d = (e4m3_decode(sb).astype(np.float32) * g).astype(np.float32)
    safe = np.where(d > 0, d, np.float32(1.0)).astype(np.float32)
    v = (blocks / safe[..., None]).astype(np.float32)
    grid = np.asarray(E2M1_GRID, dtype=np.float32)
    dist = np.abs(np.abs(v)[..., None] - grid).astype(np.float32)
    j = np.argmin(dist, axis=-1).astype(np.uint8)
    sign = (blocks < 0).astype(np.uint8)
    codes = np.where((d > 0)[..., None], (sign << 3) | j, 0).astype(np.uint8).reshape(rows, cols)
    data = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return data, sb, g


def nv_dequantize(data: np.ndarray, scales: np.ndarray, g) -> np.ndarray:
    """x_hat = e2m1(code) * e4m3(scale of its 16-element block) * g, float64."""
    vals = e2m1_decode(mx_unpack_codes(data))
    rows, cols = vals.shape
    s = e4m3_decode(scales)[..., None]
    return (vals.reshape(rows, cols // NV_BLOCK, NV_BLOCK) * s).reshape(rows, cols) * float(np.float32(g))


def nv_gemm_fp4(a_data, a_scales, ga, w_data, w_scales, gw, rows=None) -> np.ndarray:
    """C = A @ W^T for NVFP4 operands, float64: for every output (m, n) and
    every 16-element K block b,

        dC = e4m3(sA[m, b]) * e4m3(sW[n, b]) * sum_{i<16} a[m, b, i] * w[n, b, i],

    C = ga * gw * sum_b dC (the block dot, then its two block scales, then
    the running sum, then the two tensor scales).  A ``[M, K/2]`` +
    ``[M, K/16]``, W ``[N, K/2]`` + ``[N, K/16]``, both K-contiguous; ``rows``
    optionally restricts the output to a subset of A's rows."""
    ca = e2m1_decode(mx_unpack_codes(a_data))
    cw = e2m1_decode(mx_unpack_codes(w_data))
    sa = e4m3_decode(a_scales)
    sw = e4m3_decode(w_scales)
    if rows is not None:
        ca, sa = ca[rows], sa[rows]
    m, k = ca.shape
    n = cw.shape[0]
    out = np.zeros((m, n), dtype=np.float64)
    for b in range(k // NV_BLOCK):
        sl = slice(b * NV_BLOCK, (b + 1) * NV_BLOCK)
        block_dot = ca[:, sl] @ cw[:, sl].T  # exact: small dyadic rationals
        out += block_dot * (sa[:, b][:, None] * sw[:, b][None, :])
    return out * (float(np.float32(ga)) * float(np.float32(gw)))


# --------------------------------------------------------------------------
# Block scales in the tensor cores' order.  This is not arithmetic of the
# pages: the block-scaled tensor cores (MXFP4 page §二.1-§二.2, the exponents
# added inside the dot product) take their scales in 512-byte chunks of 128
# rows x 4 blocks, and the CUDA library's GEMMs read scales stored in that
# order.  The library documents the layout with its re-layout call; this is a
# plain restatement of that definition, element by element, against which
# the call is checked byte for byte.
# --------------------------------------------------------------------------

TC_CHUNK = 512


def fp4_scales_tc(scales: np.ndarray, K: int, block: int) -> np.ndarray:
    """Row-major block scales uint8 ``[rows, K / block]`` (block 32: E8M0,
    block 16: E4M3) -> the flat tensor-core layout.

    Rows pad to a multiple of 256 and K to a multiple of 256 elements.  Row
    group g (rows 128 g .. 128 g + 127) holds ``kc`` chunks of 512 bytes,
    kc = (padded K / 256) * (256 / block / 4); chunk c of group g starts at
    byte 512 (g kc + c) and holds blocks 4 c .. 4 c + 3; the scale of row r,
    block b sits at byte 16 (r % 32) + 4 ((r // 32) % 4) + b % 4 of its chunk.
    Padding is 0x7F (2^0) for E8M0 and 0x00 for E4M3."""
    rows, nb = scales.shape
    assert K % block == 0 and nb == K // block
    steps = -(-K // 256)
    kc = steps * (256 // block) // 4
    groups = 2 * (-(-rows // 256))
    out = np.full(groups * kc * TC_CHUNK, 0x7F if block == 32 else 0x00, dtype=np.uint8)
    r = np.arange(rows)[:, None]
    b = np.arange(nb)[None, :]
    offset = ((r // 128) * kc + b // 4) * TC_CHUNK + 16 * (r % 32) + 4 * ((r // 32) % 4) + b % 4
    out[offset] = scales
    return out


# --------------------------------------------------------------------------
# Output rounding and the comparison rule
# --------------------------------------------------------------------------


def ulp(values: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the output type at each |value| (fp16, bf16 or fp32)."""
    v = np.abs(np.asarray(values, dtype=np.float64))
    mant_bits, min_exp = {"fp16": (10, -14), "bf16": (7, -126), "fp32": (23, -126)}[dtype]
    _, x = np.frexp(np.where(v > 0, v, np.finfo(np.float64).tiny))
    ex = np.maximum(x - 1, min_exp)  # floor(log2 |v|), clamped at the subnormal range
    return np.ldexp(1.0, (ex - mant_bits).astype(np.int64))


def gemm_tolerance(y_ref: np.ndarray, dtype: str, rel: float = 5e-3) -> np.ndarray:
    """Per-element bound: rel * max|y_ref| + 1 ulp of the output dtype at y_ref."""
    y_ref = np.asarray(y_ref, dtype=np.float64)
    amax = float(np.abs(y_ref).max()) if y_ref.size else 0.0
    return rel * amax + ulp(y_ref, dtype)
