"""Python binding of libwq, the GB300 fused dequantization GEMM library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libwq.so`` (built in-tree by ``build.py``).  The functions keep
the C ABI's names and take PyTorch CUDA tensors, which are used for device
memory and streams; pointers, leading dimensions and the current stream are
passed through ``ctypes``.  There is no CPU fallback: importing this package
without a built ``libwq.so`` raises, and every non-zero status raises
``WqError``.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwq.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "wq.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libwq.so is not built ({LIB_PATH} missing); run "
        "`python -c 'import __graft_entry__ as g; g.build()'` first")

lib = ctypes.CDLL(LIB_PATH)

WQ_OK = 0
WQ_ERR_INVALID_ARG = 1
WQ_ERR_MISALIGNED = 2
WQ_ERR_UNSUPPORTED = 3
WQ_ERR_WORKSPACE = 4
WQ_ERR_LAUNCH = 5
WQ_ERR_DEVICE = 6

WQ_OP_W4A16, WQ_OP_W8A16, WQ_OP_MX_QUANTIZE, WQ_OP_MX_GEMM, WQ_OP_FP8_GEMM, WQ_OP_NV_GEMM, WQ_OP_MX_GEMM_QA = range(7)
WQ_FP4_MX, WQ_FP4_NV = 0, 1

_i, _i64, _p, _sz, _f = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float
_SIGS = {
    "wq_gemm_w4a16": [_i, _i, _i, _p, _i64, _p, _i64, _p, _p, _i64, _p, _sz, _p],
    "wq_gemm_w8a16": [_i, _i, _i, _p, _i64, _p, _i64, _p, _p, _i64, _p, _sz, _p],
    "wq_gemm_w8a16_noalloc": [_i, _i, _i, _p, _i64, _p, _i64, _p, _p, _i64, _p],
    "wq_gemm_w4a16_grouped": [_i, _i, _i, _p, _i64, _p, _i64, _p, _p, _i, _p, _i64, _p, _sz, _p],
    "wq_gemm_w8a16_grouped": [_i, _i, _i, _p, _i64, _p, _i64, _p, _p, _i, _p, _i64, _p, _sz, _p],
    "mx_quantize_fp4": [_i, _i, _p, _i64, _p, _i64, _p, _i64, _p],
    "mx_gemm_fp4": [_i, _i, _i, _p, _i64, _p, _i64, _p, _i64, _p, _i64, _p, _i64, _p, _sz, _p],
    "fp8_gemm": [_i, _i, _i, _p, _i64, _p, _i64, _f, _f, _p, _i64, _p, _sz, _p],
    "nv_quantize_fp4": [_i, _i, _p, _i64, _p, _i64, _p, _i64, _p, _p],
    "nv_gemm_fp4": [_i, _i, _i, _p, _i64, _p, _i64, _p, _p, _i64, _p, _i64, _p, _p, _i64, _p, _sz, _p],
    "fp4_scales_tc_size": [_i, _i, _i],
    "fp4_scales_tc": [_i, _i, _i, _p, _i64, _p, _sz, _p],
    "mx_gemm_fp4_tc": [_i, _i, _i, _p, _i64, _p, _sz, _p, _i64, _p, _sz, _p, _i64, _p],
    "mx_gemm_fp4_qa": [_i, _i, _i, _p, _i64, _p, _i64, _p, _sz, _p, _i64, _p, _sz, _p],
    "nv_gemm_fp4_tc": [_i, _i, _i, _p, _i64, _p, _sz, _p, _p, _i64, _p, _sz, _p, _p, _i64, _p],
    "wq_workspace_size": [_i, _i, _i, _i],
    "wq_status_string": [_i],
    "wq_get_device_error": [_p, ctypes.POINTER(_i)],
    "wq_version": [],
    "wq_debug_set_wait_limit": [_i64],
    "wq_set_static_weights": [_i],
}


class WqProblem(ctypes.Structure):
    """The C ABI's wq_problem: one weight-only GEMM of a batched call."""
    _fields_ = [("M", _i), ("N", _i), ("K", _i), ("X", _p), ("ldx", _i64), ("W", _p), ("ldw", _i64),
                ("scales", _p), ("group_n", _i), ("Y", _p), ("ldy", _i64)]


WQ_MAX_BATCH = 8
_SIGS["wq_gemm_w4a16_batched"] = [_i, ctypes.POINTER(WqProblem), _p, _sz, _p]
_SIGS["wq_gemm_w8a16_batched"] = [_i, ctypes.POINTER(WqProblem), _p, _sz, _p]
_SIGS["wq_batched_workspace_size"] = [_i, _i, ctypes.POINTER(WqProblem)]
for _name, _args in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = _i
lib.wq_workspace_size.restype = _sz
lib.fp4_scales_tc_size.restype = _sz
lib.wq_batched_workspace_size.restype = _sz
lib.wq_status_string.restype = ctypes.c_char_p


class WqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib.wq_status_string(status).decode()}")


def header_functions(path: str = HEADER_PATH) -> list[str]:
    """Names of the functions include/wq.h declares."""
    with open(path) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?(?:int|size_t|char\s*\*|void)\s*\**\s*(\w+)\s*\(", text, flags=re.M)


def _check(status: int, where: str) -> None:
    if status != WQ_OK:
        raise WqError(status, where)


def _stream(stream):
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _require(cond, where, what):
    if not cond:
        raise WqError(WQ_ERR_INVALID_ARG, f"{where}: {what}")


def _on_gpu(where, *tensors):
    """Every given tensor lives in the memory of one CUDA device: the C ABI takes
    device pointers, and a host pointer handed to a kernel would fault."""
    dev = None
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise WqError(WQ_ERR_INVALID_ARG, f"{where}: tensors must be CUDA tensors")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise WqError(WQ_ERR_INVALID_ARG, f"{where}: tensors must be on one device")


_DTYPES: dict = {}


def _dtype(name):
    d = _DTYPES.get(name)
    if d is None:
        import torch

        d = _DTYPES[name] = getattr(torch, name)
    return d


def _kind(where, t, name, *, size=None, dtype=None):
    """Element size or dtype of one argument."""
    if t is None:
        return
    if dtype is not None and t.dtype is not _dtype(dtype):
        raise WqError(WQ_ERR_INVALID_ARG, f"{where}: {name} must be {dtype}, got {t.dtype}")
    if size is not None and t.element_size() != size:
        raise WqError(WQ_ERR_INVALID_ARG, f"{where}: {name} must have {size}-byte elements, got {t.dtype}")


def _weight_only_checks(where, bits, x, w, scales, y, zeros=None, group_n=1):
    _on_gpu(where, x, w, scales, y, zeros)
    _kind(where, x, "x", dtype="float16")
    _kind(where, w, "w", size=1)
    _kind(where, scales, "scales", dtype="float16")
    _kind(where, y, "y", dtype="float16")
    _kind(where, zeros, "zeros", size=1)
    if x.dim() != 2 or w.dim() != 2:
        raise WqError(WQ_ERR_INVALID_ARG, f"{where}: x and w must be 2-D")
    M, K = x.shape
    N = w.shape[1]
    if w.shape[0] * (2 if bits == 4 else 1) != K:
        raise WqError(WQ_ERR_INVALID_ARG, f"{where}: w has {w.shape[0]} rows; K = {K} needs "
                                          f"{K // 2 if bits == 4 else K}")
    if group_n < 1:
        raise WqError(WQ_ERR_INVALID_ARG, f"{where}: group_n must be >= 1")
    groups = -(-N // group_n)
    if scales.numel() < groups or (zeros is not None and zeros.numel() < groups):
        raise WqError(WQ_ERR_INVALID_ARG, f"{where}: scales and zeros need {groups} entries")
    if y is not None and (y.shape[0] != M or y.shape[1] != N):
        raise WqError(WQ_ERR_INVALID_ARG, f"{where}: y must be [{M}, {N}]")


def _ld(t):
    if t.dim() != 2 or t.stride(1) != 1:
        raise WqError(WQ_ERR_UNSUPPORTED, "matrices must be 2-D with unit inner stride")
    return t.stride(0)


def _ws(workspace):
    return (_ptr(workspace), workspace.numel() * workspace.element_size()) if workspace is not None else (_p(0), 0)


_WS_CACHE: dict = {}


def auto_workspace(op: int, M: int, N: int, K: int, device):
    """A device workspace of at least wq_workspace_size(op, M, N, K) bytes,
    zero-filled when created, cached per (device, stream) and grown on demand.
    Every successful call leaves its counter area zero again, so the cached
    buffer is reused as is; calls that share one must not overlap on the GPU
    (one cache entry per stream).  The FP4 GEMMs' scratch (rewritten scales,
    no counters) and the quantize-A GEMM's (its barrier words first, then
    scratch) have cache entries of their own, so that no call's scratch
    overwrites another's counters."""
    import torch

    tag = {WQ_OP_MX_GEMM: "fp4", WQ_OP_NV_GEMM: "fp4", WQ_OP_MX_GEMM_QA: "fp4qa"}.get(op, "counters")
    return _cached_workspace(wq_workspace_size(op, M, N, K), device, tag)


def _cached_workspace(need: int, device, tag: str = "counters"):
    import torch

    if need == 0:
        return None
    key = (tag, torch.device(device).index, torch.cuda.current_stream(device).cuda_stream)
    buf = _WS_CACHE.get(key)
    if buf is None or buf.numel() < need:
        buf = torch.zeros(max(need, 1 << 20), dtype=torch.uint8, device=device)
        _WS_CACHE[key] = buf
    return buf


def wq_gemm_w4a16(x, wq, scales, y=None, workspace=None, stream=None):
    """Y fp16 [M, N] = X fp16 [M, K] * ((unpack(wq [K/2, N]) - 8) * scales[N])."""
    import torch

    _weight_only_checks("wq_gemm_w4a16", 4, x, wq, scales, y)
    _on_gpu("wq_gemm_w4a16", x, workspace)
    M, K = x.shape
    N = wq.shape[1]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    if workspace is None:
        workspace = auto_workspace(WQ_OP_W4A16, M, N, K, x.device)
    wsp, wsb = _ws(workspace)
    _check(lib.wq_gemm_w4a16(M, N, K, _ptr(x), _ld(x), _ptr(wq), _ld(wq), _ptr(scales), _ptr(y), _ld(y),
                             wsp, wsb, _stream(stream)), "wq_gemm_w4a16")
    return y


def wq_gemm_w8a16(x, w, scales, y=None, workspace=None, stream=None):
    """Y fp16 [M, N] = X fp16 [M, K] * (w int8 [K, N] * scales[N])."""
    import torch

    _weight_only_checks("wq_gemm_w8a16", 8, x, w, scales, y)
    _on_gpu("wq_gemm_w8a16", x, workspace)
    M, K = x.shape
    N = w.shape[1]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    if workspace is None:
        workspace = auto_workspace(WQ_OP_W8A16, M, N, K, x.device)
    wsp, wsb = _ws(workspace)
    _check(lib.wq_gemm_w8a16(M, N, K, _ptr(x), _ld(x), _ptr(w), _ld(w), _ptr(scales), _ptr(y), _ld(y),
                             wsp, wsb, _stream(stream)), "wq_gemm_w8a16")
    return y


def wq_gemm_w8a16_noalloc(x, w, scales, y=None, stream=None):
    """wq_gemm_w8a16 with the library's built-in scratch instead of a workspace
    (for callers that cannot allocate device memory at call time)."""
    import torch

    _weight_only_checks("wq_gemm_w8a16_noalloc", 8, x, w, scales, y)
    M, K = x.shape
    N = w.shape[1]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _check(lib.wq_gemm_w8a16_noalloc(M, N, K, _ptr(x), _ld(x), _ptr(w), _ld(w), _ptr(scales), _ptr(y), _ld(y),
                                     _stream(stream)), "wq_gemm_w8a16_noalloc")
    return y


def _grouped(name, op, x, w, scales, zeros, group_n, y, workspace, stream):
    import torch

    _weight_only_checks(name, 4 if op == WQ_OP_W4A16 else 8, x, w, scales, y, zeros, int(group_n))
    _on_gpu(name, x, workspace)
    M, K = x.shape
    N = w.shape[1]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    if workspace is None:
        workspace = auto_workspace(op, M, N, K, x.device)
    wsp, wsb = _ws(workspace)
    _check(getattr(lib, name)(M, N, K, _ptr(x), _ld(x), _ptr(w), _ld(w), _ptr(scales), _ptr(zeros), int(group_n),
                              _ptr(y), _ld(y), wsp, wsb, _stream(stream)), name)
    return y


def wq_gemm_w4a16_grouped(x, wq, scales, zeros=None, group_n=1, y=None, workspace=None, stream=None):
    """Y = X * ((unpack(wq) - z[n // group_n]) * scales[n // group_n]); zeros uint8
    [ceil(N / group_n)] or None (zero point 8)."""
    return _grouped("wq_gemm_w4a16_grouped", WQ_OP_W4A16, x, wq, scales, zeros, group_n, y, workspace, stream)


def wq_gemm_w8a16_grouped(x, w, scales, zeros=None, group_n=1, y=None, workspace=None, stream=None):
    """Y = X * ((w - z[n // group_n]) * scales[n // group_n]); zeros int8
    [ceil(N / group_n)] or None (symmetric)."""
    return _grouped("wq_gemm_w8a16_grouped", WQ_OP_W8A16, x, w, scales, zeros, group_n, y, workspace, stream)


def _batched(name, bits, xs, ws, scales, ys, group_n, workspace, stream):
    import torch

    count = len(xs)
    if not (len(ws) == len(scales) == count) or (ys is not None and len(ys) != count):
        raise WqError(WQ_ERR_INVALID_ARG, f"{name}: xs, ws, scales (and ys) must have the same length")
    if not 1 <= count <= WQ_MAX_BATCH:
        raise WqError(WQ_ERR_INVALID_ARG, f"{name}: 1..{WQ_MAX_BATCH} problems per call")
    groups = list(group_n) if isinstance(group_n, (list, tuple)) else [group_n] * count
    _require(len(groups) == count, name, "one group_n per problem")
    probs = (WqProblem * count)()
    outs = []
    for i in range(count):
        x, w, sc = xs[i], ws[i], scales[i]
        y = ys[i] if ys is not None else None
        _weight_only_checks(name, bits, x, w, sc, y, None, int(groups[i]))
        _on_gpu(name, x, w, sc, y, xs[0], workspace)
        M, K = x.shape
        N = w.shape[1]
        if y is None:
            y = torch.empty((M, N), dtype=torch.float16, device=x.device)
        outs.append(y)
        probs[i] = WqProblem(M, N, K, x.data_ptr(), _ld(x), w.data_ptr(), _ld(w), sc.data_ptr(), int(groups[i]),
                             y.data_ptr(), _ld(y))
    op = WQ_OP_W4A16 if bits == 4 else WQ_OP_W8A16
    if workspace is None:
        workspace = _cached_workspace(int(lib.wq_batched_workspace_size(op, count, probs)), xs[0].device)
    wsp, wsb = _ws(workspace)
    _check(getattr(lib, name)(count, probs, wsp, wsb, _stream(stream)), name)
    return outs


def wq_gemm_w4a16_batched(xs, wqs, scales, ys=None, group_n=1, workspace=None, stream=None):
    """Several INT4 weight-only GEMMs (M <= 64 each) in one launch: for every
    i, ys[i] = xs[i] * ((unpack(wqs[i]) - 8) * scales[i][n // group_n]).
    Returns the list of outputs."""
    return _batched("wq_gemm_w4a16_batched", 4, xs, wqs, scales, ys, group_n, workspace, stream)


def wq_gemm_w8a16_batched(xs, ws, scales, ys=None, group_n=1, workspace=None, stream=None):
    """Several INT8 weight-only GEMMs (M <= 64 each) in one launch: for every
    i, ys[i] = xs[i] * (ws[i] * scales[i][n // group_n]).  Returns the list of
    outputs."""
    return _batched("wq_gemm_w8a16_batched", 8, xs, ws, scales, ys, group_n, workspace, stream)


def mx_quantize_fp4(src, data=None, scales=None, stream=None):
    """fp32 [R, C] -> (uint8 data [R, C/2], uint8 E8M0 scales [R, C/32])."""
    import torch

    where = "mx_quantize_fp4"
    _on_gpu(where, src, data, scales)
    _kind(where, src, "src", dtype="float32")
    _kind(where, data, "data", size=1)
    _kind(where, scales, "scales", size=1)
    _require(src.dim() == 2, where, "src must be 2-D")
    R, C = src.shape
    _require(data is None or tuple(data.shape) == (R, C // 2), where, f"data must be [{R}, {C // 2}]")
    _require(scales is None or tuple(scales.shape) == (R, C // 32), where, f"scales must be [{R}, {C // 32}]")
    if data is None:
        data = torch.empty((R, C // 2), dtype=torch.uint8, device=src.device)
    if scales is None:
        scales = torch.empty((R, C // 32), dtype=torch.uint8, device=src.device)
    _check(lib.mx_quantize_fp4(R, C, _ptr(src), _ld(src), _ptr(data), _ld(data), _ptr(scales), _ld(scales),
                               _stream(stream)), "mx_quantize_fp4")
    return data, scales


def mx_gemm_fp4(a, sa, w, sw, c=None, workspace=None, stream=None):
    """C fp32 [M, N] = A * W^T for MXFP4 operands (data [rows, K/2] + scales [rows, K/32])."""
    import torch

    where = "mx_gemm_fp4"
    _on_gpu(where, a, sa, w, sw, c, workspace)
    for t, n in ((a, "a"), (sa, "sa"), (w, "w"), (sw, "sw")):
        _kind(where, t, n, size=1)
        _require(t.dim() == 2, where, f"{n} must be 2-D")
    _kind(where, c, "c", dtype="float32")
    M, N, K = a.shape[0], w.shape[0], a.shape[1] * 2
    _require(w.shape[1] * 2 == K, where, "a and w must have the same K")
    _require(tuple(sa.shape) == (M, K // 32) and tuple(sw.shape) == (N, K // 32), where,
             f"scales must be [{M}, {K // 32}] and [{N}, {K // 32}]")
    _require(c is None or tuple(c.shape) == (M, N), where, f"c must be [{M}, {N}]")
    if c is None:
        c = torch.empty((M, N), dtype=torch.float32, device=a.device)
    if workspace is None:
        workspace = auto_workspace(WQ_OP_MX_GEMM, M, N, K, a.device)
    wsp, wsb = _ws(workspace)
    _check(lib.mx_gemm_fp4(M, N, K, _ptr(a), _ld(a), _ptr(sa), _ld(sa), _ptr(w), _ld(w), _ptr(sw), _ld(sw),
                           _ptr(c), _ld(c), wsp, wsb, _stream(stream)), "mx_gemm_fp4")
    return c


def set_static_weights(enable: bool) -> bool:
    """wq_set_static_weights: promise that weight and scale arrays are not
    written by any kernel still running when a weight-only call launches, so
    that the decode kernels may load their first weight boxes early.
    Returns the previous setting."""
    return bool(lib.wq_set_static_weights(1 if enable else 0))


def mx_gemm_fp4_qa(a, w, sw_tc, c=None, workspace=None, stream=None):
    """C fp32 [M, N] = MXFP4(A) * W^T with A fp32 [M, K] quantized inside the
    GEMM launch; W uint8 [N, K/2] with its scales in the tensor-core layout
    (fp4_scales_tc)."""
    import torch

    where = "mx_gemm_fp4_qa"
    _on_gpu(where, a, w, sw_tc, c, workspace)
    _kind(where, a, "a", dtype="float32")
    _kind(where, w, "w", size=1)
    _kind(where, sw_tc, "sw_tc", size=1)
    _kind(where, c, "c", dtype="float32")
    _require(a.dim() == 2 and w.dim() == 2, where, "a and w must be 2-D")
    _require(sw_tc.is_contiguous(), where, "tensor-core scales must be contiguous")
    M, K, N = a.shape[0], a.shape[1], w.shape[0]
    _require(w.shape[1] * 2 == K, where, "w must be [N, K/2]")
    _require(c is None or tuple(c.shape) == (M, N), where, f"c must be [{M}, {N}]")
    if c is None:
        c = torch.empty((M, N), dtype=torch.float32, device=a.device)
    if workspace is None:
        workspace = auto_workspace(WQ_OP_MX_GEMM_QA, M, N, K, a.device)
    wsp, wsb = _ws(workspace)
    _check(lib.mx_gemm_fp4_qa(M, N, K, _ptr(a), _ld(a), _ptr(w), _ld(w), _ptr(sw_tc), sw_tc.numel(), _ptr(c), _ld(c),
                              wsp, wsb, _stream(stream)), where)
    return c


def fp4_scales_tc(scales, K, fmt=WQ_FP4_MX, out=None, stream=None):
    """Block scales uint8 [rows, K / block] -> the tensor-core layout (a flat
    uint8 tensor of fp4_scales_tc_size bytes) that mx_gemm_fp4_tc and
    nv_gemm_fp4_tc read."""
    import torch

    where = "fp4_scales_tc"
    _on_gpu(where, scales, out)
    _kind(where, scales, "scales", size=1)
    _require(scales.dim() == 2, where, "scales must be 2-D")
    block = 16 if fmt == WQ_FP4_NV else 32
    rows = scales.shape[0]
    _require(K % block == 0 and scales.shape[1] == K // block, where, f"scales must be [rows, {K // block}]")
    need = int(lib.fp4_scales_tc_size(fmt, rows, K))
    if out is None:
        out = torch.empty(max(need, 1), dtype=torch.uint8, device=scales.device)
    _kind(where, out, "out", size=1)
    _check(lib.fp4_scales_tc(fmt, rows, K, _ptr(scales), _ld(scales), _ptr(out), out.numel(), _stream(stream)), where)
    return out


def mx_gemm_fp4_tc(a, sa_tc, w, sw_tc, c=None, stream=None):
    """mx_gemm_fp4 with both scale arrays already in the tensor-core layout
    (fp4_scales_tc): C fp32 [M, N] = A * W^T."""
    import torch

    where = "mx_gemm_fp4_tc"
    _on_gpu(where, a, sa_tc, w, sw_tc, c)
    for t, n in ((a, "a"), (sa_tc, "sa_tc"), (w, "w"), (sw_tc, "sw_tc")):
        _kind(where, t, n, size=1)
    _require(a.dim() == 2 and w.dim() == 2, where, "a and w must be 2-D")
    _require(sa_tc.is_contiguous() and sw_tc.is_contiguous(), where, "tensor-core scales must be contiguous")
    _kind(where, c, "c", dtype="float32")
    M, N, K = a.shape[0], w.shape[0], a.shape[1] * 2
    _require(w.shape[1] * 2 == K, where, "a and w must have the same K")
    _require(c is None or tuple(c.shape) == (M, N), where, f"c must be [{M}, {N}]")
    if c is None:
        c = torch.empty((M, N), dtype=torch.float32, device=a.device)
    _check(lib.mx_gemm_fp4_tc(M, N, K, _ptr(a), _ld(a), _ptr(sa_tc), sa_tc.numel(), _ptr(w), _ld(w), _ptr(sw_tc),
                              sw_tc.numel(), _ptr(c), _ld(c), _stream(stream)), where)
    return c


def nv_quantize_fp4(src, data=None, scales=None, tensor_scale=None, stream=None):
    """fp32 [R, C] -> (uint8 data [R, C/2], uint8 E4M3 scales [R, C/16], fp32
    tensor scale [1] on the device)."""
    import torch

    where = "nv_quantize_fp4"
    _on_gpu(where, src, data, scales, tensor_scale)
    _kind(where, src, "src", dtype="float32")
    _kind(where, data, "data", size=1)
    _kind(where, scales, "scales", size=1)
    _kind(where, tensor_scale, "tensor_scale", dtype="float32")
    _require(src.dim() == 2, where, "src must be 2-D")
    R, C = src.shape
    _require(data is None or tuple(data.shape) == (R, C // 2), where, f"data must be [{R}, {C // 2}]")
    _require(scales is None or tuple(scales.shape) == (R, C // 16), where, f"scales must be [{R}, {C // 16}]")
    _require(tensor_scale is None or tensor_scale.numel() >= 1, where, "tensor_scale needs one element")
    if data is None:
        data = torch.empty((R, C // 2), dtype=torch.uint8, device=src.device)
    if scales is None:
        scales = torch.empty((R, C // 16), dtype=torch.uint8, device=src.device)
    if tensor_scale is None:
        tensor_scale = torch.empty(1, dtype=torch.float32, device=src.device)
    _check(lib.nv_quantize_fp4(R, C, _ptr(src), _ld(src), _ptr(data), _ld(data), _ptr(scales), _ld(scales),
                               _ptr(tensor_scale), _stream(stream)), where)
    return data, scales, tensor_scale


def nv_gemm_fp4(a, sa, ga, w, sw, gw, c=None, workspace=None, stream=None):
    """C fp32 [M, N] = A * W^T for NVFP4 operands (data [rows, K/2], E4M3
    scales [rows, K/16], tensor scale [1] on the device)."""
    import torch

    where = "nv_gemm_fp4"
    _on_gpu(where, a, sa, ga, w, sw, gw, c)
    for t, n in ((a, "a"), (sa, "sa"), (w, "w"), (sw, "sw")):
        _kind(where, t, n, size=1)
        _require(t.dim() == 2, where, f"{n} must be 2-D")
    for t, n in ((ga, "ga"), (gw, "gw")):
        _kind(where, t, n, dtype="float32")
    _kind(where, c, "c", dtype="float32")
    M, N, K = a.shape[0], w.shape[0], a.shape[1] * 2
    _require(w.shape[1] * 2 == K, where, "a and w must have the same K")
    _require(tuple(sa.shape) == (M, K // 16) and tuple(sw.shape) == (N, K // 16), where,
             f"scales must be [{M}, {K // 16}] and [{N}, {K // 16}]")
    _require(c is None or tuple(c.shape) == (M, N), where, f"c must be [{M}, {N}]")
    if c is None:
        c = torch.empty((M, N), dtype=torch.float32, device=a.device)
    if workspace is None:
        workspace = auto_workspace(WQ_OP_NV_GEMM, M, N, K, a.device)
    wsp, wsb = _ws(workspace)
    _check(lib.nv_gemm_fp4(M, N, K, _ptr(a), _ld(a), _ptr(sa), _ld(sa), _ptr(ga), _ptr(w), _ld(w), _ptr(sw), _ld(sw),
                           _ptr(gw), _ptr(c), _ld(c), wsp, wsb, _stream(stream)), where)
    return c


def nv_gemm_fp4_tc(a, sa_tc, ga, w, sw_tc, gw, c=None, stream=None):
    """nv_gemm_fp4 with both E4M3 scale arrays already in the tensor-core
    layout (fp4_scales_tc with WQ_FP4_NV)."""
    import torch

    where = "nv_gemm_fp4_tc"
    _on_gpu(where, a, sa_tc, ga, w, sw_tc, gw, c)
    for t, n in ((a, "a"), (sa_tc, "sa_tc"), (w, "w"), (sw_tc, "sw_tc")):
        _kind(where, t, n, size=1)
    _require(a.dim() == 2 and w.dim() == 2, where, "a and w must be 2-D")
    _require(sa_tc.is_contiguous() and sw_tc.is_contiguous(), where, "tensor-core scales must be contiguous")
    for t, n in ((ga, "ga"), (gw, "gw")):
        _kind(where, t, n, dtype="float32")
    _kind(where, c, "c", dtype="float32")
    M, N, K = a.shape[0], w.shape[0], a.shape[1] * 2
    _require(w.shape[1] * 2 == K, where, "a and w must have the same K")
    _require(c is None or tuple(c.shape) == (M, N), where, f"c must be [{M}, {N}]")
    if c is None:
        c = torch.empty((M, N), dtype=torch.float32, device=a.device)
    _check(lib.nv_gemm_fp4_tc(M, N, K, _ptr(a), _ld(a), _ptr(sa_tc), sa_tc.numel(), _ptr(ga), _ptr(w), _ld(w),
                              _ptr(sw_tc), sw_tc.numel(), _ptr(gw), _ptr(c), _ld(c), _stream(stream)), where)
    return c


def fp8_gemm(a, b, scale_a, scale_b, c=None, workspace=None, stream=None):
    """C bf16 [M, N] = (A e4m3 [M, K] * B e4m3 [K, N]) * scale_a * scale_b."""
    import torch

    where = "fp8_gemm"
    _on_gpu(where, a, b, c, workspace)
    _kind(where, a, "a", size=1)
    _kind(where, b, "b", size=1)
    _kind(where, c, "c", dtype="bfloat16")
    _require(a.dim() == 2 and b.dim() == 2 and b.shape[0] == a.shape[1], where, "a [M, K] and b [K, N] needed")
    M, K = a.shape
    N = b.shape[1]
    _require(c is None or tuple(c.shape) == (M, N), where, f"c must be [{M}, {N}]")
    if c is None:
        c = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    if workspace is None:
        workspace = auto_workspace(WQ_OP_FP8_GEMM, M, N, K, a.device)
    wsp, wsb = _ws(workspace)
    _check(lib.fp8_gemm(M, N, K, _ptr(a), _ld(a), _ptr(b), _ld(b), float(scale_a), float(scale_b), _ptr(c), _ld(c),
                        wsp, wsb, _stream(stream)), "fp8_gemm")
    return c


def wq_workspace_size(op: int, M: int, N: int, K: int) -> int:
    return int(lib.wq_workspace_size(op, M, N, K))


def wq_status_string(status: int) -> str:
    return lib.wq_status_string(status).decode()


def wq_get_device_error(stream=None) -> tuple[int, int]:
    site = _i(0)
    st = lib.wq_get_device_error(_stream(stream), ctypes.byref(site))
    return st, site.value


def wq_debug_set_wait_limit(ns: int) -> None:
    """Testing hook: shorten (ns > 0) or restore (ns <= 0) the limit of the
    skinny kernels' bounded waits."""
    _check(lib.wq_debug_set_wait_limit(int(ns)), "wq_debug_set_wait_limit")


def wq_version() -> int:
    return int(lib.wq_version())
