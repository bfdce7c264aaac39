"""The C ABI library builds, loads, exports every function include/wq.h
declares, and rejects bad arguments on the host before any launch.  Nothing
here touches a GPU: the validation paths return before the first CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def wq():
    import __graft_entry__

    __graft_entry__.build()
    import bit_quantized_gemm_dequant_gb300 as mod

    return mod


def test_header_declares_the_five_entry_points(wq):
    names = wq.header_functions()
    for n in ("wq_gemm_w4a16", "wq_gemm_w8a16", "mx_quantize_fp4", "mx_gemm_fp4", "fp8_gemm",
              "wq_gemm_w4a16_grouped", "wq_gemm_w8a16_grouped",
              "wq_workspace_size", "wq_status_string", "wq_get_device_error", "wq_version"):
        assert n in names


def test_library_exports_every_declared_symbol(wq):
    out = subprocess.run(["nm", "-D", "--defined-only", wq.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in wq.header_functions():
        assert name in exported, name
        assert getattr(wq.lib, name) is not None


def test_status_strings(wq):
    for code in range(7):
        assert wq.wq_status_string(code).startswith("WQ_")
    assert wq.wq_status_string(99) == "WQ_ERR_UNKNOWN"
    assert wq.wq_version() >= 200


FAKE = 0x10000  # never dereferenced: validation returns first


def _w4(wq, M=4, N=64, K=64, X=FAKE, ldx=64, W=FAKE, ldw=64, S=FAKE, Y=FAKE, ldy=64):
    return wq.lib.wq_gemm_w4a16(M, N, K, X, ldx, W, ldw, S, Y, ldy, None, 0, None)


def test_weight_only_validation(wq):
    assert _w4(wq, M=-1) == wq.WQ_ERR_INVALID_ARG
    assert _w4(wq, K=63) == wq.WQ_ERR_INVALID_ARG          # INT4 packs two codes per byte
    assert _w4(wq, X=0) == wq.WQ_ERR_INVALID_ARG
    assert _w4(wq, ldx=32) == wq.WQ_ERR_INVALID_ARG        # ldx < K
    assert _w4(wq, ldy=32) == wq.WQ_ERR_INVALID_ARG
    assert _w4(wq, ldw=32) == wq.WQ_ERR_INVALID_ARG        # ldw < N
    assert _w4(wq, X=FAKE + 2) == wq.WQ_ERR_MISALIGNED
    assert _w4(wq, ldw=72) == wq.WQ_ERR_MISALIGNED
    assert _w4(wq, ldx=68) == wq.WQ_ERR_MISALIGNED
    assert _w4(wq, M=0) == wq.WQ_OK and _w4(wq, N=0) == wq.WQ_OK   # empty: no launch
    assert wq.lib.wq_gemm_w8a16(4, 64, 63, FAKE, 64, FAKE, 64, FAKE, FAKE, 64, None, 0, None) == wq.WQ_ERR_UNSUPPORTED


def _g(wq, bits=4, M=4, N=64, K=64, X=FAKE, ldx=64, W=FAKE, ldw=64, S=FAKE, Z=FAKE, G=8, Y=FAKE, ldy=64):
    fn = wq.lib.wq_gemm_w4a16_grouped if bits == 4 else wq.lib.wq_gemm_w8a16_grouped
    return fn(M, N, K, X, ldx, W, ldw, S, Z, G, Y, ldy, None, 0, None)


def test_grouped_validation(wq):
    for bits in (4, 8):
        assert _g(wq, bits, G=0) == wq.WQ_ERR_INVALID_ARG      # a group has at least one column
        assert _g(wq, bits, G=-3) == wq.WQ_ERR_INVALID_ARG
        assert _g(wq, bits, X=0) == wq.WQ_ERR_INVALID_ARG
        assert _g(wq, bits, S=0) == wq.WQ_ERR_INVALID_ARG
        assert _g(wq, bits, ldw=32) == wq.WQ_ERR_INVALID_ARG
        assert _g(wq, bits, X=FAKE + 2) == wq.WQ_ERR_MISALIGNED
        assert _g(wq, bits, M=0) == wq.WQ_OK and _g(wq, bits, N=0) == wq.WQ_OK
    assert _g(wq, 4, K=63) == wq.WQ_ERR_INVALID_ARG
    assert _g(wq, 8, K=63) == wq.WQ_ERR_UNSUPPORTED


def test_mx_and_fp8_validation(wq):
    L = wq.lib
    assert L.mx_quantize_fp4(4, 48, FAKE, 48, FAKE, 24, FAKE, 2, None) == wq.WQ_ERR_INVALID_ARG  # cols % 32
    assert L.mx_quantize_fp4(4, 64, FAKE + 4, 64, FAKE, 32, FAKE, 2, None) == wq.WQ_ERR_MISALIGNED
    assert L.mx_quantize_fp4(0, 64, 0, 64, 0, 32, 0, 2, None) == wq.WQ_OK
    assert L.mx_gemm_fp4(8, 8, 48, FAKE, 32, FAKE, 2, FAKE, 32, FAKE, 2, FAKE, 8, None, 0, None) == wq.WQ_ERR_INVALID_ARG
    assert L.mx_gemm_fp4(8, 8, 64, FAKE, 40, FAKE, 2, FAKE, 32, FAKE, 2, FAKE, 8, None, 0, None) == wq.WQ_ERR_MISALIGNED
    assert L.fp8_gemm(8, 8, 32, 0, 32, FAKE, 16, ctypes.c_float(1), ctypes.c_float(1), FAKE, 8, None, 0, None) \
        == wq.WQ_ERR_INVALID_ARG
    assert L.fp8_gemm(8, 8, 32, FAKE, 40, FAKE, 16, ctypes.c_float(1), ctypes.c_float(1), FAKE, 8, None, 0, None) \
        == wq.WQ_ERR_MISALIGNED
    assert L.fp8_gemm(0, 8, 32, 0, 32, 0, 16, ctypes.c_float(1), ctypes.c_float(1), 0, 8, None, 0, None) == wq.WQ_OK


def test_fp4_tensor_core_scale_validation(wq):
    """Sizes of the tensor-core scale layout (worked by hand: MXFP4 300 rows,
    K 1024 -> 4 row groups x 8 chunks x 512 bytes; 520 rows -> 6 groups), and
    argument checks that return before any CUDA call."""
    L = wq.lib
    MX, NV = wq.WQ_FP4_MX, wq.WQ_FP4_NV
    assert L.fp4_scales_tc_size(MX, 300, 1024) == 4 * 8 * 512
    assert L.fp4_scales_tc_size(MX, 520, 1024) == 6 * 8 * 512
    assert L.fp4_scales_tc_size(NV, 5, 80) == 2 * 4 * 512
    assert L.fp4_scales_tc_size(MX, 8, 48) == 0 and L.fp4_scales_tc_size(2, 8, 64) == 0
    # the row-major GEMMs' workspace: A's part rounded up to 256 bytes, then W's
    assert L.wq_workspace_size(wq.WQ_OP_MX_GEMM, 300, 520, 1024) == 4 * 8 * 512 + 6 * 8 * 512
    assert L.wq_workspace_size(wq.WQ_OP_NV_GEMM, 300, 520, 1024) == 4 * 16 * 512 + 6 * 16 * 512
    assert L.fp4_scales_tc(2, 8, 64, FAKE, 2, FAKE, 1 << 20, None) == wq.WQ_ERR_INVALID_ARG       # format
    assert L.fp4_scales_tc(MX, 8, 48, FAKE, 2, FAKE, 1 << 20, None) == wq.WQ_ERR_INVALID_ARG      # K % 32
    assert L.fp4_scales_tc(MX, 8, 64, FAKE, 1, FAKE, 1 << 20, None) == wq.WQ_ERR_INVALID_ARG      # lds < K / 32
    assert L.fp4_scales_tc(MX, 8, 64, FAKE, 2, FAKE, 100, None) == wq.WQ_ERR_INVALID_ARG          # out too small
    assert L.fp4_scales_tc(MX, 8, 64, FAKE, 2, FAKE + 8, 1 << 20, None) == wq.WQ_ERR_MISALIGNED
    assert L.fp4_scales_tc(MX, 0, 64, 0, 2, 0, 0, None) == wq.WQ_OK
    # a scale buffer smaller than the layout of its operand
    assert L.mx_gemm_fp4_tc(8, 8, 64, FAKE, 32, FAKE, 100, FAKE, 32, FAKE, 1 << 20, FAKE, 8, None) \
        == wq.WQ_ERR_INVALID_ARG
    assert L.nv_gemm_fp4_tc(8, 8, 64, FAKE, 32, FAKE, 1 << 20, FAKE, FAKE, 32, FAKE, 100, FAKE, FAKE, 8, None) \
        == wq.WQ_ERR_INVALID_ARG
    # row-major scales need the workspace
    assert L.mx_gemm_fp4(8, 8, 64, FAKE, 32, FAKE, 2, FAKE, 32, FAKE, 2, FAKE, 8, None, 0, None) == wq.WQ_ERR_WORKSPACE
    assert L.nv_gemm_fp4(8, 8, 64, FAKE, 32, FAKE, 4, FAKE, FAKE, 32, FAKE, 4, FAKE, FAKE, 8, None, 0, None) \
        == wq.WQ_ERR_WORKSPACE


def test_problem_struct_matches_header(wq, tmp_path):
    """The binding's wq_problem has the C layout of include/wq.h (checked with
    the host C compiler)."""
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "wq.h"\n'
                   'int main(void) { printf("%zu %zu %zu %zu %zu", sizeof(wq_problem), offsetof(wq_problem, X), '
                   'offsetof(wq_problem, scales), offsetof(wq_problem, group_n), offsetof(wq_problem, ldy)); '
                   'return 0; }\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    P = wq.WqProblem
    assert got == [ctypes.sizeof(P), P.X.offset, P.scales.offset, P.group_n.offset, P.ldy.offset]


def _prob(wq, M=4, N=64, K=64, X=FAKE, ldx=64, W=FAKE, ldw=64, S=FAKE, G=1, Y=FAKE, ldy=64):
    return wq.WqProblem(M, N, K, X, ldx, W, ldw, S, G, Y, ldy)


def test_batched_validation(wq):
    L = wq.lib
    for fn in (L.wq_gemm_w4a16_batched, L.wq_gemm_w8a16_batched):
        one = (wq.WqProblem * 1)(_prob(wq))
        assert fn(0, one, None, 0, None) == wq.WQ_ERR_INVALID_ARG          # no problems
        nine = (wq.WqProblem * 9)(*[_prob(wq)] * 9)
        assert fn(9, nine, None, 0, None) == wq.WQ_ERR_INVALID_ARG         # beyond WQ_MAX_BATCH
        assert fn(1, None, None, 0, None) == wq.WQ_ERR_INVALID_ARG
        for bad, code in ((dict(M=65), wq.WQ_ERR_UNSUPPORTED),             # the skinny path ends at M = 64
                          (dict(G=0), wq.WQ_ERR_INVALID_ARG),
                          (dict(X=0), wq.WQ_ERR_INVALID_ARG),
                          (dict(ldw=32), wq.WQ_ERR_INVALID_ARG),
                          (dict(X=FAKE + 2), wq.WQ_ERR_MISALIGNED),
                          (dict(ldy=68), wq.WQ_ERR_MISALIGNED)):
            two = (wq.WqProblem * 2)(_prob(wq), _prob(wq, **bad))
            assert fn(2, two, None, 0, None) == code, bad
        empty = (wq.WqProblem * 2)(_prob(wq, M=0), _prob(wq, N=0))
        assert fn(2, empty, None, 0, None) == wq.WQ_OK                       # nothing to launch
    odd = (wq.WqProblem * 1)(_prob(wq, K=63))
    assert L.wq_gemm_w4a16_batched(1, odd, None, 0, None) == wq.WQ_ERR_INVALID_ARG
    assert L.wq_gemm_w8a16_batched(1, odd, None, 0, None) == wq.WQ_ERR_UNSUPPORTED
    assert L.wq_batched_workspace_size(wq.WQ_OP_W8A16, 1, odd) == 0


def test_workspace_query(wq):
    for op in range(5):
        assert wq.wq_workspace_size(op, 16, 4096, 4096) >= 0


def test_product_does_not_import_oracle():
    pkg = os.path.join(ROOT, "bit_quantized_gemm_dequant_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cuh")):
                with open(os.path.join(dirpath, f)) as fh:
                    text = fh.read()
                assert not re.search(r"(^|\s)(import|from)\s+oracle", text), f


def test_binding_refuses_host_tensors(wq):
    """The C ABI takes device pointers; the binding refuses CPU tensors before
    any call (a host pointer in a kernel would fault)."""
    import torch

    x = torch.zeros((4, 64), dtype=torch.float16)
    s = torch.zeros(64, dtype=torch.float16)
    calls = [
        lambda: wq.wq_gemm_w4a16(x, torch.zeros((32, 64), dtype=torch.uint8), s),
        lambda: wq.wq_gemm_w8a16(x, torch.zeros((64, 64), dtype=torch.int8), s),
        lambda: wq.wq_gemm_w8a16_grouped(x, torch.zeros((64, 64), dtype=torch.int8), s, None, 4),
        lambda: wq.mx_quantize_fp4(torch.zeros((4, 64))),
        lambda: wq.fp8_gemm(torch.zeros((4, 8), dtype=torch.uint8), torch.zeros((8, 16), dtype=torch.uint8), 1.0, 1.0),
    ]
    for call in calls:
        with pytest.raises(wq.WqError) as ei:
            call()
        assert ei.value.status == wq.WQ_ERR_INVALID_ARG


def test_binding_shape_and_dtype_checks(wq, monkeypatch):
    """Shapes and element types are checked against each other before any call
    (a short scales or zeros array would be read past its end)."""
    import torch

    monkeypatch.setattr(wq, "_on_gpu", lambda where, *t: None)
    x = torch.zeros((4, 64), dtype=torch.float16)
    w4 = torch.zeros((32, 80), dtype=torch.uint8)
    w8 = torch.zeros((64, 80), dtype=torch.int8)
    s = torch.zeros(80, dtype=torch.float16)
    ok = [(4, x, w4, s, None, None, 1), (8, x, w8, s, None, None, 1),
          (8, x, w8, torch.zeros(3, dtype=torch.float16), None, torch.zeros(3, dtype=torch.int8), 32)]
    for bits, xx, w, sc, y, z, g in ok:
        wq._weight_only_checks("t", bits, xx, w, sc, y, z, g)
    bad = [
        (4, x, w8, s, None, None, 1),                                  # INT8-shaped weights for INT4
        (8, x.float(), w8, s, None, None, 1),                          # fp32 activations
        (8, x, w8, torch.zeros(79, dtype=torch.float16), None, None, 1),  # one scale short
        (8, x, w8, torch.zeros(2, dtype=torch.float16), None, None, 32),  # 80 columns need 3 groups
        (8, x, w8, torch.zeros(3, dtype=torch.float16), None, torch.zeros(2, dtype=torch.int8), 32),
        (8, x, w8, s, torch.zeros((4, 64), dtype=torch.float16), None, 1),  # y of the wrong shape
        (8, x, w8, s, None, None, 0),                                  # empty groups
    ]
    for bits, xx, w, sc, y, z, g in bad:
        with pytest.raises(wq.WqError):
            wq._weight_only_checks("t", bits, xx, w, sc, y, z, g)


class _FakeLib:
    """Records the C calls a binding function makes (no CUDA needed)."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if name == "wq_status_string":
            return lambda status: b"WQ_STATUS"

        def call(*args):
            self.calls.append((name, args))
            return 0
        return call


def test_binding_functions_marshal_without_cuda(wq, monkeypatch):
    """Every binding function runs its checks and marshals its call: a fake
    library stands in for libwq.so and host tensors stand in for device ones."""
    import ctypes

    import torch

    fake = _FakeLib()
    monkeypatch.setattr(wq, "lib", fake)
    monkeypatch.setattr(wq, "_on_gpu", lambda where, *t: None)
    monkeypatch.setattr(wq, "_stream", lambda stream: ctypes.c_void_p(0))
    monkeypatch.setattr(wq, "auto_workspace", lambda *a, **k: None)
    x = torch.zeros((4, 64), dtype=torch.float16)
    s = torch.zeros(96, dtype=torch.float16)
    w4 = torch.zeros((32, 96), dtype=torch.uint8)
    w8 = torch.zeros((64, 96), dtype=torch.int8)
    assert wq.wq_gemm_w4a16(x, w4, s).shape == (4, 96)
    assert wq.wq_gemm_w8a16(x, w8, s).shape == (4, 96)
    assert wq.wq_gemm_w8a16_noalloc(x, w8, s).shape == (4, 96)
    assert wq.wq_gemm_w4a16_grouped(x, w4, s[:3], torch.zeros(3, dtype=torch.uint8), 32).shape == (4, 96)
    assert wq.wq_gemm_w8a16_grouped(x, w8, s[:3], None, 32).shape == (4, 96)
    d, e = wq.mx_quantize_fp4(torch.zeros((4, 64)))
    assert d.shape == (4, 32) and e.shape == (4, 2)
    c = wq.mx_gemm_fp4(d, e, torch.zeros((8, 32), dtype=torch.uint8), torch.zeros((8, 2), dtype=torch.uint8))
    assert c.shape == (4, 8) and c.dtype == torch.float32
    c8 = wq.fp8_gemm(torch.zeros((4, 64), dtype=torch.uint8), torch.zeros((64, 16), dtype=torch.uint8), 1.0, 2.0)
    assert c8.shape == (4, 16) and c8.dtype == torch.bfloat16
    sa_tc = wq.fp4_scales_tc(e, 64)
    ct = wq.mx_gemm_fp4_tc(d, sa_tc, torch.zeros((8, 32), dtype=torch.uint8), sa_tc)
    assert ct.shape == (4, 8) and ct.dtype == torch.float32
    g1 = torch.ones(1, dtype=torch.float32)
    e16 = torch.zeros((4, 4), dtype=torch.uint8)
    cn = wq.nv_gemm_fp4(d, e16, g1, torch.zeros((8, 32), dtype=torch.uint8), torch.zeros((8, 4), dtype=torch.uint8), g1)
    cnt = wq.nv_gemm_fp4_tc(d, sa_tc, g1, torch.zeros((8, 32), dtype=torch.uint8), sa_tc, g1)
    assert cn.shape == cnt.shape == (4, 8)
    names = [n for n, _ in fake.calls]
    assert names == ["wq_gemm_w4a16", "wq_gemm_w8a16", "wq_gemm_w8a16_noalloc", "wq_gemm_w4a16_grouped",
                     "wq_gemm_w8a16_grouped", "mx_quantize_fp4", "mx_gemm_fp4", "fp8_gemm",
                     "fp4_scales_tc_size", "fp4_scales_tc", "mx_gemm_fp4_tc", "nv_gemm_fp4", "nv_gemm_fp4_tc"]
    argc = {n: len(a) for n, a in fake.calls}
    for n, sig in wq._SIGS.items():
        if n in argc:
            assert argc[n] == len(sig), n
    with pytest.raises(wq.WqError):
        wq.mx_gemm_fp4(d, e, torch.zeros((8, 30), dtype=torch.uint8), torch.zeros((8, 2), dtype=torch.uint8))


def test_shapes_beyond_the_grid_limits_are_refused(wq):
    """Validation returns before any CUDA call, so fake pointers are never used."""
    L = wq.lib
    big_m = 65535 * 128 + 1
    assert _w4(wq, M=big_m, ldy=64) == wq.WQ_ERR_UNSUPPORTED
    assert L.wq_gemm_w8a16(big_m, 64, 64, FAKE, 64, FAKE, 64, FAKE, FAKE, 64, None, 0, None) == wq.WQ_ERR_UNSUPPORTED
    assert L.mx_gemm_fp4(big_m, 64, 64, FAKE, 32, FAKE, 2, FAKE, 32, FAKE, 2, FAKE, 64, None, 0, None) \
        == wq.WQ_ERR_UNSUPPORTED
    assert L.fp8_gemm(big_m, 64, 64, FAKE, 64, FAKE, 64, 1.0, 1.0, FAKE, 64, None, 0, None) == wq.WQ_ERR_UNSUPPORTED
    assert L.fp8_gemm(64, big_m, 64, FAKE, 64, FAKE, big_m + 15, 1.0, 1.0, FAKE, big_m + 7, None, 0, None) \
        == wq.WQ_ERR_UNSUPPORTED
    rows, cols = 1 << 21, 1 << 15  # 2^31 blocks of 32
    assert L.mx_quantize_fp4(rows, cols, FAKE, cols, FAKE, cols // 2, FAKE, cols // 32, None) == wq.WQ_ERR_UNSUPPORTED
