"""GPU NVFP4 (nv_quantize_fp4, nv_gemm_fp4) against the CPU oracle.

The quantizer must match byte for byte (data, E4M3 block scales) and the
tensor scale bit for bit.  GEMM tolerance: |c - c_ref| <= 5e-3 * max|c_ref|
+ 1 fp32 ulp at c_ref, per element."""
import json
import os

import numpy as np
import pytest

import workloads
from oracle import wq_oracle as O
from tests.gpu_util import assert_gemm_close, dev_empty, dev_matrix

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_worked.json")


@pytest.fixture(scope="module")
def wq():
    import bit_quantized_gemm_dequant_gb300 as mod

    return mod


def _quant(wq, src, ld_src=None, ld_data=None, ld_scales=None):
    R, C = src.shape
    s = dev_matrix(torch, src, ld_src)
    d = dev_empty(torch, R, C // 2, torch.uint8, ld_data, fill=0xEE)
    e = dev_empty(torch, R, C // 16, torch.uint8, ld_scales, fill=0xEE)
    g = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    wq.nv_quantize_fp4(s, d, e, g)
    torch.cuda.synchronize()
    return d.cpu().numpy(), e.cpu().numpy(), np.float32(g.item())


def _assert_exact(got, want):
    gd, ge, gg = got
    rd, re_, rg = want
    assert gg == rg, f"tensor scale {gg!r} vs {rg!r}"
    assert np.array_equal(ge, re_), f"scales differ at {np.argwhere(ge != re_)[:5].tolist()}"
    assert np.array_equal(gd, rd), f"data differ at {np.argwhere(gd != rd)[:5].tolist()}"


def test_quantize_worked_example(wq):
    with open(GOLDEN) as f:
        q = json.load(f)["quantize"]
    x = np.array(q["src"], np.float32)
    x[0, 21] = np.float32(-0.0)
    d, e, g = _quant(wq, x)
    assert float(g) == q["g"]
    assert np.array_equal(d, np.array(q["data"], np.uint8))
    assert np.array_equal(e, np.array(q["scales"], np.uint8))


@pytest.mark.parametrize("R,C,ld_src,ld_data,ld_scales", [
    (1, 16, None, None, None),
    (5, 48, 52, 32, 7),               # padded strides, odd scale stride
    (64, 1024, None, None, None),
    (300, 4112, 4116, 2064, 300),     # several column blocks of a launch, ragged
])
def test_quantize_random_bit_exact(wq, R, C, ld_src, ld_data, ld_scales):
    rng = np.random.default_rng(R + C)
    x = (rng.standard_normal((R, C)) * rng.choice([1e-4, 1.0, 30.0], size=(R, 1))).astype(np.float32)
    _assert_exact(_quant(wq, x, ld_src, ld_data, ld_scales), O.nv_quantize_fp4(x))


def test_quantize_wide_range_ties_and_zero_blocks(wq):
    """Blocks whose scales fall into E4M3's subnormal range or round to zero,
    all-zero blocks, exact grid points and midpoints (ties) at several block
    scales."""
    rng = np.random.default_rng(4)
    R, C = 64, 256
    x = (rng.standard_normal((R, C)) * np.exp2(rng.integers(-30, 12, size=(R, C // 16))).repeat(16, axis=1))
    x = x.astype(np.float32)
    x[0, :] = 3000.0  # sets the tensor scale high, so that small blocks get tiny scales
    x[1, :16] = 0.0
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, -0.75, -3.5],
                    np.float32)
    for r in range(2, 12):
        x[r, :16] = mids * np.float32(2.0 ** (r - 6))
    _assert_exact(_quant(wq, x), O.nv_quantize_fp4(x))


def test_quantize_full_operand_rows(wq):
    """The 8192 x 8192 workload operand: every scale byte, and the data of 256
    rows (the tensor scale comes from the whole tensor)."""
    src = workloads.mx_source(8192, 8192, seed=0, stream=1)
    d, e, g = _quant(wq, src)
    rg = O.nv_tensor_scale(src)
    assert g == rg
    rows = np.random.default_rng(0).choice(8192, 256, replace=False)
    rd, re_, _ = O.nv_quantize_fp4(src[rows], rg)
    assert np.array_equal(e[rows], re_) and np.array_equal(d[rows], rd)


def _gemm(wq, ad, asc, ga, wd, wsc, gw, lda=None, ldsa=None, ldw=None, ldsw=None, ldc=None):
    M, N = ad.shape[0], wd.shape[0]
    c = dev_empty(torch, M, N, torch.float32, ldc, fill=float("nan"))
    gat = torch.tensor([float(ga)], dtype=torch.float32, device="cuda")
    gwt = torch.tensor([float(gw)], dtype=torch.float32, device="cuda")
    wq.nv_gemm_fp4(dev_matrix(torch, ad, lda), dev_matrix(torch, asc, ldsa), gat,
                   dev_matrix(torch, wd, ldw), dev_matrix(torch, wsc, ldsw), gwt, c=c)
    torch.cuda.synchronize()
    return c


def test_gemm_worked_example(wq):
    with open(GOLDEN) as f:
        q = json.load(f)["gemm"]
    c = _gemm(wq, np.array(q["a_data"], np.uint8), np.array(q["a_scales"], np.uint8), q["ga"],
              np.array(q["w_data"], np.uint8), np.array(q["w_scales"], np.uint8), q["gw"], lda=16, ldw=16, ldc=4)
    assert c.cpu().numpy().astype(np.float64).tolist() == q["c"]


def test_gemm_per_row_and_per_block_scales(wq):
    """All data +1.0 (code 2); scales vary by row and by 16-element block in a
    pattern that makes every scale position visible in the result."""
    M, N, K = 256, 256, 1024
    nkb = K // 16
    ad = np.full((M, K // 2), 0x22, np.uint8)
    wd = np.full((N, K // 2), 0x22, np.uint8)
    asc = np.full((M, nkb), 0x38, np.uint8)  # 1.0
    wsc = np.full((N, nkb), 0x38, np.uint8)
    for kb in range(nkb):
        if kb % 3 == 0:
            asc[:, kb] = 0x38 + (np.arange(M) % 7) - 3
        if kb % 5 == 2:
            wsc[:, kb] = 0x30 + (np.arange(N) % 9)
    c = _gemm(wq, ad, asc, 0.5, wd, wsc, 3.0)
    assert_gemm_close(c, O.nv_gemm_fp4(ad, asc, 0.5, wd, wsc, 3.0), "fp32", rel=1e-6)


@pytest.mark.parametrize("M,N,K,lda,ldsa,ldw,ldsw,ldc", [
    (128, 256, 256, None, None, None, None, None),
    (1, 16, 16, 16, None, 16, None, None),            # one scale block
    (200, 300, 800, 400, 50, 400, 51, 304),           # ragged M/N/K, odd scale stride (byte loads in the re-layout)
    (130, 256, 8192, None, None, None, None, None),
    (384, 128, 4096, 2064, 272, 2048, 256, 132),
    (300, 520, 1040, 528, None, 528, None, None),     # K not a multiple of 256: partial last step
    (64, 256, 1040, 528, 80, 528, 80, None),          # partial last step, 16-byte scale rows
    # The persistent kernel (at least half as many 128 x 256 tiles as SMs),
    # whose epilogue warps stage the scales: more tiles than CTAs, fewer K
    # steps than ring slots, ragged edges:
    (1300, 4100, 256, None, None, None, None, 4104),  # 187 tiles, one K step
    (2048, 2560, 800, None, None, None, None, None),  # 160 tiles, partial fourth K step
    (1030, 5000, 1312, 1312, 96, None, None, None),   # 180 tiles, six K steps, the last partial
])
def test_gemm_random_quantized(wq, M, N, K, lda, ldsa, ldw, ldsw, ldc):
    a = workloads.mx_source(M, K, seed=M + K, stream=0)
    w = workloads.mx_source(N, K, seed=N + K, stream=1)
    ad, asc, ga = O.nv_quantize_fp4(a)
    wd, wsc, gw = O.nv_quantize_fp4(w)
    c = _gemm(wq, ad, asc, ga, wd, wsc, gw, lda, ldsa, ldw, ldsw, ldc)
    assert_gemm_close(c, O.nv_gemm_fp4(ad, asc, ga, wd, wsc, gw), "fp32")


_W_REF: dict = {}


def _w_reference():
    if not _W_REF:
        w = workloads.mx_source(8192, 8192, seed=0, stream=1)
        wd, ws, gw = O.nv_quantize_fp4(w)
        _W_REF.update(w=w, wd=wd, ws=ws, gw=gw, wdq=O.nv_dequantize(wd, ws, gw))
    return _W_REF


@pytest.mark.parametrize("M", [128, 2048, 8192])
def test_nvfp4_workload_quantize_then_gemm(wq, M):
    """The NVFP4 workload end to end on the device (both operands quantized by
    nv_quantize_fp4, then nv_gemm_fp4).  M = 128 (the K-split path) and 2048 on
    every element; M = 8192 on three rows of every 128-row tile.  The full
    references use the dequantize-then-matmul form, which the oracle pins
    hold equal to the block-by-block sum."""
    K = N = 8192
    ref_w = _w_reference()
    a = workloads.mx_source(M, K, seed=0, stream=0)
    ad, asc, ga = wq.nv_quantize_fp4(torch.from_numpy(a).cuda())
    wd, wsc, gw = wq.nv_quantize_fp4(torch.from_numpy(ref_w["w"]).cuda())
    c = wq.nv_gemm_fp4(ad, asc, ga, wd, wsc, gw)
    torch.cuda.synchronize()
    assert np.float32(gw.item()) == ref_w["gw"]
    assert np.array_equal(wd.cpu().numpy(), ref_w["wd"]) and np.array_equal(wsc.cpu().numpy(), ref_w["ws"])
    rga = O.nv_tensor_scale(a)
    assert np.float32(ga.item()) == rga
    if M <= 2048:
        rad, ras, _ = O.nv_quantize_fp4(a, rga)
        assert np.array_equal(ad.cpu().numpy(), rad) and np.array_equal(asc.cpu().numpy(), ras)
        assert_gemm_close(c, O.nv_dequantize(rad, ras, rga) @ ref_w["wdq"].T, "fp32")
    else:
        inner = np.random.default_rng(M).integers(1, 127, size=M // 128)
        rows = np.sort(np.concatenate([np.arange(0, M, 128), np.arange(127, M, 128),
                                       np.arange(0, M, 128) + inner]))
        rad, ras, _ = O.nv_quantize_fp4(a[rows], rga)
        assert np.array_equal(ad.cpu().numpy()[rows], rad) and np.array_equal(asc.cpu().numpy()[rows], ras)
        ref = O.nv_gemm_fp4(rad, ras, rga, ref_w["wd"], ref_w["ws"], ref_w["gw"])
        assert_gemm_close(c[torch.from_numpy(rows).cuda()], ref, "fp32")


def test_empty_and_k_zero(wq):
    g = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    e = torch.empty((0, 32), dtype=torch.float32, device="cuda")
    wq.nv_quantize_fp4(e, tensor_scale=g)
    torch.cuda.synchronize()
    assert g.item() == 1.0  # an empty (all-zero) tensor has scale 1
    c = dev_empty(torch, 3, 20, torch.float32, 20, fill=float("nan"))
    ea = torch.empty((3, 0), dtype=torch.uint8, device="cuda")
    ew = torch.empty((20, 0), dtype=torch.uint8, device="cuda")
    wq.nv_gemm_fp4(ea, ea, g, ew, ew, g, c=c)
    torch.cuda.synchronize()
    assert torch.all(c == 0)
