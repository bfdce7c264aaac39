"""GPU mx_gemm_fp4 against the CPU oracle.

Tolerance: |c - c_ref| <= 5e-3 * max|c_ref| + 1 fp32 ulp at c_ref, per element.
Structured cases (one non-trivial scale per row / per block) come first: a
wrong scale-factor placement shows up there as a clean pattern."""
import json
import os

import numpy as np
import pytest

import workloads
from oracle import wq_oracle as O
from tests.gpu_util import assert_gemm_close, dev_empty, dev_matrix

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def wq():
    import bit_quantized_gemm_dequant_gb300 as mod

    return mod


def _gemm(wq, ad, asc, wd, wsc, lda=None, ldsa=None, ldw=None, ldsw=None, ldc=None):
    M, N = ad.shape[0], wd.shape[0]
    c = dev_empty(torch, M, N, torch.float32, ldc, fill=float("nan"))
    wq.mx_gemm_fp4(dev_matrix(torch, ad, lda), dev_matrix(torch, asc, ldsa), dev_matrix(torch, wd, ldw),
                   dev_matrix(torch, wsc, ldsw), c=c)
    torch.cuda.synchronize()
    return c


def test_worked_example(wq):
    with open(os.path.join(os.path.dirname(__file__), "golden", "mx_gemm_worked.json")) as f:
        g = json.load(f)
    ad, asc = np.array(g["a_data"], np.uint8), np.array(g["a_scales"], np.uint8)
    wd, wsc = np.array(g["w_data"], np.uint8), np.array(g["w_scales"], np.uint8)
    c = _gemm(wq, ad, asc, wd, wsc, lda=32, ldw=32, ldc=4)
    np.testing.assert_array_equal(c.cpu().numpy().astype(np.float64), np.array(g["c"]))


def test_per_row_and_per_block_scales(wq):
    """All data +1.0 (code 2); A row m gets exponent 127 + (m % 7) - 3 in block
    kb % 3 == 0 and 127 elsewhere, W row n gets 127 + (n % 5) - 2 in blocks
    kb % 4 == 1: every scale position is distinguishable in the result."""
    M, N, K = 256, 256, 1024
    nkb = K // 32
    ad = np.full((M, K // 2), 0x22, np.uint8)
    wd = np.full((N, K // 2), 0x22, np.uint8)
    asc = np.full((M, nkb), 127, np.uint8)
    wsc = np.full((N, nkb), 127, np.uint8)
    for kb in range(nkb):
        if kb % 3 == 0:
            asc[:, kb] = 127 + (np.arange(M) % 7) - 3
        if kb % 4 == 1:
            wsc[:, kb] = 127 + (np.arange(N) % 5) - 2
    c = _gemm(wq, ad, asc, wd, wsc)
    assert_gemm_close(c, O.mx_gemm_fp4(ad, asc, wd, wsc), "fp32", rel=1e-6)


@pytest.mark.parametrize("M,N,K,lda,ldsa,ldw,ldsw,ldc", [
    (128, 128, 256, None, None, None, None, None),
    (1, 16, 32, 16, None, 16, None, None),          # a single scale block
    (200, 300, 800, 400, 25, 400, 27, 304),         # ragged M/N/K, odd scale strides
    (130, 256, 8192, None, None, None, None, None),
    (384, 128, 4096, 2064, 130, 2048, 128, 132),
    (300, 520, 1024, None, None, None, None, None),  # odd number of 128-row tiles, ragged N
    # The persistent kernel (at least half as many 128 x 256 tiles as SMs),
    # with more tiles than CTAs, fewer K steps than ring slots, ragged edges:
    (1300, 4100, 256, None, None, None, None, 4104),  # 187 tiles, one K step
    (2048, 2560, 800, None, None, None, None, None),  # 160 tiles, partial fourth K step
    (1030, 5000, 1312, 1312, 48, None, None, None),   # 180 tiles, six K steps, the last partial
])
def test_random_quantized(wq, M, N, K, lda, ldsa, ldw, ldsw, ldc):
    a = workloads.mx_source(M, K, seed=M + K, stream=0)
    w = workloads.mx_source(N, K, seed=N + K, stream=1)
    ad, asc = O.mx_quantize_fp4(a)
    wd, wsc = O.mx_quantize_fp4(w)
    c = _gemm(wq, ad, asc, wd, wsc, lda, ldsa, ldw, ldsw, ldc)
    assert_gemm_close(c, O.mx_gemm_fp4(ad, asc, wd, wsc), "fp32")


_W_REF: dict = {}


def _w_reference():
    """The workload's W [8192, 8192] and its oracle quantization and
    dequantization, computed once per test session."""
    if not _W_REF:
        w = workloads.mx_source(8192, 8192, seed=0, stream=1)
        wd, ws = O.mx_quantize_fp4(w)
        _W_REF.update(w=w, wd=wd, ws=ws, wdq=O.mx_dequantize(wd, ws))
    return _W_REF


@pytest.mark.parametrize("M", [128, 2048, 8192])
def test_mxfp4_workload_quantize_then_gemm(wq, M):
    """The MXFP4 workload end to end on the device: both fp32 operands quantized
    by mx_quantize_fp4 (bit-exact), then mx_gemm_fp4.  M = 128 and 2048 are
    compared on every element; M = 8192 on the first, last and one inner row
    of every 128-row tile.  The full references use the dequantize-then-matmul
    form of the oracle, which the oracle pins hold equal to its block-by-block
    sum (test_mx_gemm_equals_dequantize_then_matmul)."""
    K = N = 8192
    ref_w = _w_reference()
    a = workloads.mx_source(M, K, seed=0, stream=0)
    ad, asc = wq.mx_quantize_fp4(torch.from_numpy(a).cuda())
    wd, wsc = wq.mx_quantize_fp4(torch.from_numpy(ref_w["w"]).cuda())
    c = wq.mx_gemm_fp4(ad, asc, wd, wsc)
    torch.cuda.synchronize()
    assert np.array_equal(wd.cpu().numpy(), ref_w["wd"]) and np.array_equal(wsc.cpu().numpy(), ref_w["ws"])
    if M <= 2048:
        rad, ras = O.mx_quantize_fp4(a)
        assert np.array_equal(ad.cpu().numpy(), rad) and np.array_equal(asc.cpu().numpy(), ras)
        assert_gemm_close(c, O.mx_dequantize(rad, ras) @ ref_w["wdq"].T, "fp32")
    else:
        inner = np.random.default_rng(M).integers(1, 127, size=M // 128)
        rows = np.sort(np.concatenate([np.arange(0, M, 128), np.arange(127, M, 128),
                                       np.arange(0, M, 128) + inner]))
        rad, ras = O.mx_quantize_fp4(a[rows])
        assert np.array_equal(ad.cpu().numpy()[rows], rad) and np.array_equal(asc.cpu().numpy()[rows], ras)
        ref = O.mx_gemm_fp4(rad, ras, ref_w["wd"], ref_w["ws"])
        assert_gemm_close(c[torch.from_numpy(rows).cuda()], ref, "fp32")


def test_k_zero(wq):
    c = dev_empty(torch, 3, 20, torch.float32, 20, fill=float("nan"))
    e = torch.empty((3, 0), dtype=torch.uint8, device="cuda")
    f = torch.empty((20, 0), dtype=torch.uint8, device="cuda")
    wq.mx_gemm_fp4(e, e, f, f, c=c)
    torch.cuda.synchronize()
    assert torch.all(c == 0)


def test_split_k_cluster_is_deterministic(wq):
    """M = 128 at N = 8192 has too few tiles to fill the GPU, so K is split
    over a cluster of CTAs that add their partial tiles in distributed shared
    memory, in rank order.  The split needs no scratch: the workspace holds
    only the two rewritten scale arrays.  C's previous contents do not
    matter; two calls give identical bits; every element matches the
    oracle."""
    M, N, K = 128, 8192, 4096
    sizes = [int(wq.lib.fp4_scales_tc_size(wq.WQ_FP4_MX, r, K)) for r in (M, N)]
    assert wq.wq_workspace_size(wq.WQ_OP_MX_GEMM, M, N, K) == -(-sizes[0] // 256) * 256 + sizes[1]
    a = workloads.mx_source(M, K, seed=3, stream=0)
    w = workloads.mx_source(N, K, seed=3, stream=1)
    ad, asc = wq.mx_quantize_fp4(torch.from_numpy(a).cuda())
    wd, wsc = wq.mx_quantize_fp4(torch.from_numpy(w).cuda())
    c = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    wq.mx_gemm_fp4(ad, asc, wd, wsc, c=c)
    c2 = wq.mx_gemm_fp4(ad, asc, wd, wsc)
    torch.cuda.synchronize()
    assert torch.equal(c, c2)
    ref = O.mx_dequantize(ad.cpu().numpy(), asc.cpu().numpy()) @ O.mx_dequantize(wd.cpu().numpy(), wsc.cpu().numpy()).T
    assert_gemm_close(c, ref, "fp32")


@pytest.mark.parametrize("M,N,K,ldc", [(1, 2560, 8192, 2564), (1, 2048, 8192, None), (100, 300, 2048, 304),
                                     (8, 256, 4096, None)])
def test_split_k_cluster_ragged(wq, M, N, K, ldc):
    """Split-K clusters on 128-column tiles with ragged M and N (the rows and
    columns past the matrix are neither read nor written) and a padded ldc:
    clusters of 7 (20 tiles), 8 (16 tiles), 2 and 4."""
    a = workloads.mx_source(M, K, seed=M, stream=0)
    w = workloads.mx_source(N, K, seed=N, stream=1)
    ad, asc = O.mx_quantize_fp4(a)
    wd, wsc = O.mx_quantize_fp4(w)
    c = dev_empty(torch, M, N, torch.float32, ldc, fill=float("nan"))
    wq.mx_gemm_fp4(dev_matrix(torch, ad), dev_matrix(torch, asc), dev_matrix(torch, wd), dev_matrix(torch, wsc), c=c)
    torch.cuda.synchronize()
    assert_gemm_close(c, O.mx_dequantize(ad, asc) @ O.mx_dequantize(wd, wsc).T, "fp32")
