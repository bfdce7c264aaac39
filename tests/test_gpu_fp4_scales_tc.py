"""GPU fp4_scales_tc (block scales in the tensor cores' chunk order) byte for
byte against the oracle's restatement of that layout, and the GEMM entry
points that take such scales (mx_gemm_fp4_tc, nv_gemm_fp4_tc) against the
oracle GEMMs and, bit for bit, against the row-major entry points.

GEMM tolerance: |c - c_ref| <= 5e-3 * max|c_ref| + 1 fp32 ulp at c_ref."""
import numpy as np
import pytest

import workloads
from oracle import wq_oracle as O
from tests.gpu_util import assert_gemm_close, dev_matrix

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def wq():
    import bit_quantized_gemm_dequant_gb300 as mod

    return mod


@pytest.mark.parametrize("fmt,rows,K,lds", [
    ("mx", 300, 512, None),   # ragged rows: row groups 2 and 3 partly or wholly padding
    ("mx", 1, 32, None),      # one scale
    ("mx", 257, 8192, 263),   # odd row stride: byte loads
    ("mx", 128, 800, None),   # K not a multiple of 256: padded blocks in the last chunks
    ("nv", 5, 80, None),
    ("nv", 130, 4096, 300),
    ("nv", 512, 1040, None),
])
def test_scales_tc_bytes(wq, fmt, rows, K, lds):
    block = 32 if fmt == "mx" else 16
    s = np.random.default_rng(rows + K).integers(0, 256, size=(rows, K // block), dtype=np.uint8)
    out = wq.fp4_scales_tc(dev_matrix(torch, s, lds), K, wq.WQ_FP4_MX if fmt == "mx" else wq.WQ_FP4_NV)
    torch.cuda.synchronize()
    want = O.fp4_scales_tc(s, K, block)
    got = out.cpu().numpy()
    assert got.shape == want.shape
    assert np.array_equal(got, want), f"first difference at byte {int(np.argmax(got != want))}"


def test_scales_tc_sizes(wq):
    for fmt, block in ((wq.WQ_FP4_MX, 32), (wq.WQ_FP4_NV, 16)):
        for rows, K in ((1, 32), (300, 512), (8192, 8192), (129, 1056)):
            want = O.fp4_scales_tc(np.zeros((rows, K // block), np.uint8), K, block).size
            assert int(wq.lib.fp4_scales_tc_size(fmt, rows, K)) == want


@pytest.mark.parametrize("M,N,K", [
    (1, 16, 32),
    (200, 300, 800),       # ragged M, N and K
    (128, 8192, 4096),     # the K-split cluster path
    (2048, 512, 2048),     # the persistent path
])
def test_mx_gemm_tc(wq, M, N, K):
    a = workloads.mx_source(M, K, seed=M + K, stream=0)
    w = workloads.mx_source(N, K, seed=N + K, stream=1)
    ad, asc = O.mx_quantize_fp4(a)
    wd, wsc = O.mx_quantize_fp4(w)
    A, SA, W, SW = (dev_matrix(torch, x) for x in (ad, asc, wd, wsc))
    c_tc = wq.mx_gemm_fp4_tc(A, wq.fp4_scales_tc(SA, K), W, wq.fp4_scales_tc(SW, K))
    c_rm = wq.mx_gemm_fp4(A, SA, W, SW)
    torch.cuda.synchronize()
    assert torch.equal(c_tc, c_rm)
    assert_gemm_close(c_tc, O.mx_gemm_fp4(ad, asc, wd, wsc), "fp32")


@pytest.mark.parametrize("M,N,K", [
    (1, 16, 16),
    (200, 300, 1040),
    (128, 8192, 4096),
    (2048, 512, 2048),
])
def test_nv_gemm_tc(wq, M, N, K):
    a = workloads.mx_source(M, K, seed=M + K, stream=0)
    w = workloads.mx_source(N, K, seed=N + K, stream=1)
    ad, asc, ga = O.nv_quantize_fp4(a)
    wd, wsc, gw = O.nv_quantize_fp4(w)
    ld = -(-K // 32) * 16  # packed rows padded to 16 bytes
    A, W = dev_matrix(torch, ad, ld), dev_matrix(torch, wd, ld)
    SA, SW = dev_matrix(torch, asc), dev_matrix(torch, wsc)
    GA = torch.tensor([ga], dtype=torch.float32, device="cuda")
    GW = torch.tensor([gw], dtype=torch.float32, device="cuda")
    nv = wq.WQ_FP4_NV
    c_tc = wq.nv_gemm_fp4_tc(A, wq.fp4_scales_tc(SA, K, nv), GA, W, wq.fp4_scales_tc(SW, K, nv), GW)
    c_rm = wq.nv_gemm_fp4(A, SA, GA, W, SW, GW)
    torch.cuda.synchronize()
    assert torch.equal(c_tc, c_rm)
    assert_gemm_close(c_tc, O.nv_gemm_fp4(ad, asc, ga, wd, wsc, gw), "fp32")


def test_tc_scale_buffers_too_small(wq):
    M = N = 256
    K = 512
    A = torch.zeros((M, K // 2), dtype=torch.uint8, device="cuda")
    W = torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda")
    S = torch.zeros((M, K // 32), dtype=torch.uint8, device="cuda")
    sa = wq.fp4_scales_tc(S, K)
    with pytest.raises(wq.WqError) as e:
        wq.mx_gemm_fp4_tc(A, sa[:-16], W, sa)
    assert e.value.status == wq.WQ_ERR_INVALID_ARG
    ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(wq.WqError) as e:
        wq.mx_gemm_fp4(A, S, W, S, workspace=ws)
    assert e.value.status == wq.WQ_ERR_WORKSPACE
