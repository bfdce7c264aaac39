"""GPU mx_gemm_fp4_qa (A given in FP32 and quantized inside the GEMM launch)
against the CPU oracle: the quantized A it leaves in the workspace byte for
byte (codes and tensor-core-layout scales), C against the oracle GEMM, and C
bit for bit against mx_quantize_fp4 followed by mx_gemm_fp4.

GEMM tolerance: |c - c_ref| <= 5e-3 * max|c_ref| + 1 fp32 ulp at c_ref."""
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


def _workspace(wq, M, N, K):
    return torch.zeros(int(wq.lib.wq_workspace_size(wq.WQ_OP_MX_GEMM_QA, M, N, K)), dtype=torch.uint8,
                       device="cuda")


def _quantized_a(ws, M, K):
    """The workspace's documented contents after a call: codes [M, ldq] at
    byte 256, then the scales (tensor-core layout) at the next 256-byte
    boundary."""
    ldq = -(-(K // 2) // 16) * 16
    codes = ws[256:256 + M * ldq].view(M, ldq)[:, :K // 2]
    s0 = 256 + -(-(M * ldq) // 256) * 256
    return codes, ws[s0:]


@pytest.mark.parametrize("M,N,K,lda,ldc", [
    (1, 16, 32, None, None),
    (200, 300, 800, 808, 304),      # ragged M, N, K; padded rows of A and C
    (128, 8192, 4096, None, None),  # the K-split cluster path
    (300, 520, 1024, None, None),   # three 128-row tiles, ragged N (persistent path)
    (2048, 512, 2048, None, None),
    # The persistent instance (at least half as many 128 x 256 tiles as SMs):
    (1300, 4100, 256, None, 4104),  # 187 tiles, one K step
    (2048, 2560, 800, 804, None),   # 160 tiles, partial fourth K step, padded rows of A
    (1030, 5000, 1312, None, None), # 180 tiles, six K steps
])
def test_fused_quantize_gemm(wq, M, N, K, lda, ldc):
    a = workloads.mx_source(M, K, seed=M + K, stream=0)
    w = workloads.mx_source(N, K, seed=N + K, stream=1)
    ad, asc = O.mx_quantize_fp4(a)
    wd, wsc = O.mx_quantize_fp4(w)
    A = dev_matrix(torch, a, lda)
    W, SW = dev_matrix(torch, wd), dev_matrix(torch, wsc)
    sw_tc = wq.fp4_scales_tc(SW, K)
    ws = _workspace(wq, M, N, K)
    c = dev_empty(torch, M, N, torch.float32, ldc, fill=float("nan"))
    wq.mx_gemm_fp4_qa(A, W, sw_tc, c=c, workspace=ws)
    qd, qs = wq.mx_quantize_fp4(A)
    c_two = wq.mx_gemm_fp4(qd, qs, W, SW)
    torch.cuda.synchronize()
    codes, scales = _quantized_a(ws, M, K)
    assert np.array_equal(codes.cpu().numpy(), ad), "quantized A codes differ from the oracle"
    want_s = O.fp4_scales_tc(asc, K, 32)
    assert np.array_equal(scales[:want_s.size].cpu().numpy(), want_s), "quantized A scales differ from the oracle"
    assert torch.count_nonzero(ws[:8]).item() == 0, "grid barrier words not reset"
    assert torch.equal(c, c_two)
    assert_gemm_close(c, O.mx_gemm_fp4(ad, asc, wd, wsc), "fp32")


def test_repeated_calls_identical(wq):
    M, N, K = 256, 1024, 2048
    a = torch.from_numpy(workloads.mx_source(M, K, seed=5, stream=0)).cuda()
    wd, wsc = wq.mx_quantize_fp4(torch.from_numpy(workloads.mx_source(N, K, seed=5, stream=1)).cuda())
    sw_tc = wq.fp4_scales_tc(wsc, K)
    first = wq.mx_gemm_fp4_qa(a, wd, sw_tc)
    for _ in range(3):
        assert torch.equal(first, wq.mx_gemm_fp4_qa(a, wd, sw_tc))
    torch.cuda.synchronize()


def test_workspace_checks(wq):
    M, N, K = 64, 256, 512
    a = torch.zeros((M, K), dtype=torch.float32, device="cuda")
    wd = torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda")
    sw_tc = wq.fp4_scales_tc(torch.zeros((N, K // 32), dtype=torch.uint8, device="cuda"), K)
    with pytest.raises(wq.WqError) as e:
        wq.mx_gemm_fp4_qa(a, wd, sw_tc, workspace=torch.zeros(64, dtype=torch.uint8, device="cuda"))
    assert e.value.status == wq.WQ_ERR_WORKSPACE
    with pytest.raises(wq.WqError) as e:
        wq.mx_gemm_fp4_qa(a, wd, sw_tc[:-16])
    assert e.value.status == wq.WQ_ERR_INVALID_ARG
