"""GPU fp8_gemm against the CPU oracle.

Tolerance: |c - c_ref| <= 5e-3 * max|c_ref| + 1 bf16 ulp at c_ref, per element."""
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


def _run(wq, case, lda=None, ldb=None, ldc=None):
    M, K = case.a8.shape
    N = case.b8.shape[1]
    a = dev_matrix(torch, case.a8, lda)
    b = dev_matrix(torch, case.b8, ldb)
    c = dev_empty(torch, M, N, torch.bfloat16, ldc, fill=float("nan"))
    wq.fp8_gemm(a, b, case.scale_a, case.scale_b, c=c)
    torch.cuda.synchronize()
    return c


@pytest.mark.parametrize("M,K,N,lda,ldb,ldc", [
    (128, 128, 256, None, None, None),   # exactly one tile
    (1, 32, 16, None, None, None),
    (200, 96, 300, None, 304, 304),      # ragged M, N, K (K below one 128-byte step)
    (257, 640, 520, 656, 528, 528),      # padded leading dimensions
    (384, 1000, 1024, 1008, None, None),
    # The persistent kernel with more 128 x 256 tiles than CTAs (187), so
    # both TMEM accumulators take several tiles, with ragged M, N and K:
    (1300, 1000, 4100, 1008, 4112, 4104),
    (16, 8192, 8192, None, None, None),  # the M = 16 FP8 workload (skinny e4m3 path)
    (3, 99, 300, 112, 304, 304),         # K not a multiple of 4: zero-masked tail bytes of A
    (12, 1000, 520, 1008, 528, 528),     # second MMA column block, ragged N
    (9, 4096, 14336, None, None, None),
    (17, 512, 384, None, None, None),    # just above the skinny bound
    (2048, 512, 2500, None, 2512, 2504),  # 160 persistent tiles on 152 SMs, ragged N, padded strides
])
def test_fp8_cases(wq, M, K, N, lda, ldb, ldc):
    case = workloads.fp8_case(M, K, N, seed=M + K + N)
    c = _run(wq, case, lda, ldb, ldc)
    assert_gemm_close(c, O.fp8_gemm(case.a8, case.b8, case.scale_a, case.scale_b), "bf16")


@pytest.mark.parametrize("S", [4096, 8192])
def test_fp8_square_every_element(wq, S):
    """The square FP8 workloads at full size, every output element against the
    oracle (every 128 x 256 tile of the persistent kernel, both TMEM
    accumulators)."""
    case = workloads.fp8_case(S, S, S, seed=0)
    c = _run(wq, case)
    assert_gemm_close(c, O.fp8_gemm(case.a8, case.b8, case.scale_a, case.scale_b), "bf16")


def test_fp8_identity_and_k_zero(wq):
    eye = np.where(np.eye(128, dtype=bool), 0x38, 0).astype(np.uint8)  # 1.0 on the diagonal
    b = workloads.fp8_case(128, 128, 256, seed=1).b8
    case = workloads.Fp8Case(eye, b, 0.5, 2.0)
    assert_gemm_close(_run(wq, case), O.fp8_gemm(eye, b, 0.5, 2.0), "bf16")
    z = workloads.Fp8Case(np.zeros((5, 0), np.uint8), np.zeros((0, 40), np.uint8), 1.0, 1.0)
    a = torch.empty((5, 0), dtype=torch.uint8, device="cuda")
    bb = torch.empty((0, 48), dtype=torch.uint8, device="cuda")[:, :40]
    c = dev_empty(torch, 5, 40, torch.bfloat16, 48, fill=float("nan"))
    wq.fp8_gemm(a, bb, 1.0, 1.0, c=c)
    torch.cuda.synchronize()
    assert torch.all(c == 0)
    del z
