"""GPU parity of wq_gemm_w4a16_grouped / wq_gemm_w8a16_grouped (column-grouped
scales, optional zero points) against the CPU oracle.

Tolerance as for the per-column GEMMs: |y - y_ref| <= 5e-3 * max|y_ref| + 1
fp16 ulp at y_ref, per element.  The shapes reach every plan of both kernels:
one cluster per tile (N = 4096), one CTA per tile (N = 14336), the K-split
through the workspace (small N), several 16-row M tiles (M = 64), and the
tensor-memory GEMM (M > 64); groups that do not divide N leave a short last
group."""
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


def _run(wq, case, ldx=None, ldw=None, ldy=None):
    M, K = case.x.shape
    N = case.w.shape[1]
    x = dev_matrix(torch, case.x, ldx)
    w = dev_matrix(torch, case.w, ldw)
    s = torch.from_numpy(case.scales).cuda()
    z = torch.from_numpy(case.zeros).cuda() if case.zeros is not None else None
    y = dev_empty(torch, M, N, torch.float16, ldy, fill=float("nan"))
    fn = wq.wq_gemm_w4a16_grouped if case.bits == 4 else wq.wq_gemm_w8a16_grouped
    fn(x, w, s, z, case.group_n, y=y)
    torch.cuda.synchronize()
    return y


def _ref(case, rows=None):
    x = case.x if rows is None else case.x[rows]
    fn = O.gemm_w4a16_grouped if case.bits == 4 else O.gemm_w8a16_grouped
    return fn(x, case.w, case.scales, case.zeros, case.group_n)


CASES = [  # (M, K, N, group_n, ldx, ldw, ldy)
    (1, 4096, 4096, 128, None, None, None),       # clusters of CTAs per tile
    (16, 4096, 14336, 128, None, None, None),     # one CTA per tile
    (4, 4096, 512, 32, None, None, None),         # K split through the workspace
    (5, 1000, 3008, 7, None, None, None),         # short last group, ragged K
    (3, 96, 257, 5, None, 272, 264),              # ragged N, padded strides
    (9, 2048, 1000, 1000, 2056, 1008, 1000),      # one group for all columns
    (64, 2048, 640, 1, None, None, None),         # mid M: K split over a cluster, per-column groups
    (40, 4096, 4096, 128, None, None, None),      # mid M, eight-CTA clusters
    (17, 1000, 300, 7, 1008, 304, 312),           # mid M, ragged K and N, padded strides
    (300, 1024, 520, 64, None, 528, None),        # tensor-memory GEMM, ragged M and N
]


@pytest.mark.parametrize("asym", [False, True])
@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,K,N,G,ldx,ldw,ldy", CASES)
def test_grouped_matches_oracle(wq, bits, asym, M, K, N, G, ldx, ldw, ldy):
    case = workloads.grouped_case(bits, M, K, N, G, asym, seed=M + N + G)
    assert_gemm_close(_run(wq, case, ldx, ldw, ldy), _ref(case), "fp16")


@pytest.mark.parametrize("bits", [4, 8])
def test_grouped_large_m_sampled_rows(wq, bits):
    case = workloads.grouped_case(bits, 4096, 4096, 4096, 128, True, seed=3)
    y = _run(wq, case)
    rows = np.array([0, 1, 127, 128, 2047, 4095])
    assert_gemm_close(y[rows], _ref(case, rows), "fp16")


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,K,N", [(1, 4096, 4096), (16, 4096, 14336), (4, 4096, 512), (300, 1024, 528)])
def test_one_column_groups_without_zeros_equal_the_per_column_call(wq, bits, M, K, N):
    """group_n = 1 and no zero points is the per-column symmetric GEMM, bit for bit."""
    base = workloads.w4a16_case(M, K, N, 5) if bits == 4 else workloads.w8a16_case(M, K, N, 5)
    x = torch.from_numpy(base.x).cuda()
    w = torch.from_numpy(base.w).cuda()
    s = torch.from_numpy(base.scales).cuda()
    if bits == 4:
        y0, y1 = wq.wq_gemm_w4a16(x, w, s), wq.wq_gemm_w4a16_grouped(x, w, s, None, 1)
    else:
        y0, y1 = wq.wq_gemm_w8a16(x, w, s), wq.wq_gemm_w8a16_grouped(x, w, s, None, 1)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
