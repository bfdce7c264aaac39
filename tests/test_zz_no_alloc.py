"""The allocation-free INT8 entry point, called through the C ABI.

wq_gemm_w8a16_noalloc serves callers that cannot allocate device memory at
call time (engine plugins, real-time loops, runtimes that plan every byte up
front): it keeps its split-K scratch in an array inside the library.  Its
output must match the ordinary entry point, wq_gemm_w8a16, which is given a
fresh workspace, on two calls in a row (the second one starts from whatever
the first left in the shared array).  This file is collected last so that a
run stopping at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import workloads
from tests.gpu_util import assert_gemm_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def wq():
    import bit_quantized_gemm_dequant_gb300 as mod

    return mod


def _noalloc(wq, x, w, s, y):
    M, K = x.shape
    N = w.shape[1]
    return wq.lib.wq_gemm_w8a16_noalloc(M, N, K, ctypes.c_void_p(x.data_ptr()), K, ctypes.c_void_p(w.data_ptr()), N,
                                        ctypes.c_void_p(s.data_ptr()), ctypes.c_void_p(y.data_ptr()), N,
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


# The first two shapes split K across CTAs and so use the built-in scratch;
# the others need none (whole tiles per CTA, or a cluster per tile).
@pytest.mark.parametrize("M,K,N", [(4, 4096, 512), (1, 8192, 1024), (16, 4096, 14336), (5, 1000, 3008)])
def test_noalloc_matches_workspace_entry_point_twice(wq, M, K, N):
    case = workloads.w8a16_case(M, K, N, seed=21)
    x = torch.from_numpy(case.x).cuda()
    w = torch.from_numpy(case.w).cuda()
    s = torch.from_numpy(case.scales).cuda()
    need = wq.wq_workspace_size(wq.WQ_OP_W8A16, M, N, K)
    if N <= 1024:
        assert 0 < need <= 1 << 20  # these shapes do go through the scratch, and fit it
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")
    ref = wq.wq_gemm_w8a16(x, w, s, workspace=ws)
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        assert _noalloc(wq, x, w, s, y) == wq.WQ_OK
        torch.cuda.synchronize()
        assert_gemm_close(y, ref.float().cpu().numpy().astype(np.float64), "fp16")
    st, site = wq.wq_get_device_error()
    assert st == wq.WQ_OK and site == 0


def test_noalloc_refuses_shapes_beyond_its_scratch(wq):
    """A shape whose split-K scratch exceeds the built-in 1 MiB is refused before launch."""
    M, K, N = 16, 16384, 1024
    assert wq.wq_workspace_size(wq.WQ_OP_W8A16, M, N, K) > 1 << 20
    x = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    w = torch.zeros((K, N), dtype=torch.int8, device="cuda")
    s = torch.ones(N, dtype=torch.float16, device="cuda")
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert _noalloc(wq, x, w, s, y) == wq.WQ_ERR_WORKSPACE
