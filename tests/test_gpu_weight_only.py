"""GPU parity of wq_gemm_w4a16 / wq_gemm_w8a16 against the CPU oracle.

Tolerance: |y - y_ref| <= 5e-3 * max|y_ref| + 1 fp16 ulp at y_ref, per element.
Small cases span several 128-column tiles, ragged N/K/M tails and padded leading
dimensions; the decode workloads, the mid-M (17..64 rows) Llama shapes and
M = 4096 run at full size with every output checked."""
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


def _run(wq, bits, case, ldx=None, ldw=None, ldy=None):
    M, K = case.x.shape
    N = case.w.shape[1]
    x = dev_matrix(torch, case.x, ldx)
    w = dev_matrix(torch, case.w, ldw)
    s = torch.from_numpy(case.scales).cuda()
    y = dev_empty(torch, M, N, torch.float16, ldy, fill=float("nan"))
    fn = wq.wq_gemm_w4a16 if bits == 4 else wq.wq_gemm_w8a16
    fn(x, w, s, y=y)
    torch.cuda.synchronize()
    return y


def _ref(bits, case, rows=None):
    x = case.x if rows is None else case.x[rows]
    return O.gemm_w4a16(x, case.w, case.scales) if bits == 4 else O.gemm_w8a16(x, case.w, case.scales)


def _case(bits, M, K, N, seed):
    return workloads.w4a16_case(M, K, N, seed) if bits == 4 else workloads.w8a16_case(M, K, N, seed)


SMALL = [  # (M, K, N, ldx, ldw, ldy)
    (16, 512, 512, None, None, None),     # the tiny W4A16 workload
    (1, 64, 128, None, None, None),
    (3, 96, 257, None, 272, 264),         # ragged N inside the last 16-column vector
    (8, 50, 384, 56, 400, 392),           # K not a multiple of 16, padded strides
    (9, 1024, 200, None, 208, 200),       # second MMA column block, ragged N
    (16, 2048, 1000, 2056, 1008, 1000),
    (5, 4096, 4096, None, None, None),
    (12, 11008, 640, None, None, None),   # down-projection K
]


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,K,N,ldx,ldw,ldy", SMALL)
def test_small_cases(wq, bits, M, K, N, ldx, ldw, ldy):
    case = _case(bits, M, K, N, seed=M + K + N)
    y = _run(wq, bits, case, ldx, ldw, ldy)
    assert_gemm_close(y, _ref(bits, case), "fp16")


@pytest.mark.parametrize("M,K,N", workloads.WORKLOADS["w8a16_decode"]["shapes"])
def test_w8a16_decode_full_size(wq, M, K, N):
    case = workloads.w8a16_case(M, K, N, seed=0)
    assert_gemm_close(_run(wq, 8, case), _ref(8, case), "fp16")


@pytest.mark.parametrize("M,K,N", [s for s in workloads.WORKLOADS["w4a16_llama7b"]["shapes"]])
def test_w4a16_llama_shapes(wq, M, K, N):
    case = workloads.w4a16_case(M, K, N, seed=0)
    y = _run(wq, 4, case)
    assert_gemm_close(y, _ref(4, case), "fp16")  # every element, at every M


@pytest.mark.parametrize("bits", [4, 8])
def test_k_zero_writes_zeros(wq, bits):
    x = torch.empty((3, 0), dtype=torch.float16, device="cuda")
    w = torch.empty((0, 64), dtype=torch.uint8 if bits == 4 else torch.int8, device="cuda")
    s = torch.ones(64, dtype=torch.float16, device="cuda")
    y = torch.full((3, 64), float("nan"), dtype=torch.float16, device="cuda")
    (wq.wq_gemm_w4a16 if bits == 4 else wq.wq_gemm_w8a16)(x, w, s, y=y)
    torch.cuda.synchronize()
    assert torch.all(y == 0)


def test_int8_extremes(wq):
    """-128 and 127 codes, scales near the fp16 subnormal edge and large."""
    rng = np.random.default_rng(11)
    K, N = 256, 256
    w = rng.choice(np.array([-128, 127, -1, 0, 1], np.int8), size=(K, N))
    x = rng.standard_normal((7, K)).astype(np.float16)
    s = np.concatenate([np.full(128, 6.1e-5, np.float16), np.full(128, 3.0, np.float16)])
    case = workloads.WeightOnlyCase(x, w, s, 8)
    assert_gemm_close(_run(wq, 8, case), _ref(8, case), "fp16")


def test_out_of_tile_columns_untouched(wq):
    """Padding columns of Y beyond N keep their contents (the kernel writes only [M, N])."""
    case = workloads.w4a16_case(4, 128, 100, seed=3)
    x = dev_matrix(torch, case.x)
    w = dev_matrix(torch, case.w, 112)
    s = torch.from_numpy(case.scales).cuda()
    buf = torch.full((4, 128), 7.0, dtype=torch.float16, device="cuda")
    wq.wq_gemm_w4a16(x, w, s, y=buf[:, :100])
    torch.cuda.synchronize()
    assert torch.all(buf[:, 100:] == 7.0)
    assert_gemm_close(buf[:, :100], _ref(4, case), "fp16")


MID_M = [  # (M, K, N, ldx, ldw, ldy): one 64-row activation tile, K split over a cluster
    (17, 4096, 4096, None, None, None),
    (64, 64, 128, None, None, None),          # one k-step: clusters of one CTA
    (48, 128, 4000, None, None, None),        # two k-steps: clusters of two
    (20, 1000, 300, 1008, 304, 312),          # ragged N and K (partial last k-step), padded strides
    (33, 712, 1000, None, 1008, None),        # 12 k-steps over clusters of 8
    (64, 4096, 14336, None, None, None),
]


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,K,N,ldx,ldw,ldy", MID_M)
def test_mid_m_cases(wq, bits, M, K, N, ldx, ldw, ldy):
    case = _case(bits, M, K, N, seed=M * 5 + K + N)
    y = _run(wq, bits, case, ldx, ldw, ldy)
    assert_gemm_close(y, _ref(bits, case), "fp16")


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M", [17, 33, 64])
@pytest.mark.parametrize("K,N", [(4096, 4096), (4096, 11008), (11008, 4096)])
def test_mid_m_llama_shapes(wq, bits, M, K, N):
    """Every output of the Llama-7B-shaped linears at M in {17, 33, 64}."""
    case = _case(bits, M, K, N, seed=M + K + N)
    assert_gemm_close(_run(wq, bits, case), _ref(bits, case), "fp16")


@pytest.mark.parametrize("bits", [4, 8])
def test_mid_m_needs_no_workspace_and_is_deterministic(wq, bits):
    """The cluster K-split adds the partial tiles in a fixed rank order, so two
    calls give identical bits; it needs no workspace; the padding columns of
    Y beyond N keep their contents."""
    M, K, N = 40, 4096, 1000
    op = wq.WQ_OP_W4A16 if bits == 4 else wq.WQ_OP_W8A16
    assert wq.wq_workspace_size(op, M, N, K) == 0
    case = _case(bits, M, K, N, seed=21)
    x = torch.from_numpy(case.x).cuda()
    w = dev_matrix(torch, case.w, 1008)
    s = torch.from_numpy(case.scales).cuda()
    fn = wq.wq_gemm_w4a16 if bits == 4 else wq.wq_gemm_w8a16
    buf = torch.full((M, 1024), 7.0, dtype=torch.float16, device="cuda")
    fn(x, w, s, y=buf[:, :N])
    y2 = fn(x, w, s)
    torch.cuda.synchronize()
    assert torch.all(buf[:, N:] == 7.0)
    assert torch.equal(buf[:, :N], y2)
    assert_gemm_close(y2, _ref(bits, case), "fp16")


LARGE_M = [  # (M, K, N, ldx, ldw, ldy): the tensor-memory path (M > 64)
    (65, 64, 128, None, None, None),
    (100, 256, 384, None, None, None),
    (257, 1000, 200, 1008, 208, 200),   # ragged M, N, K (K not a multiple of 64)
    (300, 4096, 640, None, None, None),
    (512, 2048, 1024, None, None, None),
    (2100, 1000, 4100, 1008, 4112, 4104),  # two rounds of CTAs (297 tiles), ragged M, N and K
]


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("M,K,N,ldx,ldw,ldy", LARGE_M)
def test_large_m_cases(wq, bits, M, K, N, ldx, ldw, ldy):
    case = _case(bits, M, K, N, seed=M * 7 + K + N)
    y = _run(wq, bits, case, ldx, ldw, ldy)
    assert_gemm_close(y, _ref(bits, case), "fp16")


@pytest.mark.parametrize("M,K,N", [(4096, 4096, 4096), (4096, 4096, 14336)])
def test_w8a16_large_m_every_element(wq, M, K, N):
    case = workloads.w8a16_case(M, K, N, seed=1)
    assert_gemm_close(_run(wq, 8, case), _ref(8, case), "fp16")


# Activations with a non-zero mean.  The INT8 skinny path feeds the tensor
# cores 1152 + q and removes 1152 * sum(x) afterwards; that cancellation grows
# with |sum(x)|, which zero-mean activations keep small.  Long K and shifted
# activations check it against the tolerance (the tensor-memory path, M > 64,
# subtracts before its MMAs and is checked too).
SHIFTED = [(1, 14336, 4096), (16, 14336, 4096), (16, 11008, 1024), (40, 14336, 1024), (100, 14336, 512)]


@pytest.mark.parametrize("kind", ["normal_mean2", "uniform01"])
@pytest.mark.parametrize("M,K,N", SHIFTED)
def test_int8_shifted_activations_long_k(wq, kind, M, K, N):
    base = workloads.w8a16_case(M, K, N, seed=13)
    case = workloads.WeightOnlyCase(workloads.activations_fp16_shifted(M, K, kind, seed=13), base.w, base.scales, 8)
    assert_gemm_close(_run(wq, 8, case), _ref(8, case), "fp16")


@pytest.mark.parametrize("kind", ["normal_mean2", "uniform01"])
@pytest.mark.parametrize("M,K,N", SHIFTED)
def test_int8_shifted_activations_grouped_zero_points(wq, kind, M, K, N):
    g = workloads.grouped_case(8, M, K, N, 128, True, seed=17)
    x = workloads.activations_fp16_shifted(M, K, kind, seed=17)
    y = wq.wq_gemm_w8a16_grouped(torch.from_numpy(x).cuda(), torch.from_numpy(g.w).cuda(),
                                 torch.from_numpy(g.scales).cuda(), torch.from_numpy(g.zeros).cuda(), 128)
    torch.cuda.synchronize()
    assert_gemm_close(y, O.gemm_w8a16_grouped(x, g.w, g.scales, g.zeros, 128), "fp16")


@pytest.mark.parametrize("bits,M,K,N", [(8, 16, 4096, 512), (4, 1, 11008, 512), (4, 16, 4096, 256)])
def test_split_k_workspace_contract(wq, bits, M, K, N):
    """Split tiles need scratch; a call leaves the counter area (the first
    64 KiB) zero again, repeated calls are bit-identical (fixed reduction
    order), and a short buffer is refused before any launch."""
    op = wq.WQ_OP_W4A16 if bits == 4 else wq.WQ_OP_W8A16
    need = wq.wq_workspace_size(op, M, N, K)
    assert need > 0
    case = _case(bits, M, K, N, seed=5)
    x = torch.from_numpy(case.x).cuda()
    w = torch.from_numpy(case.w).cuda()
    s = torch.from_numpy(case.scales).cuda()
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    fn = wq.wq_gemm_w4a16 if bits == 4 else wq.wq_gemm_w8a16
    y1 = fn(x, w, s, workspace=ws)
    torch.cuda.synchronize()
    assert int(ws[: 64 * 1024].count_nonzero()) == 0
    y2 = fn(x, w, s, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert_gemm_close(y1, _ref(bits, case), "fp16")
    with pytest.raises(wq.WqError) as ei:
        fn(x, w, s, workspace=ws[: need - 16])
    assert ei.value.status == wq.WQ_ERR_WORKSPACE
    st, site = wq.wq_get_device_error()
    assert st == wq.WQ_OK and site == 0


@pytest.mark.parametrize("bits,M,K,N", [(8, 16, 4096, 14336), (4, 1, 4096, 11008), (8, 1, 4096, 4096),
                                         (4, 16, 11008, 4096), (8, 9, 1000, 4000)])
def test_cluster_plans(wq, bits, M, K, N):
    """Shapes that the cluster plans (whole tiles per cluster of CTAs, partial
    tiles added in distributed shared memory) may take.  Whatever plan is
    chosen, the call runs with the workspace it asks for and matches the
    oracle; at N = 4096 (32 tiles) the plan is a cluster one and asks for no
    workspace at all."""
    op = wq.WQ_OP_W4A16 if bits == 4 else wq.WQ_OP_W8A16
    need = wq.wq_workspace_size(op, M, N, K)
    if N == 4096:
        assert need == 0
    case = _case(bits, M, K, N, seed=6)
    fn = wq.wq_gemm_w4a16 if bits == 4 else wq.wq_gemm_w8a16
    y = fn(torch.from_numpy(case.x).cuda(), torch.from_numpy(case.w).cuda(), torch.from_numpy(case.scales).cuda())
    torch.cuda.synchronize()
    assert_gemm_close(y, _ref(bits, case, np.arange(M)), "fp16")


@pytest.mark.parametrize("bits", [4, 8])
def test_static_weights_same_bits(wq, bits):
    """With the static-weights promise the decode kernels load their first
    weight boxes before the previous call on the stream has finished.  Calls
    issued back to back (so that launches overlap) give the same bits as
    without the promise, and match the oracle."""
    shapes = [(1, 4096, 4096), (16, 4096, 14336), (4, 1024, 304), (9, 512, 4096)]
    cases = [workloads.w4a16_case(*s, seed=i) if bits == 4 else workloads.w8a16_case(*s, seed=i)
             for i, s in enumerate(shapes)]
    fn = wq.wq_gemm_w4a16 if bits == 4 else wq.wq_gemm_w8a16
    xs = [torch.from_numpy(c.x).cuda() for c in cases]
    ws = [torch.from_numpy(c.w).cuda() for c in cases]
    ss = [torch.from_numpy(c.scales).cuda() for c in cases]

    def sweep():
        return [fn(x, w, s) for _ in range(3) for x, w, s in zip(xs, ws, ss)]

    prev = wq.set_static_weights(True)
    try:
        on = sweep()
    finally:
        wq.set_static_weights(prev)
    off = sweep()
    torch.cuda.synchronize()
    for a, b in zip(on, off):
        assert torch.equal(a, b)
    for c, y in zip(cases, on[:len(cases)]):
        assert_gemm_close(y, _ref(bits, c), "fp16")
