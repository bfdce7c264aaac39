"""GPU parity of the batched weight-only calls (wq_gemm_w4a16_batched,
wq_gemm_w8a16_batched) against the CPU oracle, problem by problem.

Tolerance: |y - y_ref| <= 5e-3 * max|y_ref| + 1 fp16 ulp at y_ref, per element,
every output checked.  The batches cover the decode workloads at full size,
ragged shapes (N inside a 16-column vector, K off the chunk size, several M
tiles), column-grouped scales, padded leading dimensions, empty problems, and
repeated calls on one workspace (deterministic, counters left zero)."""
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


def _cases(bits, shapes, seed=0, group_n=None):
    out = []
    for i, (M, K, N) in enumerate(shapes):
        if group_n:
            out.append(workloads.grouped_case(bits, M, K, N, group_n, False, seed + i))
        else:
            out.append((workloads.w4a16_case if bits == 4 else workloads.w8a16_case)(M, K, N, seed + i))
    return out


def _ref(bits, case, group_n=None):
    if group_n:
        fn = O.gemm_w4a16_grouped if bits == 4 else O.gemm_w8a16_grouped
        return fn(case.x, case.w, case.scales, None, group_n)
    return O.gemm_w4a16(case.x, case.w, case.scales) if bits == 4 else O.gemm_w8a16(case.x, case.w, case.scales)


def _run(wq, bits, cases, group_n=1, pads=None, workspace=None):
    xs, ws, ss, ys = [], [], [], []
    for i, c in enumerate(cases):
        M, K = c.x.shape
        N = c.w.shape[1]
        ldx, ldw, ldy = pads[i] if pads else (None, None, None)
        xs.append(dev_matrix(torch, c.x, ldx))
        ws.append(dev_matrix(torch, c.w, ldw))
        ss.append(torch.from_numpy(c.scales).cuda())
        ys.append(dev_empty(torch, M, N, torch.float16, ldy, fill=float("nan")))
    fn = wq.wq_gemm_w4a16_batched if bits == 4 else wq.wq_gemm_w8a16_batched
    fn(xs, ws, ss, ys=ys, group_n=group_n, workspace=workspace)
    torch.cuda.synchronize()
    return ys


@pytest.mark.parametrize("name", ["w8a16_decode", "w4a16_decode"])
def test_decode_workloads_full_size(wq, name):
    spec = workloads.WORKLOADS[name]
    bits = 8 if spec["op"] == "w8a16" else 4
    cases = _cases(bits, spec["shapes"])
    for c, y in zip(cases, _run(wq, bits, cases)):
        assert_gemm_close(y, _ref(bits, c), "fp16")


RAGGED = [  # (M, K, N, ldx, ldw, ldy)
    (1, 64, 128, None, None, None),
    (3, 96, 257, None, 272, 264),
    (8, 50, 384, 56, 400, 392),
    (16, 2048, 1000, 2056, 1008, 1000),
    (17, 1024, 200, None, 208, 200),      # two M tiles
    (64, 512, 640, None, None, None),     # four M tiles
    (5, 4096, 4096, None, None, None),
    (12, 11008, 640, None, None, None),
]


@pytest.mark.parametrize("bits", [4, 8])
def test_ragged_batch(wq, bits):
    shapes = [(M, K, N) for (M, K, N, *_ ) in RAGGED]
    cases = _cases(bits, shapes, seed=7)
    ys = _run(wq, bits, cases, pads=[p[3:] for p in RAGGED])
    for c, y in zip(cases, ys):
        assert_gemm_close(y, _ref(bits, c), "fp16")


@pytest.mark.parametrize("bits", [4, 8])
def test_small_m_only_batch(wq, bits):
    """All problems at M <= 8 (the 8-row kernel instance)."""
    shapes = [(1, 4096, 4096), (8, 4096, 1408), (4, 2048, 130), (2, 11008, 512)]
    pads = [(None, None, None), (None, None, None), (None, 144, 136), (None, None, None)]
    cases = _cases(bits, shapes, seed=3)
    for c, y in zip(cases, _run(wq, bits, cases, pads=pads)):
        assert_gemm_close(y, _ref(bits, c), "fp16")


@pytest.mark.parametrize("bits", [4, 8])
def test_fewer_units_than_sms(wq, bits):
    """A batch smaller than the GPU: one CTA per unit."""
    cases = _cases(bits, [(1, 64, 128), (2, 128, 256)], seed=11)
    for c, y in zip(cases, _run(wq, bits, cases)):
        assert_gemm_close(y, _ref(bits, c), "fp16")


@pytest.mark.parametrize("bits", [4, 8])
def test_grouped_scales(wq, bits):
    shapes = [(1, 4096, 4096), (16, 4096, 1000), (3, 1024, 300)]
    pads = [(None, None, None), (None, 1008, 1000), (None, 304, 304)]
    cases = _cases(bits, shapes, seed=5, group_n=64)
    for c, y in zip(cases, _run(wq, bits, cases, group_n=64, pads=pads)):
        assert_gemm_close(y, _ref(bits, c, 64), "fp16")


def test_single_problem_matches_oracle(wq):
    cases = _cases(8, [(16, 4096, 14336)], seed=2)
    assert_gemm_close(_run(wq, 8, cases)[0], _ref(8, cases[0]), "fp16")


def test_empty_problems_in_batch(wq):
    """M = 0 and N = 0 problems are skipped; K = 0 gives Y = 0."""
    c = workloads.w8a16_case(4, 256, 384, seed=1)
    x = torch.from_numpy(c.x).cuda()
    w = torch.from_numpy(c.w).cuda()
    s = torch.from_numpy(c.scales).cuda()
    x0 = torch.zeros((0, 256), dtype=torch.float16, device="cuda")
    xk0 = torch.zeros((3, 0), dtype=torch.float16, device="cuda")
    wk0 = torch.zeros((0, 64), dtype=torch.int8, device="cuda")
    yk0 = torch.full((3, 64), float("nan"), dtype=torch.float16, device="cuda")
    ys = wq.wq_gemm_w8a16_batched([x0, x, xk0], [w, w, wk0], [s, s, s[:64]], ys=[None, None, yk0])
    torch.cuda.synchronize()
    assert tuple(ys[0].shape) == (0, 384)
    assert_gemm_close(ys[1], O.gemm_w8a16(c.x, c.w, c.scales), "fp16")
    assert torch.count_nonzero(yk0).item() == 0


@pytest.mark.parametrize("bits", [4, 8])
def test_repeated_calls_deterministic_and_counters_zero(wq, bits):
    """Calls on one workspace give bit-identical results, and every call leaves
    the counter area zero again."""
    cases = _cases(bits, workloads.WORKLOADS["w8a16_decode"]["shapes"][:4], seed=9)
    xs = [torch.from_numpy(c.x).cuda() for c in cases]
    ws = [torch.from_numpy(c.w).cuda() for c in cases]
    ss = [torch.from_numpy(c.scales).cuda() for c in cases]
    if bits == 4:  # INT4 weights of the same K: half the rows
        ws = [torch.from_numpy(workloads.int4_codes_packed(c.x.shape[1], c.w.shape[1], 9)).cuda() for c in cases]
    fn = wq.wq_gemm_w4a16_batched if bits == 4 else wq.wq_gemm_w8a16_batched
    first = fn(xs, ws, ss)
    for _ in range(3):
        again = fn(xs, ws, ss)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    torch.cuda.synchronize()
    buf = wq._WS_CACHE[("counters", torch.cuda.current_device(), torch.cuda.current_stream().cuda_stream)]
    assert torch.count_nonzero(buf[:65536]).item() == 0


def test_matches_single_calls(wq):
    """The batch computes what the single calls compute (within the rounding
    of a different split of the K sums)."""
    cases = _cases(8, [(1, 4096, 4096), (16, 4096, 14336)], seed=4)
    ys = _run(wq, 8, cases)
    for c, y in zip(cases, ys):
        single = wq.wq_gemm_w8a16(torch.from_numpy(c.x).cuda(), torch.from_numpy(c.w).cuda(),
                                  torch.from_numpy(c.scales).cuda())
        torch.cuda.synchronize()
        ref = _ref(8, c)
        tol = O.gemm_tolerance(ref, "fp16")
        diff = np.abs(y.float().cpu().numpy().astype(np.float64) - single.float().cpu().numpy().astype(np.float64))
        assert (diff <= tol).all()
