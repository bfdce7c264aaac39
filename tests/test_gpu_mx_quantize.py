"""GPU mx_quantize_fp4 against the CPU oracle: bit-exact data and scale bytes."""
import json
import os

import numpy as np
import pytest

import workloads
from oracle import wq_oracle as O
from tests.gpu_util import dev_empty, dev_matrix

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def wq():
    import bit_quantized_gemm_dequant_gb300 as mod

    return mod


def _quant(wq, src, ld_src=None, ld_data=None, ld_scales=None):
    R, C = src.shape
    s = dev_matrix(torch, src, ld_src)
    d = dev_empty(torch, R, C // 2, torch.uint8, ld_data, fill=0xEE)
    e = dev_empty(torch, R, C // 32, torch.uint8, ld_scales, fill=0xEE)
    wq.mx_quantize_fp4(s, d, e)
    torch.cuda.synchronize()
    return d.cpu().numpy(), e.cpu().numpy()


def _assert_exact(got, want):
    gd, ge = got
    rd, re_ = want
    assert np.array_equal(ge, re_), f"scales differ at {np.argwhere(ge != re_)[:5].tolist()}"
    assert np.array_equal(gd, rd), f"data differ at {np.argwhere(gd != rd)[:5].tolist()}"


def test_worked_examples(wq):
    with open(os.path.join(os.path.dirname(__file__), "golden", "mx_quantize_worked.json")) as f:
        g = json.load(f)
    x = np.array([[float.fromhex(v) for v in row["values"]] for row in g["rows"]], np.float32)
    d, e = _quant(wq, x)
    for i, row in enumerate(g["rows"]):
        assert list(d[i]) == row["data_bytes"], row["why"]
        assert int(e[i, 0]) == row["E"], row["why"]


@pytest.mark.parametrize("R,C,ld_src,ld_data,ld_scales", [
    (1, 32, None, None, None), (3, 96, 100, 52, 5), (64, 256, None, None, None),
    (257, 1024, 1028, 516, 33), (1000, 8192, None, None, None)])
def test_random_normal(wq, R, C, ld_src, ld_data, ld_scales):
    src = workloads.mx_source(R, C, seed=R + C)
    _assert_exact(_quant(wq, src, ld_src, ld_data, ld_scales), O.mx_quantize_fp4(src))


def test_wide_dynamic_range_ties_and_zeros(wq):
    """Per-block magnitudes from 2^-140 to 2^120, planted grid midpoints,
    zero blocks, -0.0 and values below the 1e-8 clamp."""
    rng = np.random.default_rng(5)
    R, C = 128, 512
    x = rng.standard_normal((R, C)).astype(np.float32)
    ex = rng.integers(-140, 121, (R, C // 32))
    x *= np.repeat(np.ldexp(np.float32(1), ex), 32, axis=1).astype(np.float32)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], np.float32)
    for r in range(0, R, 3):
        e = int(rng.integers(-20, 20))
        x[r, :8] = mids * np.float32(2.0 ** e) * np.where(rng.random(8) < .5, -1, 1).astype(np.float32)
        x[r, 8:32] = 0
    x[5, 32:64] = 0.0
    x[6, 64:96] = -0.0
    x[7, 96:128] = np.float32(3e-9) * np.sign(rng.standard_normal(32)).astype(np.float32)
    _assert_exact(_quant(wq, x), O.mx_quantize_fp4(x))


def test_one_ulp_around_every_midpoint(wq):
    """Blocks whose amax is exactly 6 * 2^e (so the block scale is 2^e) holding
    each grid midpoint times 2^e and its float32 neighbours on both sides:
    the code choice flips exactly at the midpoints, with ties to the smaller
    magnitude."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    rows = []
    for e in (-12, -1, 0, 3, 17):
        scale = np.float32(2.0 ** e)
        vals = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0))])
        block = np.zeros(32, np.float32)
        block[0] = np.float32(6.0) * scale
        block[1:22] = vals * scale
        block[22:32] = -vals[:10] * scale
        rows.append(block)
        rows.append(-block)
    x = np.stack(rows).repeat(2, axis=1).reshape(len(rows), 64)
    _assert_exact(_quant(wq, x), O.mx_quantize_fp4(x))


def test_large_operand_sampled_rows(wq):
    """The 8192 x 8192 weight operand, checked bit-exact on 256 sampled rows."""
    src = workloads.mx_source(8192, 8192, seed=0, stream=1)
    d, e = _quant(wq, src)
    rows = np.random.default_rng(0).choice(8192, 256, replace=False)
    rd, re_ = O.mx_quantize_fp4(src[rows])
    _assert_exact((d[rows], e[rows]), (rd, re_))
