"""Pins for the CPU oracle: each check ties an oracle function to something
other than itself (hand-worked examples in ``tests/golden/``, brute force with
exact rational arithmetic, closed forms, and library routines).  The mutation
tests at the end plant plausible mistakes in the oracle and show that at least
one pin catches each of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import wq_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# E2M1 magnitudes, sign and magnitude index per code, as the MXFP4 page lists
# the grid; used only by the brute-force searches below.
_E2M1_EXACT = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2),
               Fraction(2), Fraction(3), Fraction(4), Fraction(6)]


def _e2m1_exact(code):
    v = _E2M1_EXACT[code & 7]
    return -v if code & 8 else v


def _frac(x):
    return Fraction(float(x))


# ------------------------------------------------------------ weight-only pins


def check_w4_worked(gemm=None):
    gemm = gemm or O.gemm_w4a16
    g = _load("weight_only_worked.json")["w4a16"]
    y = gemm(np.array(g["x"], np.float16), np.array(g["w_bytes"], np.uint8), np.array(g["scales"], np.float16))
    np.testing.assert_array_equal(y, np.array(g["y"]))


def check_w8_worked(gemm=None):
    gemm = gemm or O.gemm_w8a16
    g = _load("weight_only_worked.json")["w8a16"]
    y = gemm(np.array(g["x"], np.float16), np.array(g["w"], np.int8), np.array(g["scales"], np.float16))
    np.testing.assert_array_equal(y, np.array(g["y"]))


def test_w4_worked_example():
    check_w4_worked()


def test_w8_worked_example():
    check_w8_worked()


def _brute_w4(x, wq, s):
    m, k = x.shape
    n = wq.shape[1]
    out = np.zeros((m, n))
    for i in range(m):
        for j in range(n):
            acc = Fraction(0)
            for kk in range(k):
                byte = int(wq[kk // 2, j])
                code = (byte >> 4) if kk % 2 else (byte & 15)
                acc += _frac(x[i, kk]) * (code - 8) * _frac(s[j])
            out[i, j] = float(acc)
    return out


def check_w4_bruteforce(gemm=None):
    gemm = gemm or O.gemm_w4a16
    rng = np.random.default_rng(7)
    x = rng.standard_normal((2, 64)).astype(np.float16)
    wq = rng.integers(0, 256, (32, 5), dtype=np.uint8)
    s = rng.uniform(0.005, 0.02, 5).astype(np.float16)
    np.testing.assert_allclose(gemm(x, wq, s), _brute_w4(x, wq, s), rtol=1e-13, atol=1e-15)


def test_w4_bruteforce_exact_rational():
    check_w4_bruteforce()


def test_w8_bruteforce_exact_rational():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((2, 64)).astype(np.float16)
    w = rng.integers(-128, 128, (64, 5)).astype(np.int8)
    s = rng.uniform(0.001, 0.01, 5).astype(np.float16)
    ref = np.zeros((2, 5))
    for i in range(2):
        for j in range(5):
            ref[i, j] = float(sum(_frac(x[i, k]) * int(w[k, j]) * _frac(s[j]) for k in range(64)))
    np.testing.assert_allclose(O.gemm_w8a16(x, w, s), ref, rtol=1e-13, atol=1e-15)


def test_w4_integer_special_case():
    """Unit scales and integer activations: the result is an exact integer that an
    integer matmul of the unpacked codes reproduces."""
    rng = np.random.default_rng(9)
    xi = rng.integers(-4, 5, (3, 40))
    codes = rng.integers(0, 16, (40, 6))
    wq = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    y = O.gemm_w4a16(xi.astype(np.float16), wq, np.ones(6, np.float16))
    np.testing.assert_array_equal(y, (xi @ (codes - 8)).astype(np.float64))


def test_w8_full_int8_range_and_sign():
    """-128 and 127 decode to themselves (two's complement, no zero point)."""
    w = np.array([[-128], [127], [-1]], np.int8)
    y = O.gemm_w8a16(np.array([[1, 1, 1]], np.float16), w, np.array([1.0], np.float16))
    assert y[0, 0] == -2.0


# ------------------------------------------- grouped / asymmetric weight-only pins


def check_grouped_worked(gemm4=None, gemm8=None):
    gemm4 = gemm4 or O.gemm_w4a16_grouped
    gemm8 = gemm8 or O.gemm_w8a16_grouped
    g = _load("weight_only_grouped_worked.json")
    a = g["w4a16"]
    y = gemm4(np.array(a["x"], np.float16), np.array(a["w_bytes"], np.uint8), np.array(a["scales"], np.float16),
              np.array(a["zeros"], np.uint8), a["group_n"])
    np.testing.assert_array_equal(y, np.array(a["y"], np.float64))
    b = g["w8a16"]
    y = gemm8(np.array(b["x"], np.float16), np.array(b["w"], np.int8), np.array(b["scales"], np.float16),
              np.array(b["zeros"], np.int8), b["group_n"])
    np.testing.assert_array_equal(y, np.array(b["y"], np.float64))


def test_grouped_worked_example():
    check_grouped_worked()


def _brute_grouped(x, codes, s, z, group_n):
    m, k = x.shape
    n = codes.shape[1]
    out = np.zeros((m, n))
    for i in range(m):
        for j in range(n):
            g = j // group_n
            out[i, j] = float(sum(_frac(x[i, kk]) * (int(codes[kk, j]) - int(z[g])) * _frac(s[g]) for kk in range(k)))
    return out


def check_grouped_bruteforce(gemm4=None, gemm8=None):
    gemm4 = gemm4 or O.gemm_w4a16_grouped
    gemm8 = gemm8 or O.gemm_w8a16_grouped
    rng = np.random.default_rng(11)
    for group_n, n in ((3, 7), (1, 4), (7, 7)):
        groups = -(-n // group_n)
        x = rng.standard_normal((2, 48)).astype(np.float16)
        s = rng.uniform(0.005, 0.02, groups).astype(np.float16)
        codes4 = rng.integers(0, 16, (48, n))
        wq = (codes4[0::2] | (codes4[1::2] << 4)).astype(np.uint8)
        z4 = rng.integers(0, 16, groups).astype(np.uint8)
        np.testing.assert_allclose(gemm4(x, wq, s, z4, group_n), _brute_grouped(x, codes4, s, z4, group_n),
                                   rtol=1e-13, atol=1e-15)
        w8 = rng.integers(-128, 128, (48, n)).astype(np.int8)
        z8 = rng.integers(-128, 128, groups).astype(np.int8)
        np.testing.assert_allclose(gemm8(x, w8, s, z8, group_n), _brute_grouped(x, w8, s, z8, group_n),
                                   rtol=1e-13, atol=1e-15)


def test_grouped_bruteforce_exact_rational():
    check_grouped_bruteforce()


def test_grouped_reduces_to_per_column_symmetric():
    """One column per group and no zero points is the per-column symmetric GEMM
    (pinned above); a constant zero point equal to the fixed one is too."""
    rng = np.random.default_rng(12)
    x = rng.standard_normal((3, 32)).astype(np.float16)
    wq = rng.integers(0, 256, (16, 6), dtype=np.uint8)
    w8 = rng.integers(-128, 128, (32, 6)).astype(np.int8)
    s = rng.uniform(0.005, 0.02, 6).astype(np.float16)
    np.testing.assert_array_equal(O.gemm_w4a16_grouped(x, wq, s), O.gemm_w4a16(x, wq, s))
    np.testing.assert_array_equal(O.gemm_w4a16_grouped(x, wq, s, np.full(6, 8, np.uint8), 1), O.gemm_w4a16(x, wq, s))
    np.testing.assert_array_equal(O.gemm_w8a16_grouped(x, w8, s), O.gemm_w8a16(x, w8, s))
    np.testing.assert_array_equal(O.gemm_w8a16_grouped(x, w8, s, np.zeros(6, np.int8), 1), O.gemm_w8a16(x, w8, s))


def test_grouped_zero_point_is_a_rank_one_correction():
    """(q - z) s = q s - z s: the zero point subtracts z[g] s[g] sum_k x[m, k]
    from every column of group g (an invariant of the definition)."""
    rng = np.random.default_rng(13)
    x = rng.integers(-3, 4, (2, 16)).astype(np.float16)
    w8 = rng.integers(-128, 128, (16, 5)).astype(np.int8)
    s = np.array([0.5, 0.25], np.float16)
    z = np.array([7, -9], np.int8)
    g = np.arange(5) // 3
    expect = O.gemm_w8a16_grouped(x, w8, s, None, 3) - np.outer(x.astype(np.float64).sum(1),
                                                                 z.astype(np.float64)[g] * s.astype(np.float64)[g])
    np.testing.assert_array_equal(O.gemm_w8a16_grouped(x, w8, s, z, 3), expect)


# ------------------------------------------------------------------ MXFP4 pins


@pytest.mark.parametrize("e", [-126, -30, -29, -3, -1, 0, 1, 20, 100, 127])
def test_ceil_log2_closed_form_around_powers_of_two(e):
    p = np.float32(2.0) ** np.float32(e) if e > -127 else None
    above = np.nextafter(p, np.float32(np.inf))
    below = np.nextafter(p, np.float32(0))
    got = O.ceil_log2_f32(np.array([p, above, below], np.float32))
    assert list(got) == [e, e + 1, e]


def test_ceil_log2_exact_rational_random():
    rng = np.random.default_rng(1)
    bits = rng.integers(0x00800000, 0x7F000000, 4000, dtype=np.uint32)
    q = bits.view(np.float32)
    got = O.ceil_log2_f32(q)
    for qi, ei in zip(q[:4000], got):
        fq = Fraction(float(qi))
        # ceil(log2 q) = e  <=>  2^(e-1) < q <= 2^e
        assert Fraction(2) ** (int(ei) - 1) < fq <= Fraction(2) ** int(ei)


def check_mx_quantize_golden(quant=None):
    quant = quant or O.mx_quantize_fp4
    g = _load("mx_quantize_worked.json")
    for row in g["rows"]:
        x = np.array([[float.fromhex(v) for v in row["values"]]], np.float32)
        data, scales = quant(x)
        assert list(data[0]) == row["data_bytes"], row["why"]
        assert int(scales[0, 0]) == row["E"], row["why"]


def test_mx_quantize_worked_examples():
    check_mx_quantize_golden()


def _brute_mx_block(vals):
    """Independent exhaustive quantizer for one 32-element block: the exponent is
    the smallest integer e with amax/6 <= 2^e (amax clamped at fp32(1e-8)); each
    element takes the code among all 16 whose value times 2^e is nearest, the
    smaller magnitude on a tie, and the sign bit of x < 0."""
    fr = [Fraction(float(v)) for v in vals]
    amax = max(max(abs(v) for v in fr), Fraction(float(np.float32(1e-8))))
    e = -200
    while Fraction(2) ** e < amax / 6:
        e += 1
    codes = []
    for v in fr:
        best = None
        for mag in range(8):
            err = abs(abs(v) - _E2M1_EXACT[mag] * Fraction(2) ** e)
            if best is None or err < best[0]:
                best = (err, mag)
        codes.append((8 if v < 0 else 0) | best[1])
    return codes, e + 127


def check_mx_quantize_bruteforce(quant=None, n_blocks=60):
    quant = quant or O.mx_quantize_fp4
    rng = np.random.default_rng(2)
    rows = []
    for b in range(n_blocks):
        scale = np.float32(2.0) ** np.float32(rng.integers(-40, 40))
        blk = (rng.standard_normal(32) * scale).astype(np.float32)
        if b % 3 == 0:  # plant exact grid midpoints relative to the block scale
            amax = np.float32(np.abs(blk).max())
            e = math.ceil(math.log2(float(amax) / 6.0))
            mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32) * np.float32(2.0 ** e)
            blk[:7] = mids * np.where(rng.random(7) < 0.5, -1, 1).astype(np.float32)
            blk[7] = np.float32(6.0 * 2.0 ** e)
        rows.append(blk)
    x = np.stack(rows)
    data, scales = quant(x)
    codes = O.mx_unpack_codes(data)
    for i in range(n_blocks):
        ref_codes, ref_e = _brute_mx_block(x[i])
        assert int(scales[i, 0]) == ref_e
        assert list(codes[i]) == ref_codes


def test_mx_quantize_bruteforce_exact_rational():
    check_mx_quantize_bruteforce()


def test_mx_quantize_error_bound_invariant():
    """Every element lands within half the local grid spacing (times 2^e) of x."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((16, 256)) * 0.5).astype(np.float32)
    data, scales = O.mx_quantize_fp4(x)
    xhat = O.mx_dequantize(data, scales)
    e = np.repeat(scales.astype(np.int64) - 127, 32, axis=1)
    v = np.abs(x.astype(np.float64)) / np.ldexp(1.0, e)
    assert v.max() <= 6.0
    half_gap = np.select([v <= 2, v <= 4], [0.25, 0.5], 1.0)
    assert np.all(np.abs(x - xhat) <= half_gap * np.ldexp(1.0, e) + 0)


def test_mx_e2m1_decode_all_codes():
    got = O.e2m1_decode(np.arange(16))
    want = [float(_e2m1_exact(c)) for c in range(16)]
    assert list(got) == want
    # each code's value re-quantizes to the same code in a block whose amax is 6
    blk = np.zeros((1, 32), np.float32)
    blk[0, :16] = got.astype(np.float32)
    blk[0, 16] = 6.0
    data, scales = O.mx_quantize_fp4(blk)
    codes = O.mx_unpack_codes(data)[0, :16]
    expect = [c if c != 8 else 0 for c in range(16)]  # -0.0 carries no sign bit
    assert list(codes) == expect and int(scales[0, 0]) == 127


def _one_block(code, e):
    return np.full((1, 16), code | (code << 4), np.uint8), np.array([[e]], np.uint8)


@pytest.mark.parametrize("ea,ew", [(0, 0), (0, 254), (254, 254), (127, 127), (1, 253), (98, 140), (200, 3)])
def test_mx_gemm_e8m0_exponent_addition(ea, ew):
    """S_A * S_W = 2^(E_A + E_W - 254): a block of +1.0 codes on both sides gives
    32 * 2^(E_A + E_W - 254) exactly."""
    ad, asc = _one_block(2, ea)
    wd, wsc = _one_block(2, ew)
    c = O.mx_gemm_fp4(ad, asc, wd, wsc)
    assert c[0, 0] == math.ldexp(32.0, ea + ew - 254)


def test_mx_e8m0_identity_exhaustive():
    """2^(E_A-127) * 2^(E_W-127) == 2^(E_A+E_W-254) for every E_A, E_W in 0..254."""
    ea = np.arange(255)[:, None]
    ew = np.arange(255)[None, :]
    lhs = np.ldexp(1.0, ea - 127) * np.ldexp(1.0, ew - 127)
    rhs = np.ldexp(1.0, ea + ew - 254)
    assert np.array_equal(lhs, rhs)


def check_mx_gemm_worked(gemm=None):
    gemm = gemm or O.mx_gemm_fp4
    g = _load("mx_gemm_worked.json")
    c = gemm(np.array(g["a_data"], np.uint8), np.array(g["a_scales"], np.uint8),
             np.array(g["w_data"], np.uint8), np.array(g["w_scales"], np.uint8))
    np.testing.assert_array_equal(c, np.array(g["c"]))


def test_mx_gemm_worked_example():
    check_mx_gemm_worked()


def check_mx_gemm_bruteforce(gemm=None):
    """2 x 64 against 2 x 64, the MXFP4 page's own demo shape, in exact rationals."""
    gemm = gemm or O.mx_gemm_fp4
    rng = np.random.default_rng(4)
    ad = rng.integers(0, 256, (2, 32), dtype=np.uint8)
    wd = rng.integers(0, 256, (3, 32), dtype=np.uint8)
    asc = rng.integers(110, 140, (2, 2), dtype=np.uint8)
    wsc = rng.integers(110, 140, (3, 2), dtype=np.uint8)
    ref = np.zeros((2, 3))
    for m in range(2):
        for n in range(3):
            acc = Fraction(0)
            for kb in range(2):
                dot = Fraction(0)
                for i in range(32):
                    t = kb * 16 + i // 2
                    ca = (int(ad[m, t]) >> 4) if i % 2 else (int(ad[m, t]) & 15)
                    cw = (int(wd[n, t]) >> 4) if i % 2 else (int(wd[n, t]) & 15)
                    dot += _e2m1_exact(ca) * _e2m1_exact(cw)
                acc += dot * Fraction(2) ** (int(asc[m, kb]) + int(wsc[n, kb]) - 254)
            ref[m, n] = float(acc)
    np.testing.assert_allclose(gemm(ad, asc, wd, wsc), ref, rtol=1e-15, atol=0)


def test_mx_gemm_bruteforce_exact_rational():
    check_mx_gemm_bruteforce()


def test_mx_gemm_equals_dequantize_then_matmul():
    rng = np.random.default_rng(5)
    a = (rng.standard_normal((4, 128)) * 0.5).astype(np.float32)
    w = (rng.standard_normal((6, 128)) * 0.5).astype(np.float32)
    ad, asc = O.mx_quantize_fp4(a)
    wd, wsc = O.mx_quantize_fp4(w)
    c = O.mx_gemm_fp4(ad, asc, wd, wsc)
    np.testing.assert_allclose(c, O.mx_dequantize(ad, asc) @ O.mx_dequantize(wd, wsc).T, rtol=1e-14)
    sub = O.mx_gemm_fp4(ad, asc, wd, wsc, rows=np.array([3, 1]))
    np.testing.assert_array_equal(sub, c[[3, 1]])


# -------------------------------------------------------------------- FP8 pins


def test_e4m3_decode_all_codes_against_torch():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    got = O.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_e4m3_range_closed_form():
    v = O.e4m3_decode(np.arange(256))
    assert np.nanmax(v) == 448.0 and np.nanmin(v) == -448.0
    assert v[0x01] == 2.0 ** -9 and v[0x38] == 1.0 and v[0x08] == 2.0 ** -6
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and np.sum(np.isnan(v)) == 2


def check_fp8_worked(gemm=None):
    gemm = gemm or O.fp8_gemm
    for case in _load("fp8_worked.json")["cases"]:
        c = gemm(np.array(case["a"], np.uint8), np.array(case["b"], np.uint8), case["scale_a"], case["scale_b"])
        np.testing.assert_array_equal(c, np.array(case["c"]))


def test_fp8_worked_examples():
    check_fp8_worked()


def test_fp8_identity_reproduces_b():
    rng = np.random.default_rng(6)
    b = rng.integers(0, 256, (8, 5), dtype=np.uint8)
    b[(b & 0x7F) == 0x7F] = 0x38
    eye = np.where(np.eye(8, dtype=bool), 0x38, 0).astype(np.uint8)
    c = O.fp8_gemm(eye, b, 0.5, 3.0)
    np.testing.assert_array_equal(c, O.e4m3_decode(b) * 1.5)


def test_fp8_bruteforce_exact_rational():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(10)
    a = rng.integers(0, 256, (2, 64), dtype=np.uint8)
    b = rng.integers(0, 256, (64, 3), dtype=np.uint8)
    a[(a & 0x7F) == 0x7F] = 0
    b[(b & 0x7F) == 0x7F] = 0
    dec = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    sa, sb = np.float32(0.37), np.float32(1.9)
    ref = np.zeros((2, 3))
    for m in range(2):
        for n in range(3):
            acc = sum(Fraction(float(dec[a[m, k]])) * Fraction(float(dec[b[k, n]])) for k in range(64))
            ref[m, n] = float(acc * Fraction(float(sa)) * Fraction(float(sb)))
    np.testing.assert_allclose(O.fp8_gemm(a, b, sa, sb), ref, rtol=1e-14, atol=0)


# ----------------------------------------------------------- tolerance helper


# ------------------------------------------------------------------- NVFP4


def _nv_golden():
    with open(os.path.join(GOLDEN, "nvfp4_worked.json")) as f:
        return json.load(f)


def test_e4m3_encode_round_trip_and_midpoints():
    """Every finite non-negative e4m3 value encodes to its own code; a value
    halfway between two neighbours goes to the even code; values from 448 up
    saturate at 0x7E."""
    codes = np.arange(0x7F)
    vals = O.e4m3_decode(codes)
    assert np.array_equal(O.e4m3_encode(vals), codes)
    mids = (vals[:-1] + vals[1:]) / 2
    want = np.where(codes[:-1] % 2 == 0, codes[:-1], codes[1:])
    assert np.array_equal(O.e4m3_encode(mids), want)
    assert (O.e4m3_encode([448.0, 460.0, 1e6]) == 0x7E).all()


def test_e4m3_encode_against_torch():
    """The encoder against PyTorch's float8_e4m3fn cast (round to nearest even)
    on random float32 values below the cast's overflow point."""
    r = np.random.default_rng(5).uniform(0, 463.9, 100000).astype(np.float32)
    r = np.concatenate([r, np.ldexp(np.float32(1), np.arange(-12, 9)).astype(np.float32)])
    ref = torch.from_numpy(r).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(r), ref)


def check_nv_quantize_golden(quant=None):
    quant = quant or O.nv_quantize_fp4
    q = _nv_golden()["quantize"]
    src = np.array(q["src"], dtype=np.float32)
    src[0, 21] = np.float32(-0.0)
    d, s, g = quant(src)
    assert float(g) == q["g"]
    assert np.array_equal(d, np.array(q["data"], np.uint8))
    assert np.array_equal(s, np.array(q["scales"], np.uint8))
    assert np.array_equal(O.nv_dequantize(d, s, g)[0], np.array(q["dequantized_row0"]))


def test_nv_quantize_worked_example():
    check_nv_quantize_golden()


def _nv_bruteforce(src):
    """Exhaustive reference on a small tensor: for every element, search all 16
    codes for the one whose value (times the block's decoded scale and g, in
    exact rationals) is nearest to x / (s g) computed in float32, preferring
    the smaller magnitude on ties."""
    x = np.asarray(src, dtype=np.float32)
    g = O.nv_tensor_scale(x)
    rows, cols = x.shape
    codes = np.zeros((rows, cols), np.int64)
    scales = np.zeros((rows, cols // 16), np.uint8)
    for r in range(rows):
        for b in range(cols // 16):
            blk = x[r, 16 * b:16 * b + 16]
            sb_f = np.float32(np.abs(blk).max() / np.float32(np.float32(6) * g))
            sb = int(O.e4m3_encode([sb_f])[0])
            scales[r, b] = sb
            d = np.float32(np.float32(O.e4m3_decode(np.array([sb]))[0]) * g)
            for i, xv in enumerate(blk):
                if d == 0:
                    continue
                v = Fraction(float(np.float32(xv / d)))
                best = None
                for mag in range(8):
                    dist = abs(abs(v) - Fraction(O.E2M1_GRID[mag]))
                    if best is None or dist < best[0]:
                        best = (dist, mag)
                codes[r, 16 * b + i] = (8 if xv < 0 else 0) | best[1]
    data = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return data, scales, g


def check_nv_quantize_bruteforce(quant=None):
    quant = quant or O.nv_quantize_fp4
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((3, 64)) * rng.choice([1e-3, 1.0, 300.0], size=(3, 1))).astype(np.float32)
    x[0, :16] = np.float32([0.75, 1.75, 3.5, -0.25, 5.0, 2.5, 1.25, 6.0, 0, 0, 0, 0, 0, 0, 0, 0.1])
    d, s, g = quant(x)
    rd, rs, rg = _nv_bruteforce(x)
    assert g == rg and np.array_equal(s, rs) and np.array_equal(d, rd)


def test_nv_quantize_bruteforce_exact_rational():
    check_nv_quantize_bruteforce()


def test_nv_quantize_error_bound_invariant():
    """|x - x_hat| <= half the local grid spacing at the block's scale, plus
    the clamp when the rounded block scale fell below amax / 6."""
    x = (np.random.default_rng(8).standard_normal((16, 256)) * 3).astype(np.float32)
    d, s, g = O.nv_quantize_fp4(x)
    xh = O.nv_dequantize(d, s, g)
    scale = np.repeat(O.e4m3_decode(s), 16, axis=1) * float(g)
    v = np.abs(x.astype(np.float64)) / scale
    half_step = np.where(v < 2, 0.25, np.where(v < 4, 0.5, 1.0))
    bound = (half_step + np.maximum(v - 6.0, 0)) * scale
    assert (np.abs(xh - x) <= bound * (1 + 1e-6) + 1e-300).all()


def check_nv_gemm_worked(gemm=None):
    gemm = gemm or O.nv_gemm_fp4
    q = _nv_golden()["gemm"]
    c = gemm(np.array(q["a_data"], np.uint8), np.array(q["a_scales"], np.uint8), q["ga"],
             np.array(q["w_data"], np.uint8), np.array(q["w_scales"], np.uint8), q["gw"])
    assert np.array_equal(c, np.array(q["c"]))


def test_nv_gemm_worked_example():
    check_nv_gemm_worked()


def check_nv_gemm_bruteforce(gemm=None):
    """2 x 64 operands (the MXFP4 page's demo shape) in exact rationals."""
    gemm = gemm or O.nv_gemm_fp4
    rng = np.random.default_rng(9)
    a = rng.standard_normal((2, 64)).astype(np.float32)
    w = (rng.standard_normal((2, 64)) * 40).astype(np.float32)
    ad, asc, ga = O.nv_quantize_fp4(a)
    wd, wsc, gw = O.nv_quantize_fp4(w)
    ca, cw = O.mx_unpack_codes(ad), O.mx_unpack_codes(wd)
    out = np.zeros((2, 2))
    for m in range(2):
        for n in range(2):
            tot = Fraction(0)
            for k in range(64):
                b = k // 16
                tot += (Fraction(float(O.e2m1_decode(ca[m, k]))) * Fraction(float(O.e2m1_decode(cw[n, k])))
                        * Fraction(float(O.e4m3_decode(asc[m, b]))) * Fraction(float(O.e4m3_decode(wsc[n, b]))))
            out[m, n] = float(tot * Fraction(float(ga)) * Fraction(float(gw)))
    assert np.array_equal(gemm(ad, asc, ga, wd, wsc, gw), out)


def test_nv_gemm_bruteforce_exact_rational():
    check_nv_gemm_bruteforce()


def test_nv_gemm_equals_dequantize_then_matmul():
    rng = np.random.default_rng(10)
    a = rng.standard_normal((5, 256)).astype(np.float32)
    w = rng.standard_normal((7, 256)).astype(np.float32)
    ad, asc, ga = O.nv_quantize_fp4(a)
    wd, wsc, gw = O.nv_quantize_fp4(w)
    ref = O.nv_dequantize(ad, asc, ga) @ O.nv_dequantize(wd, wsc, gw).T
    assert np.allclose(O.nv_gemm_fp4(ad, asc, ga, wd, wsc, gw), ref, rtol=1e-13, atol=0)


def _mutant_nv_block32(src, g=None):
    """Block scales from 32-element blocks (each shared by two 16-element halves)."""
    x = np.asarray(src, np.float32)
    g2 = O.nv_tensor_scale(x) if g is None else np.float32(g)
    amax32 = np.repeat(np.abs(x.reshape(x.shape[0], -1, 32)).max(axis=-1), 2, axis=1)
    sb = O.e4m3_encode((amax32 / np.float32(np.float32(6) * g2)).astype(np.float32))
    d = (O.e4m3_decode(sb).astype(np.float32) * g2).astype(np.float32)
    blocks = x.reshape(x.shape[0], -1, 16)
    v = (blocks / np.where(d > 0, d, 1)[..., None]).astype(np.float32)
    grid = np.asarray(O.E2M1_GRID, np.float32)
    j = np.argmin(np.abs(np.abs(v)[..., None] - grid), axis=-1)
    codes = np.where((d > 0)[..., None], ((blocks < 0) << 3) | j, 0).reshape(x.shape).astype(np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8), sb, g2


def _mutant_nv_ties_up(src, g=None):
    x = np.asarray(src, np.float32)
    d, s, g2 = O.nv_quantize_fp4(x, g)
    return O.nv_quantize_fp4((x * np.float32(1.0000001)).astype(np.float32), g2)


def _mutant_nv_no_tensor_scale(src, g=None):
    return O.nv_quantize_fp4(src, np.float32(1.0))


def _mutant_nv_scale_floor(src, g=None):
    x = np.asarray(src, np.float32)
    _, _, g2 = O.nv_quantize_fp4(x, g)
    blocks = x.reshape(x.shape[0], -1, 16)
    sb_f = (np.abs(blocks).max(axis=-1) / np.float32(np.float32(6) * g2)).astype(np.float32)
    table = O.e4m3_decode(np.arange(0x7F))
    sb = np.clip(np.searchsorted(table, sb_f, side="right") - 1, 0, 0x7E).astype(np.uint8)
    d = (O.e4m3_decode(sb).astype(np.float32) * g2).astype(np.float32)
    out = O.nv_quantize_fp4(x, g2)
    return out[0] if (d == 0).all() else out[0], sb, g2


def _mutant_nv_gemm_no_tensor_scales(ad, asc, ga, wd, wsc, gw, rows=None):
    return O.nv_gemm_fp4(ad, asc, 1.0, wd, wsc, 1.0, rows)


def _mutant_nv_gemm_w_nibbles_swapped(ad, asc, ga, wd, wsc, gw, rows=None):
    """W's element pairs read in the wrong order (A's in the right one)."""
    sw = ((np.asarray(wd, np.uint8) >> 4) | (np.asarray(wd, np.uint8) << 4)).astype(np.uint8)
    return O.nv_gemm_fp4(ad, asc, ga, sw, wsc, gw, rows)


@pytest.mark.parametrize("mutant,checks", [
    (_mutant_nv_block32, [check_nv_quantize_golden, check_nv_quantize_bruteforce]),
    (_mutant_nv_ties_up, [check_nv_quantize_golden]),
    (_mutant_nv_no_tensor_scale, [check_nv_quantize_bruteforce]),
    (_mutant_nv_scale_floor, [check_nv_quantize_golden, check_nv_quantize_bruteforce]),
])
def test_nv_quantize_pins_catch_planted_mistakes(mutant, checks):
    for check in checks:
        with pytest.raises(AssertionError):
            check(mutant)


@pytest.mark.parametrize("mutant", [_mutant_nv_gemm_no_tensor_scales, _mutant_nv_gemm_w_nibbles_swapped])
def test_nv_gemm_pins_catch_planted_mistakes(mutant):
    for check in (check_nv_gemm_worked, check_nv_gemm_bruteforce):
        with pytest.raises(AssertionError):
            check(mutant)


def _tolerance_golden():
    import json

    with open(os.path.join(GOLDEN, "tolerance_worked.json")) as f:
        return json.load(f)


def check_tolerance_worked(tol_fn):
    g = _tolerance_golden()
    y = np.array(g["y_ref"], dtype=np.float64)
    for dtype, want in g["tol"].items():
        assert np.array_equal(tol_fn(y, dtype), np.array(want)), dtype
    t = g["tiny_fp16"]
    want = np.array(t["tol"]) + t["first_term"]
    assert np.allclose(tol_fn(np.array(t["y_ref"]), "fp16"), want, rtol=1e-12, atol=0)


def test_gemm_tolerance_worked_example():
    """The comparison rule every GPU parity test rests on, against hand-worked
    values (tests/golden/tolerance_worked.json)."""
    check_tolerance_worked(O.gemm_tolerance)


def _mutant_tol_per_element(y_ref, dtype, rel=5e-3):
    y = np.asarray(y_ref, dtype=np.float64)
    return rel * np.abs(y) + O.ulp(y, dtype)


def _mutant_tol_row_max(y_ref, dtype, rel=5e-3):
    y = np.asarray(y_ref, dtype=np.float64)
    return rel * np.abs(y).max(axis=-1, keepdims=True) + O.ulp(y, dtype)


def _mutant_tol_ulp_no_subnormal(y_ref, dtype, rel=5e-3):
    y = np.asarray(y_ref, dtype=np.float64)
    mant = {"fp16": 10, "bf16": 7, "fp32": 23}[dtype]
    _, x = np.frexp(np.where(y != 0, np.abs(y), np.finfo(np.float64).tiny))
    return rel * np.abs(y).max() + np.ldexp(1.0, (x - 1 - mant).astype(np.int64))


def _mutant_tol_ulp_exponent_off(y_ref, dtype, rel=5e-3):
    y = np.asarray(y_ref, dtype=np.float64)
    return rel * np.abs(y).max() + 2.0 * O.ulp(y, dtype)


@pytest.mark.parametrize("mutant", [_mutant_tol_per_element, _mutant_tol_row_max, _mutant_tol_ulp_no_subnormal,
                                    _mutant_tol_ulp_exponent_off])
def test_gemm_tolerance_pin_catches_planted_mistakes(mutant):
    with pytest.raises(AssertionError):
        check_tolerance_worked(mutant)


def test_ulp_matches_numpy_spacing():
    for dt, name in ((np.float16, "fp16"), (np.float32, "fp32")):
        vals = np.array([1.0, 1.5, 1000.0, 3e-3, 0.0, -7.25], dt)
        np.testing.assert_array_equal(O.ulp(vals, name), np.abs(np.spacing(np.abs(vals))).astype(np.float64))
    assert O.ulp(np.array([1.0]), "bf16")[0] == 2.0 ** -7


# -------------------------------------------------------------- mutation tests
# Each plants one plausible mistake in the oracle (on the CPU) and checks that
# the pins above catch it.


def _mutant_w4_swapped_nibbles(x, wq, s):
    q = O.unpack_int4(wq)
    q2 = q.copy()
    q2[0::2], q2[1::2] = q[1::2], q[0::2]
    return x.astype(np.float64) @ ((q2 - 8) * s.astype(np.float64))


def _mutant_w4_zero_point_7(x, wq, s):
    return x.astype(np.float64) @ ((O.unpack_int4(wq) - 7) * s.astype(np.float64))


def _mutant_w4_transposed_scale(x, wq, s):
    return x.astype(np.float64) @ (O.unpack_int4(wq) - 8).astype(np.float64) * float(s.astype(np.float64).mean())


def _mutant_mx_ties_up(src):
    x = np.asarray(src, np.float32)
    rows, cols = x.shape
    blocks = x.reshape(rows, cols // 32, 32)
    amax = np.maximum(np.abs(blocks).max(-1), O.AMAX_FLOOR)
    e = O.ceil_log2_f32((amax / np.float32(6)).astype(np.float32))
    v = np.abs(blocks / np.ldexp(np.float32(1), e)[..., None])
    grid = np.asarray(O.E2M1_GRID, np.float32)
    dist = np.abs(v[..., None] - grid)
    j = 7 - np.argmin(dist[..., ::-1], axis=-1)  # last index on ties
    codes = (((blocks < 0).astype(np.uint8) << 3) | j.astype(np.uint8)).reshape(rows, cols)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8), (e + 127).astype(np.uint8)


def _mutant_mx_floor_exponent(src):
    x = np.asarray(src, np.float32)
    d, s = O.mx_quantize_fp4(x)
    amax = np.maximum(np.abs(x.reshape(x.shape[0], -1, 32)).max(-1), O.AMAX_FLOOR)
    e = np.floor(np.log2(amax / 6.0)).astype(np.int64)
    return d, (e + 127).astype(np.uint8)


def _mutant_mx_no_clamp(src):
    x = np.asarray(src, np.float32)
    saved = O.AMAX_FLOOR
    try:
        O.AMAX_FLOOR = np.float32(1e-38)
        return O.mx_quantize_fp4(x)
    finally:
        O.AMAX_FLOOR = saved


def _mutant_mx_gemm_bias_127(ad, asc, wd, wsc, rows=None):
    return O.mx_gemm_fp4(ad, asc, wd, wsc) * 2.0 ** 127


def _mutant_mx_gemm_transposed_blocks(ad, asc, wd, wsc, rows=None):
    return O.mx_gemm_fp4(ad, asc[:, ::-1], wd, wsc)


def _mutant_fp8_no_subnormals(a, b, sa, sb, rows=None):
    da = O.e4m3_decode(a)
    da = np.where((np.asarray(a) & 0x78) == 0, 0.0, da)
    return (da @ O.e4m3_decode(b)) * sa * sb


def _mutant_grouped_zero_sign(x, w, s, z=None, group_n=1, four=False):
    q = O.unpack_int4(w) if four else np.asarray(w, np.int8).astype(np.int64)
    g = np.arange(q.shape[1]) // group_n
    zz = np.full(q.shape[1], 8 if four else 0) if z is None else np.asarray(z).astype(np.int64)[g]
    return x.astype(np.float64) @ ((q + zz) * s.astype(np.float64)[g])


def _mutant_grouped_interleaved(x, w, s, z=None, group_n=1, four=False):
    q = O.unpack_int4(w) if four else np.asarray(w, np.int8).astype(np.int64)
    groups = -(-q.shape[1] // group_n)
    g = np.arange(q.shape[1]) % groups  # columns dealt round-robin instead of in runs
    zz = np.full(q.shape[1], 8 if four else 0) if z is None else np.asarray(z).astype(np.int64)[g]
    return x.astype(np.float64) @ ((q - zz) * s.astype(np.float64)[g])


def _mutant_grouped_k_axis(x, w, s, z=None, group_n=1, four=False):
    q = O.unpack_int4(w) if four else np.asarray(w, np.int8).astype(np.int64)
    g = np.minimum(np.arange(q.shape[0]) // group_n, len(s) - 1)  # grouped along K instead of N
    zz = np.full(q.shape[0], 8 if four else 0) if z is None else np.asarray(z).astype(np.int64)[g]
    return x.astype(np.float64) @ ((q - zz[:, None]) * s.astype(np.float64)[g][:, None])


@pytest.mark.parametrize("mutant", [_mutant_grouped_zero_sign, _mutant_grouped_interleaved, _mutant_grouped_k_axis])
@pytest.mark.parametrize("which", ["w4", "w8"])
def test_grouped_pins_catch_planted_mistakes(mutant, which):
    four = which == "w4"
    g4 = (lambda *a: mutant(*a, four=True)) if four else O.gemm_w4a16_grouped
    g8 = O.gemm_w8a16_grouped if four else (lambda *a: mutant(*a, four=False))
    caught = 0
    for check in (check_grouped_worked, check_grouped_bruteforce):
        try:
            check(g4, g8)
        except AssertionError:
            caught += 1
    assert caught >= 1


@pytest.mark.parametrize("mutant,checks", [
    (_mutant_w4_swapped_nibbles, [check_w4_worked, check_w4_bruteforce]),
    (_mutant_w4_zero_point_7, [check_w4_worked, check_w4_bruteforce]),
    (_mutant_w4_transposed_scale, [check_w4_worked, check_w4_bruteforce]),
    (_mutant_mx_ties_up, [check_mx_quantize_golden, check_mx_quantize_bruteforce]),
    (_mutant_mx_floor_exponent, [check_mx_quantize_golden, check_mx_quantize_bruteforce]),
    (_mutant_mx_no_clamp, [check_mx_quantize_golden]),
    (_mutant_mx_gemm_bias_127, [check_mx_gemm_worked, check_mx_gemm_bruteforce]),
    (_mutant_mx_gemm_transposed_blocks, [check_mx_gemm_worked, check_mx_gemm_bruteforce]),
    (_mutant_fp8_no_subnormals, [check_fp8_worked]),
])
def test_pins_catch_planted_mistakes(mutant, checks):
    for check in checks:
        with pytest.raises(AssertionError):
            check(mutant)


# ---------------------------------------------------------------- tensor-core scale layout
# Offsets worked by hand from the layout's definition (row group g = r // 128,
# chunk c = b // 4, kc chunks per group):
#   offset = 512 (g kc + c) + 16 (r % 32) + 4 ((r // 32) % 4) + b % 4.
# MXFP4, rows 300, K 512: 16 blocks per row, K pads to 512 = 2 steps of 256,
# kc = 2 * 8 / 4 = 4 chunks per group; rows pad to 512, 4 groups, 8192 bytes.
_TC_MX_CASES = [
    (0, 0, 0),
    (33, 5, 512 + 16 + 4 + 1),                     # g 0, c 1, line 1, word 1, byte 1
    (200, 9, (1 * 4 + 2) * 512 + 16 * 8 + 4 * 2 + 1),  # g 1, c 2, line 8, word 2 (200 // 32 = 6), byte 1 = 3209
    (299, 15, (2 * 4 + 3) * 512 + 16 * 11 + 4 * 1 + 3),  # g 2, c 3, line 11, word 1 (299 // 32 = 9), byte 3 = 5815
]


def _tc_scales(rows, nb, lo, hi, seed):
    return np.random.default_rng(seed).integers(lo, hi, size=(rows, nb), dtype=np.uint8)


def test_fp4_scales_tc_worked_offsets():
    s = _tc_scales(300, 16, 1, 127, 11)
    out = O.fp4_scales_tc(s, 512, 32)
    assert out.shape == (8192,)
    for r, b, off in _TC_MX_CASES:
        assert off in (0, 533, 3209, 5815)
        assert out[off] == s[r, b], (r, b, off)
    # padding: row 300 (g 2, line 12, word 1, block 0) and all of group 3 hold 2^0
    assert out[(2 * 4) * 512 + 16 * 12 + 4 * 1] == 0x7F
    assert np.all(out[3 * 4 * 512:] == 0x7F)
    # NVFP4, rows 5, K 80: 5 blocks, K pads to 256 = one step of 16 blocks,
    # kc = 4; rows pad to 256, 2 groups, 4096 bytes.  Row 4, block 4: chunk 1,
    # line 4, word 0, byte 0 -> 512 + 64 = 576; block 5 of row 4 is padding (0).
    sn = _tc_scales(5, 5, 1, 255, 12)
    outn = O.fp4_scales_tc(sn, 80, 16)
    assert outn.shape == (4096,)
    assert outn[576] == sn[4, 4] and outn[577] == 0 and outn[3] == sn[0, 3]


@pytest.mark.parametrize("rows,K,block", [(300, 512, 32), (1, 32, 32), (257, 8192, 32), (5, 80, 16),
                                          (130, 4096, 16)])
def test_fp4_scales_tc_is_a_permutation_plus_padding(rows, K, block):
    """Every scale lands in a distinct byte and everything else is padding:
    the non-padding bytes are exactly the input bytes (as a multiset)."""
    fill = 0x7F if block == 32 else 0x00
    s = _tc_scales(rows, K // block, 1, 127 if block == 32 else 255, rows + K)
    out = O.fp4_scales_tc(s, K, block)
    kept = out[out != fill]
    assert kept.size == s.size
    np.testing.assert_array_equal(np.sort(kept), np.sort(s.ravel()))
