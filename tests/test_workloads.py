"""The seeded input generators shared by the oracle and the CUDA path: same
seed, same arrays; the value ranges the workloads state; and weights that do
not depend on M (so every M of a sweep multiplies the same matrix)."""
import numpy as np

import workloads


def test_weight_only_cases_are_deterministic_and_in_range():
    a = workloads.w8a16_case(4, 256, 96, seed=3)
    b = workloads.w8a16_case(4, 256, 96, seed=3)
    assert np.array_equal(a.x, b.x) and np.array_equal(a.w, b.w) and np.array_equal(a.scales, b.scales)
    assert a.x.dtype == np.float16 and a.w.dtype == np.int8 and a.scales.dtype == np.float16
    assert a.w.min() >= -127 and a.w.max() <= 127
    assert 0.001 <= float(a.scales.min()) and float(a.scales.max()) <= 0.01 + 1e-5
    c = workloads.w4a16_case(16, 512, 64, seed=0)
    assert c.w.shape == (256, 64) and c.w.dtype == np.uint8
    assert 0.005 <= float(c.scales.min()) and float(c.scales.max()) <= 0.02 + 1e-5


def test_weights_do_not_depend_on_m():
    w1 = workloads.w8a16_case(1, 512, 128, seed=0).w
    w16 = workloads.w8a16_case(16, 512, 128, seed=0).w
    assert np.array_equal(w1, w16)
    assert not np.array_equal(workloads.w8a16_case(1, 512, 128, seed=1).w, w1)


def test_grouped_cases():
    g = workloads.grouped_case(4, 8, 128, 100, 32, True, seed=2)
    assert g.scales.shape == (4,) and g.zeros.shape == (4,) and g.zeros.dtype == np.uint8
    assert g.zeros.max() <= 15
    g8 = workloads.grouped_case(8, 8, 128, 100, 7, True, seed=2)
    assert g8.scales.shape == (15,) and g8.zeros.dtype == np.int8
    assert -32 <= int(g8.zeros.min()) and int(g8.zeros.max()) <= 32
    assert workloads.grouped_case(8, 8, 128, 100, 7, False, seed=2).zeros is None
    again = workloads.grouped_case(8, 8, 128, 100, 7, True, seed=2)
    assert np.array_equal(g8.zeros, again.zeros) and np.array_equal(g8.scales, again.scales)


def test_mx_source_and_fp8_case():
    s = workloads.mx_source(8, 64, seed=0)
    assert s.dtype == np.float32 and s.shape == (8, 64)
    assert np.array_equal(s, workloads.mx_source(8, 64, seed=0))
    f = workloads.fp8_case(16, 64, 32, seed=0)
    assert f.a8.dtype == np.uint8 and f.b8.shape == (64, 32)
    assert f.scale_a > 0 and f.scale_b > 0
    assert not np.any((f.a8 & 0x7F) == 0x7F)  # no e4m3 NaN codes
