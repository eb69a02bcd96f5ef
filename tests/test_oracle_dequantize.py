"""Pins of the oracle's dequantised weight, scale[n] * e4m3(q[n, k]) in fp64
(page "kadirnar/kernel-agent fp8-weights", section "The contract": the
fallback form), against what the format and the quantiser fix."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synthetic


def test_scale_one_gives_the_decode_table():
    codes = np.arange(256, dtype=np.uint8).reshape(16, 16)
    w = oracle.dequantize(codes, np.ones(16, np.float32))
    t = oracle.e4m3_decode_table()
    finite = np.isfinite(t)
    assert np.array_equal(w.reshape(-1)[finite], t[finite])
    assert np.isnan(w.reshape(-1)[~finite]).all()


def test_matches_an_independent_decode():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 256, size=(8, 64), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x42            # no NaN codes here
    scales = (rng.random(8) * 1e-2 + 1e-4).astype(np.float32)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.dequantize(codes, scales), dec * scales.astype(np.float64)[:, None])


def test_power_of_two_scales_scale_exactly():
    codes = np.arange(0, 126, dtype=np.uint8).reshape(2, 63)
    codes = np.concatenate([codes, np.zeros((2, 1), np.uint8)], axis=1)
    s = np.float32([2.0 ** -20, 2.0 ** 30])
    w = oracle.dequantize(codes, s)
    t = oracle.e4m3_decode_table()
    assert np.array_equal(w, t[codes] * s.astype(np.float64)[:, None])
    assert np.array_equal(w[0] * 2.0 ** 20, t[codes[0]])


def test_quantise_then_dequantise_is_within_half_a_code_step():
    """|w - deq(q(w))| <= half the e4m3 spacing at w times the scale (2^-4
    relative for normal codes, 2^-10 * scale absolute for subnormal ones)."""
    w = synthetic.weight_normal(11, 32, 256, 0.02)
    codes, scales = oracle.quantize(w)
    d = oracle.dequantize(codes, scales)
    s = scales.astype(np.float64)[:, None]
    bound = np.maximum(np.abs(w.astype(np.float64)) * 2.0 ** -4, 2.0 ** -10 * s) * (1 + 1e-6)
    assert np.all(np.abs(w - d) <= bound)


# ---------------------------------------------- per-group and MX scales --

def test_grouped_dequantize_with_equal_group_scales_is_the_per_row_one():
    rng = np.random.default_rng(31)
    codes = rng.integers(0, 256, size=(5, 256), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x11
    s = (rng.random(5) * 3 + 1e-3).astype(np.float32)
    for g in (32, 64, 128):
        d = oracle.dequantize_grouped(codes, np.repeat(s[:, None], 256 // g, axis=1), g)
        assert np.array_equal(d, oracle.dequantize(codes, s))


def test_grouped_and_mx_dequantize_are_exact_products():
    rng = np.random.default_rng(32)
    codes = rng.integers(0, 256, size=(3, 64), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x39
    t = oracle.e4m3_decode_table()
    gs = (rng.random((3, 2)) * 5).astype(np.float32)
    d = oracle.dequantize_grouped(codes, gs, 32)
    e8 = rng.integers(0, 255, size=(3, 2), dtype=np.uint8)
    e8[0, 0], e8[2, 1] = 0, 254
    dm = oracle.dequantize_mx(codes, e8)
    for r in range(3):
        for i in range(64):
            assert Fraction(d[r, i]) == Fraction(float(gs[r, i // 32])) * Fraction(float(t[codes[r, i]]))
            assert Fraction(dm[r, i]) == Fraction(2) ** (int(e8[r, i // 32]) - 127) * Fraction(float(t[codes[r, i]]))


@pytest.mark.parametrize("form", ["g32", "g128", "mx"])
def test_quantise_then_dequantise_is_within_half_a_code_step(form):
    """Each weight comes back within half an e4m3 step of its group's grid:
    2^-4 of |w| in the normal range, 2^-10 * scale below it."""
    w = np.concatenate([synthetic.weight_normal(33, 6, 512, 0.02), synthetic.weight_outlier(34, 6, 512)])
    if form == "mx":
        codes, e8 = oracle.quantize_mx(w)
        d = oracle.dequantize_mx(codes, e8)
        s = np.repeat(np.ldexp(1.0, e8.astype(np.int64) - 127), 32, axis=1)
    else:
        g = int(form[1:])
        codes, gs = oracle.quantize_grouped(w, g)
        d = oracle.dequantize_grouped(codes, gs, g)
        s = np.repeat(gs.astype(np.float64), g, axis=1)
    bound = np.maximum(np.abs(w.astype(np.float64)) * 2.0 ** -4, 2.0 ** -10 * s) * (1 + 1e-6)
    assert np.all(np.abs(w - d) <= bound)
