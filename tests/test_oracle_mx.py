"""Pins of the oracle's MX-style weight-only form (page "11. Inference with
NVFP4/MXFP8", section "MXFP8-Style FP8": e4m3 codes [N, K], one E8M0 scale
byte per 32 codes along K).  The scale of a block is read as the smallest
power of two 2^e with 2^e >= amax / 448, e in [-127, 127]."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synthetic


def _exact_e(amax: float) -> int:
    """Smallest e with 448 * 2^e >= amax, by exact rationals (amax > 0 finite)."""
    a = Fraction(amax)
    e = 0
    while Fraction(448) * Fraction(2) ** e < a:
        e += 1
    while Fraction(448) * Fraction(2) ** (e - 1) >= a:
        e -= 1
    return min(max(e, -127), 127)


def test_e8m0_values_are_powers_of_two():
    for b in range(255):
        assert Fraction(oracle.e8m0_decode(b)) == Fraction(2) ** (b - 127)
    assert math.isnan(oracle.e8m0_decode(255))


@pytest.mark.parametrize("amax,byte", [
    (448.0, 127),                                   # amax / 448 = 1 = 2^0
    (float(np.nextafter(np.float32(448), np.float32(1e9))), 128),
    (224.0, 126),
    (float(np.nextafter(np.float32(224), np.float32(1e9))), 127),
    (1.0, 119),                                     # 448 / 2^8 = 1.75 >= 1 > 0.875
    (0.0, 127),                                     # an all-zero block: 2^0
    (float(np.finfo(np.float32).max), 247),         # 2^119 * 448 < FLT_MAX <= 2^120 * 448
    (1e-45, 0),                                     # below 448 * 2^-127: clamped to 2^-127
    (float("inf"), 255),
])
def test_scale_byte_closed_forms(amax, byte):
    blk = np.zeros(32, np.float32)
    blk[5] = -amax
    assert oracle.mx_scale(blk) == byte


def test_scale_byte_is_the_smallest_power_of_two_not_below_amax_over_448():
    rng = np.random.default_rng(11)
    # magnitudes over the whole fp32 range, and the exact boundaries 448 * 2^e
    # with their neighbours
    mags = np.float32(2.0) ** rng.integers(-149, 127, 400).astype(np.float32) * rng.random(400).astype(np.float32)
    edges = [np.float32(448.0 * 2.0 ** e) for e in range(-120, 110, 7)]
    edges += [np.nextafter(v, np.float32(np.inf)) for v in edges] + [np.nextafter(v, np.float32(0)) for v in edges]
    for a in list(mags) + edges:
        a = np.float32(a)
        blk = np.full(32, a / np.float32(2), np.float32)
        blk[31] = a
        want = 127 if a == 0 else _exact_e(float(a)) + 127
        assert oracle.mx_scale(blk) == want, float(a)


def test_nan_weights_do_not_count_in_the_amax():
    blk = np.full(32, 0.5, np.float32)
    blk[3] = np.nan
    assert oracle.mx_scale(blk) == 118


def test_worked_example_outlier_block():
    """0.5 everywhere, 3 * 448 at column 40 (second block of 32)."""
    w = np.full((1, 128), 0.5, np.float32)
    w[0, 40] = 448.0 * 3.0
    codes, scales = oracle.quantize_mx(w)
    # 0.5 / 448 lies in (2^-10, 2^-9]; 1344 / 448 = 3 lies in (2, 4]
    assert scales.tolist() == [[118, 129, 118, 118]]
    t = oracle.e4m3_decode_table()
    assert np.all(t[codes[0, :32]] == 256.0) and np.all(t[codes[0, 64:]] == 256.0)
    # the outlier block: 1344 / 4 = 336, the midpoint of 320 and 352: even mantissa, 320
    assert t[codes[0, 40]] == 320.0
    # 0.5 / 4 = 0.125 is an e4m3 value
    assert np.all(t[np.delete(codes[0, 32:64], 8)] == 0.125)


def test_no_block_is_clipped():
    """Every |w| / 2^e is at most 448, and a block's largest reaches at
    least 224 unless its scale is clamped at 2^-127 (a floor-based exponent,
    the other common choice, fails the first)."""
    w = np.concatenate([synthetic.weight_outlier(3, 8, 512), synthetic.weight_normal(4, 8, 512, 0.02)])
    codes, scales = oracle.quantize_mx(w)
    blocks = w.reshape(-1, 32).astype(np.float64)
    s = np.array([oracle.e8m0_decode(b) for b in scales.reshape(-1)])
    q = np.abs(blocks) / s[:, None]
    assert np.all(q <= 448.0)
    amax = np.max(np.abs(blocks), axis=1)
    live = (amax > 0) & (scales.reshape(-1) > 0)
    assert np.all(np.max(q, axis=1)[live] > 224.0)
    t = oracle.e4m3_decode_table()
    dec = np.abs(t[codes.reshape(-1, 32)])
    assert np.all(np.max(dec, axis=1)[live] >= 224.0)


def test_codes_are_the_e4m3_of_the_fp32_quotient():
    w = synthetic.weight_outlier(21, 6, 256)
    codes, scales = oracle.quantize_mx(w)
    for r in range(6):
        for j in range(8):
            e = _exact_e(float(np.max(np.abs(w[r, 32 * j:32 * j + 32])))) if np.any(w[r, 32 * j:32 * j + 32]) else 0
            assert scales[r, j] == e + 127
            q = (w[r, 32 * j:32 * j + 32] / np.float32(2.0 ** e)).astype(np.float32)
            assert np.array_equal(codes[r, 32 * j:32 * j + 32], oracle.e4m3_encode(q))


def test_power_of_two_block_scales_give_the_grouped_quantiser():
    """Where every block's amax / 448 is a power of two, the MX form and the
    per-group form (g = 32) pick the same scales and codes."""
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((6, 256)) * 0.1).astype(np.float32)
    blocks = w.reshape(-1, 32)
    for i, blk in enumerate(blocks):
        j = int(np.argmax(np.abs(blk)))
        blk[j] = np.float32(448.0 * 2.0 ** (i % 9 - 12)) * np.sign(blk[j])
        others = np.arange(32) != j
        blk[others] = np.clip(blk[others], -abs(blk[j]) / 2, abs(blk[j]) / 2)
    cm, sm = oracle.quantize_mx(w)
    cg, sg = oracle.quantize_grouped(w, 32)
    assert np.array_equal(cm, cg)
    assert np.array_equal(np.vectorize(oracle.e8m0_decode)(sm).astype(np.float32), sg)


def test_infinite_block_takes_the_nan_scale_and_nan_codes():
    w = np.full((1, 64), 0.25, np.float32)
    w[0, 7] = np.inf
    codes, scales = oracle.quantize_mx(w)
    assert scales.tolist() == [[255, 117]]          # 0.25 / 448 lies in (2^-11, 2^-10]
    assert np.all(codes[0, :32] == 0x7F)
    x = synthetic.to_bf16_bits(np.ones((1, 64), np.float32))
    y = oracle.linear_mx(x, oracle.ACT_BF16, codes, scales)
    assert (int(y[0, 0]) & 0x7FFF) > 0x7F80          # NaN


def test_mx_linear_equals_exact_rationals():
    rng = np.random.default_rng(8)
    m, n, k = 2, 3, 96
    x = synthetic.to_bf16_bits(rng.standard_normal((m, k)).astype(np.float32))
    codes = rng.integers(0, 0x7E, size=(n, k), dtype=np.uint8) | rng.integers(0, 2, size=(n, k), dtype=np.uint8) << 7
    scales = rng.integers(100, 140, size=(n, k // 32), dtype=np.uint8)
    scales[0, 0], scales[1, 2] = 0, 254          # 2^-127 and 2^127 are exact
    bias = rng.standard_normal(n).astype(np.float32)
    y, acc = oracle.linear_mx(x, oracle.ACT_BF16, codes, scales, bias, want_acc=True)
    t = oracle.e4m3_decode_table()
    xv = oracle.act_values(x, oracle.ACT_BF16)
    for i in range(m):
        for r in range(n):
            exact = Fraction(float(bias[r]))
            for j in range(k // 32):
                part = sum(Fraction(float(xv[i, c])) * Fraction(float(t[codes[r, c]])) for c in range(32 * j, 32 * j + 32))
                exact += Fraction(2) ** (int(scales[r, j]) - 127) * part
            assert abs(acc[i, r] - float(exact)) <= 1e-12 * abs(float(exact)) + 1e-300
