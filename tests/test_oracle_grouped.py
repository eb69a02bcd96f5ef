"""Pins of the oracle's per-group quantiser and linear layer (page "B04
Precision & Quantization", section "Post-training quantization versus
quantization-aware training": one scale per run of g weights of a row)."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synthetic


def test_one_group_per_row_is_the_per_channel_quantiser():
    w = synthetic.weight_normal(5, 24, 256, 0.02)
    cg, sg = oracle.quantize_grouped(w, 256)
    c, s = oracle.quantize(w)
    assert np.array_equal(cg, c) and np.array_equal(sg[:, 0], s)


@pytest.mark.parametrize("g", [32, 64, 128])
def test_groups_are_independent_per_channel_quantisations(g):
    """Each group equals the per-channel quantiser run on that group alone."""
    w = synthetic.weight_outlier(7, 16, 512)
    cg, sg = oracle.quantize_grouped(w, g)
    seg = w.reshape(16, 512 // g, g).reshape(-1, g)
    c, s = oracle.quantize(seg)
    assert np.array_equal(cg.reshape(-1, g), c) and np.array_equal(sg.reshape(-1), s)


def test_group_scales_are_group_amax_over_448_and_outliers_stay_local():
    w = np.full((1, 128), 0.5, np.float32)
    w[0, 40] = 448.0 * 3.0          # an outlier in the second group of 32
    codes, scales = oracle.quantize_grouped(w, 32)
    assert np.array_equal(scales[0], np.float32([0.5 / 448.0, 3.0, 0.5 / 448.0, 0.5 / 448.0]))
    t = oracle.e4m3_decode_table()
    # the other groups keep full resolution: 0.5 / scale = 448 exactly
    assert np.all(t[codes[0, :32]] == 448.0) and np.all(t[codes[0, 64:]] == 448.0)
    assert t[codes[0, 40]] == 448.0


def test_equal_group_scales_give_the_per_channel_linear():
    rng = np.random.default_rng(9)
    x = synthetic.to_bf16_bits(rng.standard_normal((3, 256)).astype(np.float32))
    codes = rng.integers(0, 0x7E, size=(5, 256), dtype=np.uint8)
    s = np.float32([0.01, 0.02, 0.5, 1.0, 3e-3])
    bias = rng.standard_normal(5).astype(np.float32)
    yg, ag = oracle.linear_grouped(x, oracle.ACT_BF16, codes, np.repeat(s[:, None], 8, axis=1), 32, bias,
                                   want_acc=True)
    y, a = oracle.linear(x, oracle.ACT_BF16, codes, s, bias, want_acc=True)
    assert np.allclose(ag, a, rtol=1e-13, atol=0) and np.count_nonzero(yg != y) <= 1


def test_grouped_linear_equals_exact_rationals():
    rng = np.random.default_rng(2)
    m, n, k, g = 2, 3, 64, 32
    x = synthetic.to_bf16_bits(rng.standard_normal((m, k)).astype(np.float32))
    codes = rng.integers(0, 0x7E, size=(n, k), dtype=np.uint8) | rng.integers(0, 2, size=(n, k), dtype=np.uint8) << 7
    scales = (rng.random((n, k // g)) * 0.1 + 1e-3).astype(np.float32)
    bias = rng.standard_normal(n).astype(np.float32)
    _, acc = oracle.linear_grouped(x, oracle.ACT_BF16, codes, scales, g, bias, want_acc=True)
    t = oracle.e4m3_decode_table()
    xv = oracle.act_values(x, oracle.ACT_BF16)
    for i in range(m):
        for r in range(n):
            exact = Fraction(float(bias[r]))
            for j in range(k // g):
                part = sum(Fraction(float(xv[i, c])) * Fraction(float(t[codes[r, c]])) for c in range(j * g, (j + 1) * g))
                exact += Fraction(float(scales[r, j])) * part
            assert abs(acc[i, r] - float(exact)) <= 1e-12 * max(1.0, abs(float(exact)))
