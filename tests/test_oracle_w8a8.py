"""Pins of the oracle's W8A8 form (page "tensormux Write an FP8 kernel":
per-token activation scales and per-channel weight scales, both amax / 448,
the accumulator multiplied by both)."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synthetic


def test_activation_quantisation_is_the_per_row_rule_on_widened_activations():
    rng = np.random.default_rng(1)
    xb = synthetic.to_bf16_bits(rng.standard_normal((5, 96)).astype(np.float32))
    qx, sx = oracle.quantize_act(xb, oracle.ACT_BF16)
    x = oracle.act_values(xb, oracle.ACT_BF16)
    for i in range(5):
        assert sx[i] == np.float32(np.max(np.abs(x[i]))) / np.float32(448.0)
        assert np.array_equal(qx[i], oracle.e4m3_encode((x[i].astype(np.float32) / sx[i]).astype(np.float32)))


def test_w8a8_equals_exact_rationals():
    rng = np.random.default_rng(2)
    m, n, k = 2, 3, 48
    xb = synthetic.to_bf16_bits(rng.standard_normal((m, k)).astype(np.float32))
    w = synthetic.weight_normal(3, n, k, 0.05)
    qx, sx = oracle.quantize_act(xb, oracle.ACT_BF16)
    qw, sw = oracle.quantize(w)
    bias = rng.standard_normal(n).astype(np.float32)
    _, acc = oracle.linear_w8a8(qx, sx, oracle.ACT_BF16, qw, sw, bias, want_acc=True)
    t = oracle.e4m3_decode_table()
    for i in range(m):
        for r in range(n):
            s = sum(Fraction(float(t[qx[i, c]])) * Fraction(float(t[qw[r, c]])) for c in range(k))
            exact = Fraction(float(sx[i])) * Fraction(float(sw[r])) * s + Fraction(float(bias[r]))
            assert abs(acc[i, r] - float(exact)) <= 1e-12 * abs(float(exact))


def test_representable_activations_reduce_to_the_weight_only_layer():
    """Activations that are e4m3 values times a power of two, with the row
    amax 448 * 2^j: sx = 2^j and the activation codes are exact, so W8A8 and
    the weight-only layer agree bit for bit."""
    rng = np.random.default_rng(4)
    t = oracle.e4m3_decode_table()
    mid = np.nonzero(np.isfinite(t) & (np.abs(t) >= 0.25) & (np.abs(t) <= 64))[0]
    m, n, k = 4, 7, 64
    j = rng.integers(-6, 3, size=m)
    x = t[rng.choice(mid, size=(m, k))] * (2.0 ** j)[:, None]
    x[np.arange(m), 0] = 448.0 * 2.0 ** j
    xb = synthetic.to_bf16_bits(x.astype(np.float32))
    assert np.array_equal(oracle.act_values(xb, oracle.ACT_BF16), x)
    qx, sx = oracle.quantize_act(xb, oracle.ACT_BF16)
    assert np.array_equal(sx, (2.0 ** j).astype(np.float32))
    w = synthetic.weight_normal(5, n, k, 0.02)
    qw, sw = oracle.quantize(w)
    bias = rng.standard_normal(n).astype(np.float32)
    y8, a8 = oracle.linear_w8a8(qx, sx, oracle.ACT_BF16, qw, sw, bias, want_acc=True)
    yw, aw = oracle.linear(xb, oracle.ACT_BF16, qw, sw, bias, want_acc=True)
    assert np.array_equal(y8, yw) and np.allclose(a8, aw, rtol=1e-15, atol=0)


@pytest.mark.parametrize("kind", ["normal", "outlier"])
def test_w8a8_within_two_half_steps_of_the_unquantised_product(kind):
    """Both operands come back within half an e4m3 step (2^-4 relative, or
    2^-10 * scale below the normal range): |x'w' - xw| <= |x||w'-w| + |w||x'-x|
    + |x'-x||w'-w| for each product, summed; and the aggregate error sits at
    the statistical level of two independent roundings (about sqrt(2) * 0.0255)."""
    rng = np.random.default_rng(6)
    m, n, k = 3, 40, 512
    w = synthetic.weight_normal(7, n, k, 0.02) if kind == "normal" else synthetic.weight_outlier(8, n, k)
    xb = synthetic.to_bf16_bits(rng.standard_normal((m, k)).astype(np.float32))
    qx, sx = oracle.quantize_act(xb, oracle.ACT_BF16)
    qw, sw = oracle.quantize(w)
    _, acc = oracle.linear_w8a8(qx, sx, oracle.ACT_BF16, qw, sw, want_acc=True)
    x = oracle.act_values(xb, oracle.ACT_BF16)
    w64 = w.astype(np.float64)
    y_true = x @ w64.T
    ex = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * sx[:, None].astype(np.float64)) * (1 + 2.0 ** -20)
    ew = np.maximum(np.abs(w64) * 2.0 ** -4, 2.0 ** -10 * sw[:, None].astype(np.float64)) * (1 + 2.0 ** -20)
    bound = np.abs(x) @ ew.T + ex @ np.abs(w64).T + ex @ ew.T
    assert np.all(np.abs(acc - y_true) <= bound * (1 + 1e-9))
    rel = np.linalg.norm(acc - y_true) / np.linalg.norm(y_true)
    assert 0.02 <= rel <= 0.06, rel
