"""The oracle's quantise -> decode -> linear chain against the unquantised
product.  Each weight is reproduced to within half an e4m3 step: 2^-4 of its
magnitude for codes in the normal range, 2^-10 * scale below it (the e4m3
format's 3 mantissa bits and its smallest subnormal 2^-9, page "B04 Precision
& Quantization", section 2, the E4M3 row), plus the fp32 rounding of w /
scale.  So the unrounded layer output obeys

    |y_q - y_true| <= sum_k |x_k| * (2^-4 * |w_k| * (1 + 2^-20) + 2^-10 * scale_n)

for every output.  That worst case adds every weight's error with the same
sign.  The errors are independent and centred, so the output's relative
error is far smaller: for RNE to 3 mantissa bits the relative weight error is
uniform within +-2^-4 / m (m the mantissa in [1, 2)), whose rms is
2^-4 * E[1/m^2]^(1/2) / sqrt(3), about 0.0255, and the layer's rel_l2 error
against the unquantised product lands near it.  A doubled scale would give
1.0 and a permuted channel about 1.4.  y_true = x . W^T + b in fp64 on the
fp32 inputs."""
import numpy as np
import pytest

import oracle
import synthetic


def _bound_case(w, x_bits, act, bias):
    codes, scales = oracle.quantize(w)
    _, acc = oracle.linear(x_bits, act, codes, scales, bias, want_acc=True)
    x = oracle.act_values(x_bits, act)
    w64 = w.astype(np.float64)
    y_true = x @ w64.T + (0.0 if bias is None else bias.astype(np.float64))
    ax = np.abs(x)
    bound = ax @ (2.0 ** -4 * np.abs(w64) * (1 + 2.0 ** -20)).T + (ax.sum(axis=1)[:, None] * 2.0 ** -10) * scales[None, :]
    return acc, y_true, bound


@pytest.mark.parametrize("kind", ["normal", "outlier", "tiny"])
def test_quantised_layer_within_half_an_e4m3_step_of_the_unquantised_product(kind):
    rng = np.random.default_rng({"normal": 1, "outlier": 2, "tiny": 3}[kind])
    n, k, m = 40, 512, 3
    if kind == "normal":
        w = synthetic.weight_normal(11, n, k, 0.02)
    elif kind == "outlier":
        w = synthetic.weight_outlier(12, n, k)
    else:
        # rows whose codes are mostly subnormal: the 2^-10 * scale term matters
        w = (rng.standard_normal((n, k)) * 1e-3).astype(np.float32)
        w[:, 0] = 1.0
    x = synthetic.to_bf16_bits(rng.standard_normal((m, k)).astype(np.float32))
    bias = rng.standard_normal(n).astype(np.float32)
    acc, y_true, bound = _bound_case(w, x, oracle.ACT_BF16, bias)
    slack = 1e-12 * (np.abs(oracle.act_values(x, oracle.ACT_BF16)) @ np.abs(w.astype(np.float64)).T) + 1e-300
    assert np.all(np.abs(acc - y_true) <= bound + slack)
    # and the bound is not vacuous: the error reaches a fair part of it
    assert np.max(np.abs(acc - y_true) / bound) > 0.05
    if kind != "tiny":   # tiny: the exact large column dominates y
        rel = np.linalg.norm(acc - y_true) / np.linalg.norm(y_true)
        assert 0.01 <= rel <= 0.05, rel


def test_the_bound_catches_a_dropped_scale():
    """A planted mistake on the CPU: codes decoded without their scale."""
    rng = np.random.default_rng(5)
    w = synthetic.weight_normal(13, 8, 256, 0.02)
    x = synthetic.to_bf16_bits(rng.standard_normal((2, 256)).astype(np.float32))
    codes, scales = oracle.quantize(w)
    _, acc = oracle.linear(x, oracle.ACT_BF16, codes, np.ones_like(scales), None, want_acc=True)
    xv = oracle.act_values(x, oracle.ACT_BF16)
    y_true = xv @ w.astype(np.float64).T
    bound = np.abs(xv) @ (2.0 ** -4 * np.abs(w.astype(np.float64))).T + np.abs(xv).sum(1)[:, None] * 2.0 ** -10 * scales
    assert np.any(np.abs(acc - y_true) > bound)


def test_exactly_representable_weights_have_no_quantisation_error():
    """w = e4m3 value * 2^j with the row amax 448 * 2^j: scale = 2^j and the
    decoded weight is w itself, so y_q == y_true exactly."""
    rng = np.random.default_rng(6)
    t = oracle.e4m3_decode_table()
    finite = np.array([c for c in range(0x7F) if c != 0x7F])
    n, k = 6, 128
    codes = rng.choice(finite, size=(n, k))
    codes[:, 0] = 0x7E
    j = rng.integers(-12, 3, size=n)
    w = (t[codes] * (2.0 ** j)[:, None]).astype(np.float32)
    x = synthetic.to_bf16_bits(rng.integers(-4, 5, size=(2, k)).astype(np.float32))
    acc, y_true, _ = _bound_case(w, x, oracle.ACT_BF16, None)
    assert np.array_equal(acc, y_true)
