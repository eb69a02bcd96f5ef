"""Pins of the oracle's quantiser and linear layer.

Quantiser (page "kadirnar/kernel-agent fp8-weights", "The contract";
zero-row rule from page "day98 quant_matmul.cu", quantizeSymmetric):
scale = fp32(amax / 448), 1.0 when that is 0, codes = nearest-even e4m3 of
the fp32 quotient w / scale.  Checked against numpy's fp32 division and a
brute-force nearest-code search, and the invariant that every nonzero row
holds a +-448 code.

Linear layer (same page: y = scale[n] * sum_k x q + bias, one rounding):
checked against exact rational arithmetic on tiny shapes (non-square, so a
transposed operand or a swapped index fails), against an fp64 product built
from torch's own e4m3 and bf16 decoders, and on closed-form cases (x = 0,
one-hot x, all-ones, power-of-two scales with integer activations).
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synthetic
from tests.e4m3_brute import brute_encode


# -------------------------------------------------------------- quantiser --

def test_scale_is_fp32_amax_over_448():
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((64, 300)) * 10.0 ** rng.uniform(-6, 3, size=(64, 1))).astype(np.float32)
    codes, scales = oracle.quantize(w)
    amax = np.abs(w).max(axis=1).astype(np.float32)
    assert np.array_equal(scales, (amax / np.float32(448.0)).astype(np.float32))


def test_zero_and_underflowing_rows_take_scale_one():
    w = np.zeros((3, 32), dtype=np.float32)
    w[1, 5] = np.float32(1e-45)        # amax/448 rounds to 0 in fp32
    w[2, 7] = np.float32(-1e-45)
    codes, scales = oracle.quantize(w)
    assert np.array_equal(scales, np.float32([1, 1, 1]))
    assert np.all((codes & 0x7F) == 0)
    assert codes[2, 7] == 0x80          # -tiny -> -0


def test_codes_are_nearest_even_of_fp32_quotient():
    for seed, std in [(12, 0.02), (13, 1e-3), (14, 50.0)]:
        rng = np.random.default_rng(seed)
        w = (rng.standard_t(3, size=(48, 257)) * std).astype(np.float32)
        codes, scales = oracle.quantize(w)
        q = (w / scales[:, None]).astype(np.float32)   # numpy fp32 IEEE division
        assert np.array_equal(codes, brute_encode(q.ravel()).reshape(q.shape))


def test_every_nonzero_row_holds_a_max_code():
    c = synthetic.case("outlier_gemv")
    codes, scales = oracle.quantize(c["w"])
    assert np.all(np.any((codes & 0x7F) == 0x7E, axis=1))


def test_subnormal_codes_occur_and_are_kept():
    # heavy tails push small weights into e4m3 subnormals (codes 0x01..0x07)
    c = synthetic.case("outlier_gemv")
    codes, _ = oracle.quantize(c["w"][:256])
    mag = codes & 0x7F
    assert np.any((mag >= 1) & (mag <= 7))


# ---------------------------------------------------------- linear layer --

def _dec_frac(code):
    return Fraction(oracle.e4m3_decode(code))


def _nearest_even(exact: Fraction, to_frac, lo_bits, hi_bits):
    """Bits b in [lo,hi] of the value nearest to exact, ties to even bits."""
    best = None
    for b in range(lo_bits, hi_bits + 1):
        d = abs(to_frac(b) - exact)
        if best is None or d < best[0] or (d == best[0] and b % 2 == 0):
            best = (d, b)
    return best[1]


def _rounded_exact(exact: Fraction, act):
    """Exact rounding of a rational to bf16/fp16 bits (search near fp64 guess)."""
    guess = oracle.round_bf16(float(exact))[0] if act == oracle.ACT_BF16 else oracle.round_f16(float(exact))[0]
    to = (lambda b: Fraction(oracle.act_values(np.array([b], np.uint16), act)[0]))
    g = int(guess)
    cands = [b for b in (g - 2, g - 1, g, g + 1, g + 2) if 0 <= b < 65536 and (b & 0x8000) == (g & 0x8000)]
    cands = [b for b in cands if np.isfinite(oracle.act_values(np.array([b], np.uint16), act)[0])]
    best = None
    for b in cands:
        d = abs(to(b) - exact)
        if best is None or d < best[0] or (d == best[0] and b % 2 == 0):
            best = (d, b)
    return best[1]


@pytest.mark.parametrize("act", [oracle.ACT_BF16, oracle.ACT_F16])
def test_linear_equals_exact_rational_on_tiny_shapes(act):
    rng = np.random.default_rng(21 + act)
    for (m, n, k) in [(1, 1, 1), (1, 3, 5), (2, 5, 3), (3, 2, 7), (4, 3, 9), (2, 7, 16)]:
        c = synthetic.random_case(int(rng.integers(1 << 30)), m, n, k, act=act)
        codes, scales = oracle.quantize(c["w"])
        y = oracle.linear(c["x"], act, codes, scales, c["bias"])
        xv = oracle.act_values(c["x"], act)
        for i, j in itertools.product(range(m), range(n)):
            s = sum(Fraction(xv[i, t]) * _dec_frac(codes[j, t]) for t in range(k))
            exact = Fraction(float(scales[j])) * s + Fraction(float(c["bias"][j]))
            assert y[i, j] == _rounded_exact(exact, act), (m, n, k, i, j)


def test_linear_matches_torch_decoded_fp64_product():
    c = synthetic.random_case(31, 5, 70, 96)
    codes, scales = oracle.quantize(c["w"])
    y, acc = oracle.linear(c["x"], oracle.ACT_BF16, codes, scales, c["bias"], want_acc=True)
    wq = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64) * \
        torch.from_numpy(scales).to(torch.float64)[:, None]
    xv = torch.from_numpy(c["x"].view(np.int16)).view(torch.bfloat16).to(torch.float64)
    ref = xv @ wq.T + torch.from_numpy(c["bias"]).to(torch.float64)
    assert np.allclose(acc, ref.numpy(), rtol=1e-12, atol=1e-15)


def test_linear_closed_forms():
    rng = np.random.default_rng(41)
    n, k = 6, 32
    w = rng.standard_normal((n, k)).astype(np.float32) * np.float32(0.3)
    bias = rng.standard_normal(n).astype(np.float32)
    codes, scales = oracle.quantize(w)
    bias_bits = oracle.round_bf16(bias.astype(np.float64))
    # x = 0 -> y = RN(bias)
    x0 = np.zeros((2, k), dtype=np.uint16)
    assert np.array_equal(oracle.linear(x0, oracle.ACT_BF16, codes, scales, bias),
                          np.tile(bias_bits, (2, 1)))
    # one-hot x -> y = RN(scale * deq(q[n, j]) + bias)
    for j in (0, 7, 31):
        x = np.zeros((1, k), dtype=np.uint16)
        x[0, j] = 0x3F80                     # bf16 1.0
        want = [oracle.round_bf16(float(scales[r]) * oracle.e4m3_decode(codes[r, j]) + float(bias[r]))[0]
                for r in range(n)]
        assert np.array_equal(oracle.linear(x, oracle.ACT_BF16, codes, scales, bias)[0], want)
    # all-ones x -> y = RN(scale * sum_k deq + bias)
    x1 = np.full((1, k), 0x3F80, dtype=np.uint16)
    want = [oracle.round_bf16(float(scales[r]) * sum(oracle.e4m3_decode(c) for c in codes[r]) + float(bias[r]))[0]
            for r in range(n)]
    assert np.array_equal(oracle.linear(x1, oracle.ACT_BF16, codes, scales, bias)[0], want)


def test_linear_power_of_two_scales_integer_acts_exact():
    # rows with amax = 448 * 2^j have scale 2^j, and e4m3 values times 2^j
    # quantise exactly; with small-integer x the whole result is exact
    rng = np.random.default_rng(51)
    n, k, m = 8, 64, 3
    t = oracle.e4m3_decode_table()[:0x7F]
    w = np.empty((n, k), dtype=np.float32)
    for r in range(n):
        w[r] = rng.choice(t, size=k) * rng.choice([-1, 1], size=k) * 2.0 ** (r - 4)
        w[r, r] = 448.0 * 2.0 ** (r - 4)
    codes, scales = oracle.quantize(w)
    assert np.array_equal(scales, np.float32([2.0 ** (r - 4) for r in range(n)]))
    xi = rng.integers(-4, 5, size=(m, k))
    x = synthetic.to_bf16_bits(xi.astype(np.float32))
    y, acc = oracle.linear(x, oracle.ACT_BF16, codes, scales, None, want_acc=True)
    exact = [[sum(Fraction(int(xi[i, q])) * Fraction(float(w[r, q])) for q in range(k)) for r in range(n)]
             for i in range(m)]
    assert all(Fraction(acc[i, r]) == exact[i][r] for i in range(m) for r in range(n))


def test_bias_none_equals_bias_zero_and_threads_do_not_matter():
    c = synthetic.random_case(61, 3, 50, 48)
    codes, scales = oracle.quantize(c["w"])
    a = oracle.linear(c["x"], oracle.ACT_BF16, codes, scales, None)
    b = oracle.linear(c["x"], oracle.ACT_BF16, codes, scales, np.zeros(50, np.float32))
    d = oracle.linear(c["x"], oracle.ACT_BF16, codes, scales, None, threads=4)
    assert np.array_equal(a, b) and np.array_equal(a, d)
