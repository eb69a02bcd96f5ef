"""Pins of the oracle's output rounding (fp64 -> bf16 / fp16, one RNE step).

bf16: page "B04 Precision & Quantization", section 2 ("The key insight"),
prints the fp32 -> bf16 round-to-nearest-even as an integer formula on the
fp32 bits; for fp32-representable inputs the oracle must agree with it, and
with torch's independent conversion.  For fp64 inputs that fp32 cannot hold
the oracle must return the nearest bf16 value, ties to the even pattern,
checked with exact rational arithmetic (no fp32 detour, no double rounding).

fp16: numpy's float64 -> float16 conversion rounds once, directly from the
double (checked below on a case where a detour through fp32 would differ);
the oracle must agree with it everywhere, including subnormals and overflow.
"""
from fractions import Fraction

import numpy as np
import torch

import oracle


def _page_bf16_formula(f32: np.ndarray) -> np.ndarray:
    u = f32.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def _finite_f32(n, seed):
    rng = np.random.default_rng(seed)
    b = rng.integers(0, 0x7F800000, size=n, dtype=np.uint32)
    b |= rng.integers(0, 2, size=n, dtype=np.uint32) << 31
    return b.view(np.float32)


def test_bf16_equals_page_formula_on_fp32_inputs():
    f = _finite_f32(500_000, 1)
    # add every tie pattern of a few binades and values near the top of range
    ties = (np.arange(0x3F800000, 0x3F900000, 0x8000, dtype=np.uint32)).view(np.float32)
    top = np.arange(0x7F7F0000, 0x7F800000, 97, dtype=np.uint32).view(np.float32)
    f = np.concatenate([f, ties, -ties, top, -top, np.float32([0.0, -0.0])])
    got = oracle.round_bf16(f.astype(np.float64))
    assert np.array_equal(got, _page_bf16_formula(f))


def test_bf16_equals_torch_on_fp32_inputs():
    f = _finite_f32(500_000, 2)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.round_bf16(f.astype(np.float64)), ref)


def _bf16_frac(bits):
    v = oracle.act_values(np.array([bits], dtype=np.uint16), oracle.ACT_BF16)[0]
    return Fraction(v)


def _f16_frac(bits):
    v = oracle.act_values(np.array([bits], dtype=np.uint16), oracle.ACT_F16)[0]
    return Fraction(v)


def _check_nearest_even(values, rounder, to_frac, max_bits):
    got = rounder(values)
    for v, b in zip(values, got):
        b = int(b)
        mag = b & 0x7FFF
        if mag >= max_bits:                      # inf: checked elsewhere
            continue
        exact = Fraction(float(v))
        mine = to_frac(b)
        for nb in (b - 1, b + 1):
            if (nb & 0x7FFF) > max_bits or (nb & 0x8000) != (b & 0x8000) or nb < 0:
                continue
            other = to_frac(nb)
            d0, d1 = abs(exact - mine), abs(exact - other)
            assert d0 <= d1, (v, hex(b), hex(nb))
            if d0 == d1:
                assert b % 2 == 0, (v, hex(b))


def test_bf16_nearest_even_from_fp64_exact():
    rng = np.random.default_rng(3)
    base = _finite_f32(3000, 4).astype(np.float64)
    base = base[np.abs(base) < 1e38]
    # perturb below fp32 resolution so the fp64 bits matter
    v = base * (1 + rng.uniform(-2 ** -20, 2 ** -20, size=base.size))
    # exact bf16 midpoints nudged by 2^-40 relative: a detour via fp32 would tie
    mids = np.float64(1.0) + 2.0 ** -8 + np.arange(0, 64) * 2.0 ** -6
    v = np.concatenate([v, mids * (1 + 2.0 ** -40), mids * (1 - 2.0 ** -40), mids])
    _check_nearest_even(v, oracle.round_bf16, _bf16_frac, 0x7F80)


def test_bf16_no_double_rounding():
    # 1 + 2^-8 is the midpoint of bf16 1.0 | 1.0078125; nudged up by 2^-40 it
    # must round up, although its fp32 image is the midpoint itself (-> 1.0)
    v = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert np.float32(v) == np.float32(1.0 + 2.0 ** -8)
    assert oracle.round_bf16(v)[0] == 0x3F81
    assert oracle.round_bf16(1.0 + 2.0 ** -8)[0] == 0x3F80


def test_bf16_overflow_and_specials():
    mx = (2 - 2.0 ** -7) * 2.0 ** 127
    half_ulp = 2.0 ** (127 - 8)
    assert oracle.round_bf16(mx)[0] == 0x7F7F
    assert oracle.round_bf16(mx + half_ulp * 0.999)[0] == 0x7F7F
    assert oracle.round_bf16(mx + half_ulp)[0] == 0x7F80      # tie -> even -> inf
    assert oracle.round_bf16(-1e300)[0] == 0xFF80
    assert oracle.round_bf16(-0.0)[0] == 0x8000
    assert oracle.round_bf16(2.0 ** -133)[0] == 0x0001        # smallest subnormal
    assert oracle.round_bf16(2.0 ** -134)[0] == 0x0000        # tie -> even 0


def test_numpy_f16_rounds_directly_from_double():
    # 1 + 2^-9 + 2^-11 is the midpoint 0x3C02 | 0x3C03 (tie -> 0x3C02); nudged
    # up by 2^-40 a direct rounding gives 0x3C03, a detour via fp32 0x3C02
    m = 1 + 2.0 ** -9 + 2.0 ** -11
    assert np.float64(m).astype(np.float16).view(np.uint16) == 0x3C02
    assert np.float64(m + 2.0 ** -40).astype(np.float16).view(np.uint16) == 0x3C03


def test_f16_equals_numpy():
    rng = np.random.default_rng(5)
    v = np.concatenate([
        rng.standard_normal(200_000) * 10.0 ** rng.uniform(-9, 5, size=200_000),
        np.linspace(-70000, 70000, 100_001),
        np.float64([65504, 65519.99, 65520, 65536, 2.0 ** -24, 2.0 ** -25,
                    1.5 * 2.0 ** -25, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, -0.0, 0.0]),
    ])
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.round_f16(v), ref)


def test_f16_nearest_even_from_fp64_exact():
    rng = np.random.default_rng(6)
    v = rng.standard_normal(3000) * 10.0 ** rng.uniform(-8, 4.5, size=3000)
    _check_nearest_even(v, oracle.round_f16, _f16_frac, 0x7C00)


def test_activation_decoders():
    # bf16 is the top half of fp32; fp16 decoded by formula vs numpy
    b = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    f16 = b.view(np.float16).astype(np.float64)
    mine = oracle.act_values(b, oracle.ACT_F16)
    fin = np.isfinite(f16)
    assert np.array_equal(mine[fin], f16[fin])
    assert np.array_equal(np.isnan(mine), np.isnan(f16))
    bf = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    mine = oracle.act_values(b, oracle.ACT_BF16)
    fin = np.isfinite(bf)
    assert np.array_equal(mine[fin], bf[fin])


def test_widening_16_bit_weights_is_exact_for_every_pattern():
    """Every fp16 and bf16 pattern widens to the fp32 value numpy's float16
    conversion and the bf16 closed form (the pattern as the top half of an
    fp32) give; NaNs stay NaN."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f16 = oracle.widen_16(bits, oracle.ACT_F16)
    ref16 = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref16)
    assert np.array_equal(np.isnan(f16), nan) and np.array_equal(f16[~nan].view(np.uint32), ref16[~nan].view(np.uint32))
    b16 = oracle.widen_16(bits, oracle.ACT_BF16)
    refb = (bits.astype(np.uint32) << 16).view(np.float32)
    nan = np.isnan(refb)
    assert np.array_equal(np.isnan(b16), nan) and np.array_equal(b16[~nan].view(np.uint32), refb[~nan].view(np.uint32))
