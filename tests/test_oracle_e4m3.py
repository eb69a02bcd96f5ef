"""Pins of the oracle's e4m3 codec against what the pages and mathematics fix.

Decode: the format table and footnotes of page "B04 Precision &
Quantization" (section 2), the worked byte 0x38 of page "cuTile-rs tutorial
11", the closed form value = (-1)^s (1 + m/8) 2^(e-7) (e>0), m 2^-9 (e=0),
and torch's independent float8_e4m3fn decoder.

Encode: round to nearest even, saturating to +-448 (page "kadirnar/
kernel-agent fp8-weights", "The contract"; page "tensormux Write an FP8
kernel", step 4).  Pinned by brute force against the 254-entry decoded table
(nearest value, ties to the even code, saturation), by the pages' tie
examples, and by torch's independent encoder where torch saturates the same
way (|v| <= 464).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests.e4m3_brute import brute_encode, table


def _golden(golden_dir):
    out = {}
    with open(os.path.join(golden_dir, "e4m3_format.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split()[:2]
            out[key] = val
    return out


def test_format_limits_match_page_table(golden_dir):
    g = _golden(golden_dir)
    t = oracle.e4m3_decode_table()
    fin = t[np.isfinite(t)]
    pos = fin[fin > 0]
    assert float(g["max_finite"]) == fin.max() == t[0x7E]
    assert float(g["max_finite"]) == 1.75 * 2 ** 8
    # the page prints 5 significant digits; the exact values are 2^-6, 2^-9
    assert t[0x08] == 2.0 ** -6 and abs(t[0x08] - float(g["min_normal"])) < 1e-12
    assert pos.min() == t[0x01] == 2.0 ** -9
    assert abs(pos.min() - float(g["min_subnormal"])) < 1e-7
    assert t[0x39] - t[0x38] == float(g["ulp_of_one"])
    assert float(g["byte_0x38"]) == t[0x38] == 1.0
    assert t[0x80] == 0.0 and math.copysign(1.0, t[0x80]) == -1.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.isnan(t).sum() == 2
    # derived limits from (E, M, bias): emin = 1 - b; the top exponent keeps
    # seven normal mantissas, so emax = 2^E - 1 - b = 8
    E, M, b = int(g["exponent_bits"]), int(g["mantissa_bits"]), int(g["bias"])
    assert t[0x08] == 2.0 ** (1 - b)
    assert pos.min() == 2.0 ** (1 - b - M)
    # one mantissa pattern (S.1111.111) is NaN, so the top binade keeps 2^M - 1
    # normals and the largest is (1 + (2^M - 2)/2^M) * 2^(2^E - 1 - b) = 448
    assert fin.max() == (1 + (2 ** M - 2) / 2 ** M) * 2 ** (2 ** E - 1 - b)
    # number of binades of normals: emax - emin + 1 = 8 - (-6) + 1 = 15
    normals = pos[pos >= 2.0 ** -6]
    assert len(set(math.frexp(v)[1] for v in normals)) == int(g["binades"])


def test_decode_closed_form_every_code():
    t = oracle.e4m3_decode_table()
    for b in range(256):
        s, e, m = b >> 7, (b >> 3) & 15, b & 7
        if e == 15 and m == 7:
            assert np.isnan(t[b])
            continue
        mag = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        assert Fraction(t[b]) == (-mag if s else mag), hex(b)


def test_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    t = oracle.e4m3_decode_table()
    both_nan = np.isnan(ref) & np.isnan(t)
    assert np.array_equal(np.isnan(ref), np.isnan(t))
    assert np.array_equal(ref[~both_nan], t[~both_nan])
    assert np.array_equal(np.signbit(ref[~both_nan]), np.signbit(t[~both_nan]))


def test_decode_monotone_and_sign_symmetric():
    t = oracle.e4m3_decode_table()
    pos = t[0x00:0x7F]
    assert np.all(np.diff(pos) > 0)
    for b in range(0x7F):
        assert t[b | 0x80] == -t[b]


def test_every_code_exact_in_bf16_and_f16():
    # page "kadirnar/kernel-agent fp8-weights": the e4m3 -> f16 conversion is
    # exact and every e4m3 value is a bf16 value
    t = oracle.e4m3_decode_table()
    fin = torch.from_numpy(t[np.isfinite(t)])
    assert torch.equal(fin.to(torch.bfloat16).to(torch.float64), fin)
    assert torch.equal(fin.to(torch.float16).to(torch.float64), fin)


# ----------------------------------------------------------------- encode --

def _table():
    return table()


def _brute_encode(a32):
    return brute_encode(a32)


def test_encode_roundtrip_every_finite_code():
    t = oracle.e4m3_decode_table()
    for b in range(256):
        if np.isnan(t[b]):
            continue
        assert oracle.e4m3_encode(np.float32(t[b]))[0] == b, hex(b)


@pytest.mark.parametrize("v,code", [
    (1.0625, 0x38),        # midpoint 1.0 | 1.125 -> even 1.0
    (1.1875, 0x3A),        # midpoint 1.125 | 1.25 -> even 1.25
    (432.0, 0x7E),         # midpoint 416 | 448 -> even 448
    (3 * 2.0 ** -10, 0x02),  # midpoint 2^-9 | 2^-8 -> even 2^-8
    (2.0 ** -10, 0x00),    # midpoint 0 | 2^-9 -> 0
    (-(2.0 ** -10), 0x80),
    (1.0625 + 2 ** -20, 0x39),
    (1.0625 - 2 ** -20, 0x38),
    (449.0, 0x7E), (463.99, 0x7E), (464.0, 0x7E), (465.0, 0x7E), (1e30, 0x7E),
    (float(np.finfo(np.float32).max), 0x7E), (float("inf"), 0x7E),
    (-449.0, 0xFE), (-1e30, 0xFE), (float("-inf"), 0xFE),
    (0.0, 0x00), (-0.0, 0x80), (-1e-30, 0x80), (1e-45, 0x00),
])
def test_encode_ties_clamp_and_zeros(v, code):
    assert oracle.e4m3_encode(np.float32(v))[0] == code


def test_encode_nan_keeps_sign():
    assert oracle.e4m3_encode(np.float32("nan"))[0] & 0x7F == 0x7F


def _sweep_values():
    rng = np.random.default_rng(20261202)
    vals = _table()
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)   # 5-bit values, exact
    pts = np.concatenate([mids, vals.astype(np.float32), np.float32([448, 464, 480])])
    bits = pts.view(np.uint32).astype(np.int64)
    offs = np.arange(-64, 65, dtype=np.int64)
    near = (bits[:, None] + offs[None, :]).ravel()
    near = near[(near >= 0) & (near < 0x7F800000)].astype(np.uint32).view(np.float32)
    rnd = rng.integers(0, 0x7F800000, size=400_000, dtype=np.uint32).view(np.float32)
    dense = np.linspace(0, 500, 200_001, dtype=np.float32)
    small = (rng.random(100_000) * 2.0 ** -5).astype(np.float32)
    v = np.concatenate([near, rnd, dense, small])
    return np.concatenate([v, -v])


def test_encode_is_nearest_even_saturating_brute_force():
    v = _sweep_values()
    got = oracle.e4m3_encode(v)
    want = _brute_encode(v)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (v[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_encode_matches_torch_where_torch_saturates_alike():
    v = _sweep_values()
    v = v[np.abs(v) <= 464.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(v)
    assert np.array_equal(got, ref)


def test_brute_force_reference_catches_planted_mistakes():
    """The brute-force pin must be able to fail: plant a truncating and a
    ties-away rounding and check that the pin sees both."""
    v = _sweep_values()
    want = _brute_encode(v)
    a = np.abs(v.astype(np.float64))
    vals = _table()
    trunc = np.minimum(np.searchsorted(vals, a, side="right") - 1, 0x7E).astype(np.uint8)
    trunc |= np.where(np.signbit(v), 0x80, 0).astype(np.uint8)
    assert np.any(trunc != want)
    # ties away from zero at one tie point
    assert _brute_encode(np.float32([1.0625]))[0] == 0x38
