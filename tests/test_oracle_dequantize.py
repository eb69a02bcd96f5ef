"""Pins of the oracle's dequantised weight, scale[n] * e4m3(q[n, k]) in fp64
(page "kadirnar/kernel-agent fp8-weights", section "The contract": the
fallback form), against what the format and the quantiser fix."""
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
