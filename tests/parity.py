"""Parity measures between the CUDA path and the oracle (tests only).

Gates (the layer's stated tolerance): rel_l2 = ||y - y_ref||_2 / ||y_ref||_2
over all outputs <= 2e-3, cosine of every output row (one token over its N
channels) >= 0.9999, no non-finite output.  y_ref is the oracle's fp64 result
rounded once to the output dtype.  Codes and scales are compared bit for bit
elsewhere.
"""
import numpy as np

import oracle

REL_L2_MAX = 2e-3
COSINE_MIN = 0.9999


def values(bits, act):
    bits = np.asarray(bits, dtype=np.uint16)
    if act == oracle.ACT_F16:
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def compare(y_bits, ref_bits, act):
    y = values(y_bits, act)
    r = values(ref_bits, act)
    out = {"finite": bool(np.all(np.isfinite(y)))}
    d = np.linalg.norm((y - r).ravel())
    nr = np.linalg.norm(r.ravel())
    out["rel_l2"] = float(d / nr) if nr > 0 else float(d)
    yy = y.reshape(-1, y.shape[-1])
    rr = r.reshape(-1, r.shape[-1])
    num = np.sum(yy * rr, axis=1)
    den = np.linalg.norm(yy, axis=1) * np.linalg.norm(rr, axis=1)
    cos = np.where(den > 0, num / np.where(den > 0, den, 1), np.where(
        np.all(yy == rr, axis=1), 1.0, 0.0))
    out["min_cosine"] = float(cos.min())
    out["bit_equal"] = float(np.mean(np.asarray(y_bits) == np.asarray(ref_bits)))
    return out


def assert_parity(y_bits, ref_bits, act, what=""):
    c = compare(y_bits, ref_bits, act)
    assert c["finite"], (what, c)
    assert c["rel_l2"] <= REL_L2_MAX, (what, c)
    assert c["min_cosine"] >= COSINE_MIN, (what, c)
    return c
