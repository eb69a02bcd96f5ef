"""Brute-force e4m3 encoder used as a pin (not part of the oracle).

Nearest of the 127 non-negative finite e4m3 values, ties to the even code,
every |v| >= 448 to 0x7E, the sign bit copied.  The differences to the two
neighbours are exact in fp64: each neighbour is either 0 or within a factor
of two of the input.
"""
import numpy as np

import oracle


def table():
    return oracle.e4m3_decode_table()[0x00:0x7F]


def brute_encode(a32: np.ndarray) -> np.ndarray:
    vals = table()
    a32 = np.asarray(a32, dtype=np.float32)
    a = np.abs(a32.astype(np.float64))
    sign = np.where(np.signbit(a32), 0x80, 0).astype(np.uint8)
    hi = np.minimum(np.searchsorted(vals, a, side="left"), len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    exact = vals[hi] == a
    d_lo = a - vals[lo]
    d_hi = vals[hi] - a
    code = np.where(d_lo < d_hi, lo, hi)
    tie = (d_lo == d_hi) & ~exact
    code = np.where(tie, np.where(lo % 2 == 0, lo, hi), code)
    code = np.where(exact, hi, code)
    code = np.where(a >= 448.0, 0x7E, code)
    return code.astype(np.uint8) | sign
