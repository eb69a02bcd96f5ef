"""Pins of the oracle's weight error report, fp8_error(weight, q, scale).

Page "kadirnar/kernel-agent fp8-weights", section "The contract", names the
report's fields (rel_l2, worst_channel_rel_l2, underflow, crest) without
defining them.  The readings, with Wq[n, k] = scale[n] * e4m3(q[n, k]):
  rel_l2               ||W - Wq||_F / ||W||_F over the whole matrix
  worst_channel_rel_l2 the largest ||W_n - Wq_n|| / ||W_n|| over nonzero rows
  underflow            share of the nonzero weights whose code is +-0
  crest                the largest amax_n / rms_n over nonzero rows, with
                       rms_n = sqrt(mean_k W[n, k]^2) over all k of the row

Each pin below follows from the mathematics of those readings, not from the
oracle's code: closed forms (a one-spike row has crest sqrt(k), a constant
row crest 1; weights below half the smallest e4m3 step times the scale all
underflow; the one tie of [448, 1.0625] leaves an error of exactly 0.0625),
and invariances (a power-of-two rescale of W changes no code and no field;
duplicated or permuted rows change no field).  Every planted wrong
definition at the end (the rms over nonzero entries only, the underflow
share over all entries, per-row averaging, a dropped square root, absolute
instead of relative errors, the sign of -0 ignored, a dropped scale) fails
at least one pin, so a plausible mistake in the oracle cannot pass them.
"""
import numpy as np
import pytest

import oracle

TOL = 1e-13


def _q(w):
    w = np.asarray(w, dtype=np.float32)
    codes, scales = oracle.quantize(w)
    return w, codes, scales


def oracle_report(w, codes, scales):
    return oracle.fp8_error(w, codes, scales)


# ------------------------------------------------------------------ pins --
# Each pin takes a report function (w, codes, scales) -> dict and returns a
# list of failure messages (empty when it holds).

def pin_spike_crest(report):
    """One spike in a row of k: amax = a, rms = a / sqrt(k), crest sqrt(k)."""
    bad = []
    for k, a in ((64, 3.0), (400, 0.02), (16, -7.5)):
        w = np.zeros((1, k))
        w[0, 5] = a
        r = report(*_q(w))
        if abs(r["crest"] - np.sqrt(k)) > TOL * np.sqrt(k):
            bad.append("spike crest k=%d: %r" % (k, r["crest"]))
    return bad


def pin_constant_crest(report):
    """A constant row (or one of constant magnitude) has crest 1."""
    w = np.full((1, 48), 0.37)
    w2 = np.tile([1.5, -1.5], (2, 20))
    bad = []
    for m in (w, w2):
        r = report(*_q(m))
        if abs(r["crest"] - 1.0) > TOL:
            bad.append("constant crest %r" % r["crest"])
    return bad


def pin_crest_is_max_over_nonzero_rows(report):
    """Rows of crest 4 (spike, k = 16), 1 (constant) and an all-zero row:
    crest 4, finite."""
    w = np.zeros((3, 16))
    w[0, 3] = 2.0
    w[1, :] = 0.5
    r = report(*_q(w))
    ok = np.isfinite(r["crest"]) and abs(r["crest"] - 4.0) <= TOL * 4
    return [] if ok else ["crest over rows %r" % r["crest"]]


def _underflow_matrix():
    # row 0: 448 (scale exactly 1), ten weights of 1.0 (exact codes), six
    # weights of magnitude 2^-12, below half the smallest subnormal step
    # 2^-9 of e4m3, three of them negative (codes 0x00 and 0x80), the rest
    # zeros.  Row 1: row 0 times 2^-20 (scale 2^-20, same codes).
    row = np.zeros(40)
    row[0] = 448.0
    row[1:11] = 1.0
    row[11:17] = 2.0 ** -12 * np.array([1, -1, 1, -1, 1, -1])
    return np.stack([row, row * 2.0 ** -20])


def pin_underflow_share(report):
    """Six of seventeen nonzero weights a row underflow: 6/17, whatever the
    zeros and whatever the sign."""
    w, codes, scales = _q(_underflow_matrix())
    r = report(w, codes, scales)
    return [] if abs(r["underflow"] - 6.0 / 17.0) <= TOL else ["underflow %r" % r["underflow"]]


def pin_underflow_error(report):
    """The only error of the underflow matrix is the six lost weights: per
    row ||e|| = 2^-12 sqrt(6), ||W|| = sqrt(448^2 + 10 + 6 * 2^-24) (times
    2^-20 in row 1), and both rows have the same relative error."""
    w, codes, scales = _q(_underflow_matrix())
    r = report(w, codes, scales)
    rel = 2.0 ** -12 * np.sqrt(6.0) / np.sqrt(448.0 ** 2 + 10 + 6 * 2.0 ** -24)
    bad = []
    if abs(r["rel_l2"] - rel) > 1e-12 * rel:
        bad.append("rel_l2 %r vs %r" % (r["rel_l2"], rel))
    if abs(r["worst_channel_rel_l2"] - rel) > 1e-12 * rel:
        bad.append("worst %r vs %r" % (r["worst_channel_rel_l2"], rel))
    return bad


def pin_tie_row(report):
    """[448, 1.0625]: scale 1, 1.0625 is the midpoint of 1 and 1.125 and
    rounds to the even code 1.0, error 0.0625; a second, exact row [448, 448]
    adds nothing to the error and its 448^2 * 2 to ||W||_F^2."""
    w, codes, scales = _q([[448.0, 1.0625], [448.0, 448.0]])
    r = report(w, codes, scales)
    n0 = np.sqrt(448.0 ** 2 + 1.0625 ** 2)
    rel = 0.0625 / np.sqrt(3 * 448.0 ** 2 + 1.0625 ** 2)
    bad = []
    if abs(r["rel_l2"] - rel) > 1e-12 * rel:
        bad.append("rel_l2 %r vs %r" % (r["rel_l2"], rel))
    if abs(r["worst_channel_rel_l2"] - 0.0625 / n0) > 1e-12 * 0.0625 / n0:
        bad.append("worst %r" % r["worst_channel_rel_l2"])
    if r["underflow"] != 0.0:
        bad.append("underflow %r" % r["underflow"])
    return bad


def _random_w(seed):
    rng = np.random.default_rng(seed)
    w = rng.standard_t(3, size=(24, 96)) * 0.02
    w[rng.random(w.shape) < 0.05] = 0.0
    w[3] *= 50.0
    w[7, 10] = 1e-9
    return w.astype(np.float32)


def pin_power_of_two_invariance(report):
    """W * 2^j (no over- or underflow of fp32) quantises to the same codes
    with scales * 2^j: every field is unchanged."""
    w0 = _random_w(901)
    r0 = report(*_q(w0))
    bad = []
    for j in (-7, 5, -40):
        r = report(*_q(w0 * np.float32(2.0 ** j)))
        for f in r0:
            if abs(r[f] - r0[f]) > 1e-12 * max(abs(r0[f]), 1e-300):
                bad.append("2^%d changes %s: %r -> %r" % (j, f, r0[f], r[f]))
    return bad


def pin_rows_duplicated_and_permuted(report):
    """Stacking W on itself, or permuting its rows, changes no field."""
    w0 = _random_w(902)
    r0 = report(*_q(w0))
    rng = np.random.default_rng(903)
    bad = []
    for w in (np.concatenate([w0, w0]), w0[rng.permutation(w0.shape[0])]):
        r = report(*_q(w))
        for f in r0:
            if abs(r[f] - r0[f]) > 1e-12 * max(abs(r0[f]), 1e-300):
                bad.append("%s %r -> %r" % (f, r0[f], r[f]))
    return bad


def pin_worst_bounds_total(report):
    """||W - Wq||_F^2 / ||W||_F^2 is a weighted mean of the rows' squared
    relative errors, so rel_l2 <= worst_channel_rel_l2, with equality when
    every row is the same."""
    w0 = _random_w(904)
    r = report(*_q(w0))
    same = report(*_q(np.tile(w0[5], (6, 1))))
    bad = []
    if not r["rel_l2"] <= r["worst_channel_rel_l2"] * (1 + 1e-12):
        bad.append("rel_l2 %r > worst %r" % (r["rel_l2"], r["worst_channel_rel_l2"]))
    if abs(same["rel_l2"] - same["worst_channel_rel_l2"]) > 1e-12 * same["rel_l2"]:
        bad.append("equal rows: %r vs %r" % (same["rel_l2"], same["worst_channel_rel_l2"]))
    return bad


def pin_representable_weights_have_no_error(report):
    """Weights that are e4m3 values times a power of two (with 448 in every
    row, so the scale is that power) quantise exactly: zero error."""
    t = oracle.e4m3_decode_table()[:0x7F]
    rng = np.random.default_rng(71)
    w = rng.choice(t, size=(16, 40)) * 0.125
    w[:, 0] = 448 * 0.125
    r = report(*_q(w))
    ok = r["rel_l2"] == 0.0 and r["worst_channel_rel_l2"] == 0.0 and r["underflow"] == 0.0
    return [] if ok else ["representable %r" % r]


PINS = [pin_spike_crest, pin_constant_crest, pin_crest_is_max_over_nonzero_rows, pin_underflow_share,
        pin_underflow_error, pin_tie_row, pin_power_of_two_invariance, pin_rows_duplicated_and_permuted,
        pin_worst_bounds_total, pin_representable_weights_have_no_error]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_report_holds_pin(pin):
    assert pin(oracle_report) == []


def test_all_zero_matrix_reports_zeros():
    r = oracle_report(*_q(np.zeros((3, 32))))
    assert r == {"rel_l2": 0.0, "worst_channel_rel_l2": 0.0, "underflow": 0.0, "crest": 0.0}


# ------------------------------------------------- planted wrong readings --
# The report re-done in numpy with one mistake each.  A correct numpy form
# is included to show that the pins accept a second, independent
# implementation, so each failure below is the planted mistake's.

def _dequant(codes, scales, with_scale=True):
    t = oracle.e4m3_decode_table()
    d = t[codes]
    return d * scales.astype(np.float64)[:, None] if with_scale else d


def make_report(rms_nonzero=False, crest_mean_abs=False, underflow_all=False, mean_of_rows=False,
                no_sqrt=False, worst_absolute=False, minus_zero_kept=False, no_scale=False):
    def report(w, codes, scales):
        w = np.asarray(w, dtype=np.float64)
        e = w - _dequant(codes, scales, with_scale=not no_scale)
        rn = np.sum(e * e, axis=1)
        rd = np.sum(w * w, axis=1)
        nz = rd > 0
        tot = rn.sum() / rd.sum() if rd.sum() > 0 else 0.0
        rel_rows = np.sqrt(rn[nz] / rd[nz])
        if mean_of_rows:
            rel = float(np.mean(rel_rows)) if nz.any() else 0.0
        else:
            rel = float(tot if no_sqrt else np.sqrt(tot))
        if worst_absolute:
            worst = float(np.sqrt(rn[nz]).max()) if nz.any() else 0.0
        else:
            worst = float(rel_rows.max()) if nz.any() else 0.0
        nonzero = w != 0
        zero_code = codes == 0 if minus_zero_kept else (codes & 0x7F) == 0
        den = w.size if underflow_all else nonzero.sum()
        under = float((nonzero & zero_code).sum() / den) if den else 0.0
        amax = np.abs(w).max(axis=1)
        if rms_nonzero:
            cnt = np.maximum(nonzero.sum(axis=1), 1)
            rms = np.sqrt(rd / cnt)
        elif crest_mean_abs:
            rms = np.abs(w).mean(axis=1)
        else:
            rms = np.sqrt(rd / w.shape[1])
        crest = float((amax[nz] / rms[nz]).max()) if nz.any() else 0.0
        return {"rel_l2": rel, "worst_channel_rel_l2": worst, "underflow": under, "crest": crest}
    return report


def test_independent_numpy_report_holds_every_pin():
    rep = make_report()
    for pin in PINS:
        assert pin(rep) == [], pin.__name__


PLANTED = {
    "rms over nonzero entries only": dict(rms_nonzero=True),
    "crest against the mean magnitude": dict(crest_mean_abs=True),
    "underflow share over all entries": dict(underflow_all=True),
    "rel_l2 as the mean of the rows'": dict(mean_of_rows=True),
    "rel_l2 without the square root": dict(no_sqrt=True),
    "worst channel by absolute error": dict(worst_absolute=True),
    "-0 codes not counted as underflow": dict(minus_zero_kept=True),
    "dequantised without the scale": dict(no_scale=True),
}


@pytest.mark.parametrize("name", sorted(PLANTED))
def test_planted_mistake_fails_a_pin(name):
    rep = make_report(**PLANTED[name])
    failures = [p.__name__ for p in PINS if p(rep)]
    assert failures, "planted mistake '%s' passes every pin" % name
