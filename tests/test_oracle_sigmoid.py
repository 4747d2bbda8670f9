"""Pins for the oracle's pinned logistic function (CPU only).

The score is the "raw sigmoid router score" of "[Dev] Add global-batch
quantile balancing", section "Quantile estimator".  The oracle pins it to one
binary32 operation sequence; these tests tie that sequence to the mathematics
(binary64 logistic, exact Taylor coefficients, limits, symmetry, monotonicity)
rather than to itself.
"""
from fractions import Fraction
from math import factorial

import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

SIGMOID_MAX_ULP = 3.0  # bound of the pinned sequence vs exact logistic (measured max 2.48)
EXP_MAX_ULP = 1.0


def _ref_sigmoid(x):
    xd = x.astype(np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        pos = 1.0 / (1.0 + np.exp(-np.abs(xd)))
        neg = np.exp(-np.abs(xd)) / (1.0 + np.exp(-np.abs(xd)))
    return np.where(xd >= 0, pos, neg)


def _ulps(got, ref):
    r32 = ref.astype(np.float32)
    ulp = np.maximum(np.spacing(np.abs(r32)).astype(np.float64), 2.0 ** -149)
    return np.abs(got.astype(np.float64) - ref) / ulp


def _rn32(fr: Fraction) -> np.float32:
    """Round a rational to the nearest binary32 (ties to even) exactly."""
    lo = np.float32(float(fr))
    cands = [lo, np.nextafter(lo, np.float32(np.inf)), np.nextafter(lo, np.float32(-np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - fr),
                                    int(np.array([c]).view(np.uint32)[0]) & 1))
    return np.float32(best)


def test_taylor_coefficients_are_rn_of_signed_reciprocal_factorials(orc):
    c = orc.exp_coeffs()
    for i in range(8):
        assert c[i] == _rn32(Fraction((-1) ** i, factorial(i))), i


def test_exp_stage_accuracy(orc):
    xs = np.linspace(-88.0, 87.0, 20001, dtype=np.float32)
    got = np.array([orc.exp_neg(float(v)) for v in xs], np.float32)
    ref = np.exp(-xs.astype(np.float64))
    assert _ulps(got, ref).max() <= EXP_MAX_ULP
    # overflow of exp(-x) for x below about -88.72 gives +inf
    assert orc.exp_neg(-89.0) == np.inf and orc.exp_neg(-1e30) == np.inf


NORMAL_MIN = 2.0 ** -126


def _check_accuracy(orc, x):
    ref = _ref_sigmoid(x)
    got = orc.sigmoid(x)
    normal = ref >= NORMAL_MIN
    err = _ulps(got[normal], ref[normal])
    assert err.max() <= SIGMOID_MAX_ULP, (err.max(), x[normal][np.argmax(err)])
    # Below the normal range the pinned function returns a subnormal or 0:
    # never more than 2^-126 away from the exact value.
    assert np.all(np.abs(got[~normal].astype(np.float64) - ref[~normal]) <= NORMAL_MIN)


def test_sigmoid_accuracy_random_bit_patterns(orc):
    rng = np.random.default_rng(12345)
    u = rng.integers(0, 2 ** 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    _check_accuracy(orc, x[np.isfinite(x)])


def test_sigmoid_accuracy_dense_logit_range(orc):
    # Every binary32 value in [-8, 8) with a stride of 7 ulps near 1, plus the tails.
    x = np.concatenate([np.arange(-8.0, 8.0, 2.0 ** -20, dtype=np.float32)[::7],
                        np.linspace(-104.0, 104.0, 400001, dtype=np.float32)])
    _check_accuracy(orc, x)


def test_sigmoid_special_values(orc):
    assert orc.sigmoid(np.float32([0.0]))[0] == np.float32(0.5)
    assert orc.sigmoid(np.float32([-0.0]))[0] == np.float32(0.5)
    big = orc.sigmoid(np.float32([17.5, 50.0, 1e30, np.inf]))
    assert np.all(big == np.float32(1.0))
    tiny = orc.sigmoid(np.float32([-89.0, -100.0, -110.0, -1e30, -np.inf]))
    assert np.all(tiny == 0.0) and not np.any(np.signbit(tiny))
    # Between -88.72 and -87.34 the result is the subnormal 1/(1+exp(-x)).
    x = np.float32([-87.5, -88.0, -88.5])
    ref = 1.0 / (1.0 + np.exp(-x.astype(np.float64)))
    got = orc.sigmoid(x).astype(np.float64)
    assert np.all((got > 0) & (np.abs(got - ref) <= 4 * 2.0 ** -149))


def test_sigmoid_symmetry(orc):
    x = np.linspace(-16.0, 16.0, 100001, dtype=np.float32)
    s = orc.sigmoid(x).astype(np.float64)
    sm = orc.sigmoid(-x).astype(np.float64)
    # s(x) + s(-x) = 1 up to the two results' rounding.
    assert np.max(np.abs(s + sm - 1.0)) <= 3 * 2.0 ** -24


def test_sigmoid_monotone_within_one_ulp(orc):
    x = np.sort(np.concatenate([np.linspace(-110, 110, 1_000_001, dtype=np.float32),
                                np.arange(-1.0, 1.0, 2.0 ** -22, dtype=np.float32)]))
    s = orc.sigmoid(x)
    # Non-decreasing up to one ulp: e = RN(p(w) * 2^n) is a polynomial
    # approximation whose last bit can step back where n changes or p's
    # error turns, and RN(1 / RN(1 + e)) can pass that step on as one ulp.
    dips = s[:-1] - s[1:]
    assert np.all(dips <= np.spacing(s[:-1]))
    # for x >= 0 (e <= 1, absorbed by 1 + e) no dip occurs on this grid
    assert np.all(s[x >= 0][:-1] <= s[x >= 0][1:])
    assert np.all((s >= 0) & (s <= 1))
