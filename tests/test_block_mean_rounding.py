"""The rounding argument behind the device's partial-block mean: for an fp32 sum s of
n = 2 .. 15 tokens, rounding the IEEE fp32 quotient RN32(s / n) to bf16 or to FP8 E4M3
(round to nearest even, E4M3 saturating at 448) gives what rounding the exact quotient
gives.  Checked here in exact rational arithmetic on random sums and on sums placed on or
beside n times a rounding midpoint (the cases where a second rounding could go wrong)."""
from fractions import Fraction as Fr

import numpy as np

from midpoint_sums import midpoint_sums

FORMATS = {"bf16": dict(p=8, emin=-126, maxv=None), "e4m3": dict(p=4, emin=-6, maxv=448)}


def _rn(x: Fr, p: int, emin: int, maxv) -> Fr:
    """x rounded to p significant bits (exponent at least emin: fixed step below 2^emin),
    ties to even, magnitude clamped to maxv."""
    if x == 0:
        return Fr(0)
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fr(2) ** e > a:
        e -= 1
    while Fr(2) ** (e + 1) <= a:
        e += 1
    q = Fr(2) ** (max(e, emin) - (p - 1))
    r = a / q
    k = r.numerator // r.denominator
    f = r - k
    if f > Fr(1, 2) or (f == Fr(1, 2) and k % 2 == 1):
        k += 1
    v = k * q
    if maxv is not None and v > maxv:
        v = Fr(maxv)
    return v if x > 0 else -v


def _check(s: np.ndarray, n: np.ndarray, fmt: str) -> int:
    F = FORMATS[fmt]
    q32 = (s / n.astype(np.float32)).astype(np.float32)  # IEEE division, rounded once to fp32
    bad = 0
    for si, ni, qi in zip(s.ravel(), n.ravel(), q32.ravel()):
        if _rn(Fr(float(qi)), **F) != _rn(Fr(float(si)) / int(ni), **F):
            bad += 1
    return bad


def test_random_sums():
    rng = np.random.default_rng(11)
    n = rng.integers(2, 16, size=4000)
    s = (rng.standard_normal(4000) * np.exp2(rng.integers(-90, 20, size=4000))).astype(np.float32)
    for fmt in FORMATS:
        assert _check(s, n, fmt) == 0, fmt


def test_sums_at_and_beside_midpoints():
    rng = np.random.default_rng(12)
    for fmt in FORMATS:
        n = rng.integers(2, 16, size=6000)
        s = midpoint_sums(rng, n.astype(np.float64), fmt, max_steps=3)
        assert _check(s, n, fmt) == 0, fmt


def test_the_check_sees_a_second_rounding_go_wrong():
    """The same check catches the failure it rules out when the intermediate is coarser:
    rounding s / n to 12 significant bits first, then to bf16, does go wrong at some midpoints."""
    rng = np.random.default_rng(13)
    n = rng.integers(3, 16, size=3000)
    s = midpoint_sums(rng, n.astype(np.float64), "bf16", max_steps=3)
    bad = 0
    for si, ni in zip(s, n):
        x = Fr(float(si)) / int(ni)
        coarse = _rn(x, 12, -126, None)
        bad += _rn(coarse, 8, -126, None) != _rn(x, 8, -126, None)
    assert bad > 0
