"""The tests' single-rounding a * b + c (tests/_util.py ``fma_f32``), which
the GPU tests use to check parameter updates bit for bit, against exact
rational arithmetic: random operands of mixed scales, and operands built so
that the exact result lies just above or just below a float32 rounding
midpoint while the float64 sum lands on it (where rounding twice would pick
the wrong side)."""
from fractions import Fraction

import numpy as np

from tests._util import fma_f32


def _exact(a, b, c):
    """Round a * b + c, computed exactly, to the nearest float32 (ties to even)."""
    v = Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c))
    r = np.float32(float(v))  # one rounding to float64, then the neighbours decide
    cands = [np.nextafter(r, np.float32(-np.inf)), r, np.nextafter(r, np.float32(np.inf))]
    dist = [abs(Fraction(float(x)) - v) for x in cands]
    best = min(dist)
    ties = [x for x, d in zip(cands, dist) if d == best]
    if len(ties) == 1:
        return ties[0]
    return [x for x in ties if (x.view(np.uint32) & 1) == 0][0]


def test_random_operands():
    rng = np.random.default_rng(5)
    n = 4000
    a = (rng.standard_normal(n) * 10.0 ** rng.integers(-3, 3, n)).astype(np.float32)
    b = (rng.standard_normal(n) * 10.0 ** rng.integers(-6, 1, n)).astype(np.float32)
    c = (rng.standard_normal(n) * 10.0 ** rng.integers(-3, 3, n)).astype(np.float32)
    got = fma_f32(a, b, c)
    want = np.array([_exact(x, y, z) for x, y, z in zip(a, b, c)], dtype=np.float32)
    np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))


def test_midpoint_cases_round_once():
    # A * B = 2^47 + m with |m| < 2^17: a * b + 1 = 1 + 2^-24 + m 2^-71, whose float64 sum is the
    # float32 midpoint 1 + 2^-24; the exact value rounds up for m > 0 and down for m < 0
    pairs = [(8390641, 16773151, 124463), (8390644, 16773145, 100052), (8388609, 16777214, -2),
             (8388612, 16777208, -32)]
    for A, B, m in pairs:
        assert A * B - 2 ** 47 == m
        a, b = np.float32(A * 2.0 ** -23), np.float32(B * 2.0 ** -48)
        for sign in (1.0, -1.0):
            c = np.float32(sign)
            got = fma_f32(np.float32(sign) * a, b, c)
            want = _exact(np.float32(sign) * a, b, c)
            assert got.view(np.uint32) == want.view(np.uint32), (A, B, sign)
            away = np.float32(sign * (1.0 + 2.0 ** -23))
            assert (got == away) == (m > 0)
            # rounding the float64 sum lands on the even neighbour, 1, whatever the sign of m
            assert np.float32(float(sign) * float(a) * float(b) + float(c)) == c
