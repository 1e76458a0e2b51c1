"""Exact floating-point identities the CUDA path uses in place of the operation the method
states.  Each test checks, in fp32 on the CPU, that the reformulation gives the same
result as the definition on every input class that matters (ties, the neighbouring
floats of each threshold, zeros, subnormals, infinities, NaN).  The GPU parity tests then
check the kernels themselves against the oracle.

"TAH-Quant" §3.3, eq. (3): a tile is transformed when r = |a1| / (|a2| + rho) exceeds
tau = 2 (fp32 division, rho = 1e-12).  The exact path of the encoder decides this without
a division: with d = RN(|a2| + rho) >= 1e-12, RN(|a1| / d) > 2 holds iff
RN(|a1| / 2 - d) > d * 2^-24 (the halving and the product by 2^-24 are exact, the
difference is exact by Sterbenz's lemma for d <= |a1| <= 4 d, and rounding keeps its sign
and its order against d * 2^-24 elsewhere).
"""

import numpy as np

F = np.float32


def _flag_div(m1, m2):
    d = (m2 + F(1e-12)).astype(F)
    with np.errstate(all="ignore"):
        return (m1 / d).astype(F) > F(2)


def _flag_nodiv(m1, m2):
    d = (m2 + F(1e-12)).astype(F)
    with np.errstate(all="ignore"):
        return ((m1 * F(0.5)).astype(F) - d).astype(F) > (d * F(2.0 ** -24)).astype(F)


def _ulp_steps(x, k):
    up = k > 0
    for _ in range(abs(k)):
        x = np.nextafter(x, F(np.inf) if up else F(0))
    return x


def test_ratio_flag_without_division_near_the_threshold():
    rng = np.random.default_rng(11)
    n = 0
    for ex in range(-42, 127):
        m2 = (F(2.0) ** F(ex) * (1 + rng.random(512)).astype(F)).astype(F)
        m2 = m2[np.isfinite(m2)]
        d = (m2 + F(1e-12)).astype(F)
        # the ratio threshold 2 + 2^-23 and the exact tie at 2 d
        for t in ((d.astype(np.float64) * (2 + 2.0 ** -23)).astype(F),
                  (d.astype(np.float64) * 2).astype(F)):
            for k in range(-3, 4):
                m1 = _ulp_steps(t, k)
                np.testing.assert_array_equal(_flag_div(m1, m2), _flag_nodiv(m1, m2))
                n += m1.size
    assert n > 1_000_000


def test_ratio_flag_without_division_random_and_special():
    rng = np.random.default_rng(12)
    specials = np.array([0.0, 1e-45, 1e-40, 1e-13, 1e-12, 2e-12, 1.0, 2.0, 3.4028235e38,
                         np.inf, np.nan], dtype=F)
    for scale in (1e-40, 1e-20, 1e-12, 1e-3, 1.0, 1e20, 3.4e38):
        m2 = (rng.random(20000) * scale).astype(F)
        m2 = np.concatenate([m2, specials])
        for k in (0.25, 1.0, 1.5, 2.0, 2.0000002, 3.0, 4.0, 4.0001, 1e9, np.inf):
            with np.errstate(all="ignore"):
                m1 = (m2.astype(np.float64) * k).astype(F)
            np.testing.assert_array_equal(_flag_div(m1, m2), _flag_nodiv(m1, m2))
        for s in specials:
            m1 = np.full_like(m2, s)
            np.testing.assert_array_equal(_flag_div(m1, m2), _flag_nodiv(m1, m2))


def _covers_fp32(z, Q, s, mx):
    a = F(F(Q) * F(s))
    sm = F(a + F(z))
    bb = F(sm - a)
    err = F(F(a - F(sm - bb)) + F(F(z) - bb))
    return bool(sm > F(mx) or (sm == F(mx) and err >= 0))


def test_wire_cover_test_in_fp32_is_exact():
    # The wire format's scale is the smallest fp16 s with zero + Q s >= max (exact); the
    # encoder decides the inequality in fp32 with an error-free TwoSum.  Checked against
    # exact rationals where it is hardest: max at, just above and just below zero + Q s.
    from fractions import Fraction
    rng = np.random.default_rng(13)
    for _ in range(40000):
        z = float(np.float16(rng.standard_normal() * 10 ** rng.uniform(-7, 4)))
        s = float(np.float16(abs(rng.standard_normal()) * 10 ** rng.uniform(-7, 3)))
        Q = int(rng.choice([1, 3, 7, 15, 31, 255]))
        exact = Fraction(z) + Q * Fraction(s)
        near = F(float(exact))
        for mx in (near, np.nextafter(near, F(np.inf)), np.nextafter(near, F(-np.inf))):
            assert _covers_fp32(z, Q, s, float(mx)) == (exact >= Fraction(float(mx)))
