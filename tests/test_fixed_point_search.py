"""The inverse CDF's fixed-point slice masses, emulated on the host (CPU).

Kernel C and the tree walk turn each float warp share x into the integer
floor(x 2^62) and the target into floor(u R) with one 64 x 64-bit high
product.  The same integer steps are restated here and checked against exact
rational arithmetic: the conversion is exact for every share the kernels can
meet above 2^-38, the product is exactly floor(u R), and therefore the slice
found by integer prefix sums is the one exact arithmetic finds.
"""
from fractions import Fraction

import numpy as np


def f32_bits(x):
    return int(np.float32(x).view(np.uint32))


def fx_of(x):
    bits = f32_bits(x)
    e = (bits >> 23) & 0xFF
    if (bits >> 31) or e == 0:
        return 0
    e = min(e, 127)
    m = (bits & 0x7FFFFF) | 0x800000
    sh = e - 88
    return (m << sh) if sh >= 0 else ((m >> -sh) if sh > -24 else 0)


def fx_scale(u, R):
    bits = f32_bits(u)
    e = (bits >> 23) & 0xFF
    if (bits >> 31) or e == 0:
        return 0
    m = (bits & 0x7FFFFF) | 0x800000
    sh = e - 86
    ux = (m << min(sh, 40)) if sh >= 0 else ((m >> -sh) if sh > -24 else 0)
    return (ux * R) >> 64


def test_fx_of_is_exact_above_two_to_minus_38():
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.random(20000), 10.0 ** rng.uniform(-11, 0, 20000), [1.0, 0.5, 2.0 ** -38]])
    for x in xs.astype(np.float32):
        want = Fraction(float(x)) * 2 ** 62
        assert fx_of(x) == int(want) and want.denominator == 1, x  # an exact integer
    # below 2^-38 the bits under 2^-62 are dropped: less than 2^-62 lost
    for x in (10.0 ** rng.uniform(-30, -12, 2000)).astype(np.float32):
        lost = Fraction(float(x)) * 2 ** 62 - fx_of(x)
        assert 0 <= lost < 1
    assert fx_of(np.float32(0.0)) == 0 and fx_of(np.float32(-0.0)) == 0


def test_fx_scale_is_floor_of_u_times_r():
    rng = np.random.default_rng(2)
    for _ in range(20000):
        u = np.float32(rng.random())
        R = int(rng.integers(1, 2 ** 62, dtype=np.int64)) if rng.random() < 0.5 else fx_of(np.float32(rng.random()))
        if f32_bits(u) >> 23 < 86:  # u below 2^-40: truncated, within one unit
            assert fx_scale(u, R) <= int(Fraction(float(u)) * R)
            continue
        assert fx_scale(u, R) == int(Fraction(float(u)) * R)
        assert fx_scale(u, R) < R or R == 0


def test_slice_search_matches_exact_arithmetic():
    """The slice where floor(u R) first falls below the running fixed-point
    total is the slice where u * (exact total) falls, unless u * total lies
    within 2^-62 of a slice edge."""
    rng = np.random.default_rng(3)
    for _ in range(300):
        S = int(rng.integers(1, 80))
        shares = (rng.random((S, 8)) ** rng.uniform(1, 12)).astype(np.float32) * np.float32(1e-3)
        slices = [sum(fx_of(x) for x in row) for row in shares]
        R = sum(slices)
        u = np.float32(rng.random())
        x = fx_scale(u, R)
        run, cs = 0, -1
        for k, m in enumerate(slices):
            if x < run + m:
                cs = k
                break
            run += m
        exact = [sum(Fraction(float(v)) for v in row) for row in shares]
        target = Fraction(float(u)) * sum(exact)
        acc, want = Fraction(0), -1
        for k, m in enumerate(exact):
            if target < acc + m:
                want = k
                break
            acc += m
        near_edge = any(abs(target - sum(exact[:k])) * 2 ** 62 < 2 * S * 8 for k in range(S + 1))
        assert cs == want or near_edge, (cs, want)
