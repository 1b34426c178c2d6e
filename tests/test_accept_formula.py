"""The kernels' accept test, emulated on the host, against its definition
(CPU).

The test is u < min(1, q(x)/p(x)) with q(x) = exp((zq - mq)/T)/Sq and
p(x) = exp((zp - mp)/T)/Sp ("Speculative decoding -- draft, verify, repeat",
section "Core algorithm", step 4).  The kernels evaluate the ratio without a
double-precision exp or division: c = log2(e)/T once per sequence (double),
lq = (zq - mq) c, lp = (zp - mp) c, L = lq - lp, then 2^frac(L) in float32
times Sp/Sq (float32) scaled by 2^floor(L); only when lq or lp is below -1000
are q and p evaluated as the definition does.  Here the same steps run in
numpy (2^frac rounded to float32, like the SFU's result), and the ratio is
compared with the definition in extended precision over logits far outside
float32's exp range.  Below -1000 the kernels decide as the float64 oracle
does, so there the comparison is with the definition evaluated in float64:
when p(x) underflows to 0 there, both accept.
"""
import numpy as np

LOG2E = 1.4426950408889634074


def kernel_ratio(zq, zp, mq, mp, Sq, Sp, T):
    cfd = LOG2E / float(T)
    lq = (float(np.float32(zq)) - float(np.float32(mq))) * cfd
    lp = (float(np.float32(zp)) - float(np.float32(mp))) * cfd
    if lq < -1000.0 or lp < -1000.0:
        qd = 2.0 ** lq / float(Sq)
        pd = 2.0 ** lp / float(Sp)
        return np.inf if pd == 0.0 else qd / pd
    L = lq - lp
    fl = np.floor(L)
    frac = np.float32(L - fl)
    m = np.float32(np.float32(2.0) ** frac) * np.float32(np.float32(Sp) / np.float32(Sq))
    return float(np.ldexp(float(m), int(fl)))


def reference_ratio(zq, zp, mq, mp, Sq, Sp, T):
    ld = np.longdouble
    q = np.exp((ld(np.float32(zq)) - ld(np.float32(mq))) / ld(np.float32(T))) / ld(np.float32(Sq))
    p = np.exp((ld(np.float32(zp)) - ld(np.float32(mp))) / ld(np.float32(T))) / ld(np.float32(Sp))
    return q / p


def test_ratio_matches_the_definition_over_wide_ranges():
    rng = np.random.default_rng(5)
    worst = 0.0
    for _ in range(20000):
        T = np.float32(10.0 ** rng.uniform(-1.5, 1.0))
        mq, mp = np.float32(rng.normal(0, 20)), np.float32(rng.normal(0, 20))
        # logits up to a few hundred below their row maximum, scaled by 1/T
        zq = np.float32(mq - abs(rng.normal(0, 60)))
        zp = np.float32(mp - abs(rng.normal(0, 60)))
        Sq, Sp = np.float32(10.0 ** rng.uniform(0, 5)), np.float32(10.0 ** rng.uniform(0, 5))
        cfd = LOG2E / float(T)
        if (float(zq) - float(mq)) * cfd < -1000.0 or (float(zp) - float(mp)) * cfd < -1000.0:
            continue  # the float64 branch, below
        ref = reference_ratio(zq, zp, mq, mp, Sq, Sp, T)
        got = kernel_ratio(zq, zp, mq, mp, Sq, Sp, T)
        if ref > 1e300 or ref < 1e-300:
            continue
        worst = max(worst, abs(got / float(ref) - 1.0))
    # float32 2^frac and Sp/Sq: a few units in the last place of float32
    assert worst < 5e-7, worst


def test_decisions_agree_outside_the_band():
    rng = np.random.default_rng(6)
    for _ in range(20000):
        T = np.float32(10.0 ** rng.uniform(-1.0, 0.5))
        mq = mp = np.float32(0.0)
        zq = np.float32(-abs(rng.normal(0, 4)))
        zp = np.float32(-abs(rng.normal(0, 4)))
        Sq, Sp = np.float32(rng.uniform(1, 50)), np.float32(rng.uniform(1, 50))
        u = float(np.float32(rng.random()))
        ref = float(min(1.0, reference_ratio(zq, zp, mq, mp, Sq, Sp, T)))
        if abs(u - ref) < 1e-6:  # the parity tests' margin band
            continue
        assert (u < min(1.0, kernel_ratio(zq, zp, mq, mp, Sq, Sp, T))) == (u < ref)


def float64_definition(zq, zp, mq, mp, Sq, Sp, T):
    """The oracle's evaluation: q(x), p(x) in float64; p(x) == 0 accepts."""
    q = np.exp((float(np.float32(zq)) - float(np.float32(mq))) / float(np.float32(T))) / float(np.float32(Sq))
    p = np.exp((float(np.float32(zp)) - float(np.float32(mp))) / float(np.float32(T))) / float(np.float32(Sp))
    return np.inf if p == 0.0 else q / p


def test_underflow_branch_follows_the_float64_definition():
    rng = np.random.default_rng(7)
    with np.errstate(under="ignore", over="ignore"):
        # q(x) underflows, p(x) does not: the ratio is 0 and the test rejects
        T = np.float32(0.05)
        assert kernel_ratio(-200.0, -1.0, 0.0, 0.0, 1.0, 1.0, T) == float64_definition(-200.0, -1.0, 0.0, 0.0, 1.0,
                                                                                        1.0, T) == 0.0
        # both underflow in float64: p(x) == 0, both accept
        assert kernel_ratio(-60.0, -60.5, 0.0, 0.0, 2.0, 3.0, np.float32(0.04)) == np.inf
        assert float64_definition(-60.0, -60.5, 0.0, 0.0, 2.0, 3.0, np.float32(0.04)) == np.inf
        # near the threshold: the two agree to float64 rounding (q or p may be
        # subnormal there, with as few as a dozen significant bits)
        for _ in range(2000):
            T = np.float32(10.0 ** rng.uniform(-2.0, -1.0))
            zq, zp = np.float32(-rng.uniform(5, 9)), np.float32(-rng.uniform(5, 9))
            Sq, Sp = np.float32(rng.uniform(1, 10)), np.float32(rng.uniform(1, 10))
            cfd = LOG2E / float(T)
            if float(zq) * cfd >= -1000.0 and float(zp) * cfd >= -1000.0:
                continue
            a = kernel_ratio(zq, zp, 0.0, 0.0, Sq, Sp, T)
            b = float64_definition(zq, zp, 0.0, 0.0, Sq, Sp, T)
            if np.isinf(b) or b == 0.0:
                assert a == b
            else:
                assert abs(a / b - 1.0) < 1e-3


def test_sibling_test_is_exact():
    """The walk tests a later sibling with u < 1 and u * p(x) < r_k(x), u, p and
    r_k float32 promoted to double: the product of two float32 values is exact
    in double, so the comparison equals u < min(1, r_k/p) in rational
    arithmetic for every input with p > 0, ties included (no quotient is
    rounded)."""
    from fractions import Fraction
    rng = np.random.default_rng(8)
    cases = 0
    for k in range(20000):
        if k % 4 == 0:
            # exact ties: short mantissas, so u * p is a float32 and r_k = u * p
            u = np.float32(rng.integers(1, 256) / 256.0)
            p = np.float32(rng.integers(1, 4096) * 2.0 ** -int(rng.integers(12, 60)))
            r = np.float32(float(u) * float(p))
            assert float(r) == float(u) * float(p)
        else:
            u = np.float32(rng.random())
            p = np.float32(10.0 ** rng.uniform(-30, 0))
            r = np.float32(float(u) * float(p) * (1.0 + rng.uniform(-1e-6, 1e-6)))
        if p == 0 or not np.isfinite(r):
            continue
        exact = Fraction(float(u)) < min(Fraction(1), Fraction(float(r)) / Fraction(float(p)))
        product = (float(u) < 1.0) and (float(u) * float(p) < float(r))
        assert product == exact
        cases += 1
    assert cases > 19000
