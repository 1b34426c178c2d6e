"""The tree walk's closed form of the sibling residual, checked against the
recurrence it replaces (float64, CPU).

The tree rule (a reading: the lesson's "Medusa" and "EAGLE" sections name
candidate trees, and "A friend writes first and the teacher grades", section
"The guarantee that the answer does not change", requires the verifier's
distribution to be kept; the oracle's tree walk states the rule in full):
after child k of a node is rejected, the next child is tested against
r_{k+1} = (r_k - p)+ / R_{k+1}, R_{k+1} = sum (r_k - p)+, starting from r_0 = q,
and r_k stays when R_{k+1} = 0.  The GPU walk keeps two scalars instead of the
vector: r_k = (q - c_k p)+ / Z_k with c_0 = 0, Z_0 = 1; a rejection moves c to
c + Z and Z to sum (q - (c + Z) p)+ (neither moves when that sum is 0).
"""
import numpy as np
import pytest


def _recurrence(q, p, rejections):
    r = q.copy()
    out = [r.copy()]
    for _ in range(rejections):
        d = np.maximum(r - p, 0.0)
        R = d.sum()
        if R > 0.0:
            r = d / R
        out.append(r.copy())
    return out


def _closed_form(q, p, rejections):
    c, Z = 0.0, 1.0
    out = [np.maximum(q - c * p, 0.0) / Z]
    for _ in range(rejections):
        c1 = c + Z
        Z1 = np.maximum(q - c1 * p, 0.0).sum()
        if Z1 > 0.0:
            c, Z = c1, Z1
        out.append(np.maximum(q - c * p, 0.0) / Z)
    return out


def _softmax(z):
    e = np.exp(z - z.max())
    return e / e.sum()


@pytest.mark.parametrize("seed", range(6))
def test_closed_form_equals_the_recurrence(seed):
    rng = np.random.default_rng(seed)
    V = 257
    q = _softmax(rng.normal(size=V) * 2.0)
    p = _softmax(rng.normal(size=V) * 2.0 + 0.5 * np.log(q))
    for a, b in zip(_recurrence(q, p, 12), _closed_form(q, p, 12)):
        assert np.allclose(a, b, rtol=1e-9, atol=1e-15)
        assert abs(b.sum() - 1.0) < 1e-9


def test_empty_residual_keeps_the_distribution():
    """q <= p everywhere the draft has mass: the residual after the first
    rejection is q's excess only; once q - c p <= 0 everywhere the residual is
    empty and r stays."""
    q = np.array([0.5, 0.5, 0.0, 0.0])
    p = np.array([0.25, 0.25, 0.25, 0.25])
    rec = _recurrence(q, p, 4)
    cf = _closed_form(q, p, 4)
    for a, b in zip(rec, cf):
        assert np.allclose(a, b)
    # the excess (0.25, 0.25) normalises to q itself; then c grows until q - c p <= 0
    assert np.allclose(rec[1], q)


def test_zero_probability_draft_elements():
    """Elements the draft never proposes (p = 0) keep their whole q mass in
    every residual."""
    rng = np.random.default_rng(9)
    q = _softmax(rng.normal(size=64))
    p = _softmax(rng.normal(size=64))
    p[::5] = 0.0
    p /= p.sum()
    for a, b in zip(_recurrence(q, p, 8), _closed_form(q, p, 8)):
        assert np.allclose(a, b, rtol=1e-9, atol=1e-15)
