"""Pins of the oracle: checks against what the pages and the mathematics fix.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees.  The same battery runs against the real oracle
(test_oracle_pins.py) and against copies with planted mistakes
(test_oracle_mutants.py), which must each fail at least one pin.
"""
from __future__ import annotations

import math
import os

import numpy as np
from scipy.special import logsumexp, softmax

import lawlib
import treelaw

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_numbers.txt")
NEG_INF = -np.inf
ONE_MINUS = np.nextafter(1.0, 0.0)


def golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, rest = line.split("=", 1)
            parts = rest.split(";")
            val = float(parts[0])
            tol = float(parts[1]) if len(parts) > 1 else 0.0
            vals[key.strip()] = (val, tol)
    return vals


def _log(p):
    p = np.asarray(p, np.float64)
    with np.errstate(divide="ignore"):
        return np.log(p)


def _fixed_positions(q, p, N):
    """Context-free case: the same q and p at every position."""
    zq = np.stack([_log(q)] * (N + 1))
    zp = np.stack([_log(p)] * N) if N else np.zeros((0, len(q)))
    return zq, zp


def _alpha(q, p):
    return float(np.minimum(np.asarray(q), np.asarray(p)).sum())


# ---------------------------------------------------------------------------
# Softmax normaliser against scipy
# ---------------------------------------------------------------------------

def pin_softmax_matches_scipy(orc):
    rng = np.random.default_rng(11)
    for V, T, scale in [(7, 1.0, 1.0), (64, 0.7, 3.0), (257, 2.5, 5.0), (1, 1.0, 1.0)]:
        z = rng.normal(0.0, scale, V)
        probs, m, S = orc.softmax_row(z, T, dtype="f64")
        want = softmax(z / T)
        assert np.allclose(probs, want, rtol=1e-13, atol=0), (V, T)
        # log-normaliser: m/T + log S == logsumexp(z/T)
        assert abs(m / T + math.log(S) - logsumexp(z / T)) < 1e-12
    # end to end: the diagnostics q(d), p(d) and (m, S) of the batched call
    B, N, V, T = 3, 2, 40, 0.8
    zq = rng.normal(0, 2, (B, N + 1, V))
    zp = rng.normal(0, 2, (B, N, V))
    d = rng.integers(0, V, (B, N)).astype(np.int32)
    u = np.full((B, N + 1), 0.5)
    r = orc.verify(zq, zp, d, u, np.full(B, T), dtype="f64")
    for b in range(B):
        for i in range(N):
            assert abs(r["q_at_d"][b, i] - softmax(zq[b, i] / T)[d[b, i]]) < 1e-14
            assert abs(r["p_at_d"][b, i] - softmax(zp[b, i] / T)[d[b, i]]) < 1e-14
        for i in range(N + 1):
            m, S = r["tstats"][b, i]
            assert m == zq[b, i].max()
            assert abs(m / T + math.log(S) - logsumexp(zq[b, i] / T)) < 1e-12


# ---------------------------------------------------------------------------
# Exact law: output distribution equals ancestral sampling from q
# ---------------------------------------------------------------------------

def _check_law(law, zq, zp, T, tol=1e-10):
    N = zq.shape[0] - 1
    q = lawlib.target_dists(zq, T)
    p = lawlib.draft_dists(zp, T)
    total = sum(law.values())
    assert abs(total - 1.0) < tol, total
    for s in law:
        assert 1 <= len(s) <= N + 1
    for k in range(N + 1):
        # joint over (accepted prefix x of length k, next emitted token y)
        joint = {}
        for s, pr in law.items():
            if len(s) >= k + 1:
                joint.setdefault(s[:k], np.zeros(len(q[k])))[s[k]] += pr
        for x, row in joint.items():
            mass = row.sum()
            # P(first k tokens are the accepted drafts x) = prod min(p_i, q_i)
            want_mass = 1.0
            for i in range(k):
                want_mass *= min(p[i][x[i]], q[i][x[i]])
            assert abs(mass - want_mass) < tol, (k, x, mass, want_mass)
            if mass > 1e-9:
                assert np.allclose(row / mass, q[k], atol=tol / mass, rtol=0), (k, x, row / mass, q[k])


def pin_exact_law_small(orc):
    """Every draft tuple, every uniform: V <= 4, N <= 2, random q_i, p_i."""
    rng = np.random.default_rng(5)
    cases = [(3, 2, 1.0), (4, 1, 0.7), (2, 2, 1.3), (4, 2, 1.0)]
    for V, N, T in cases:
        zq = rng.normal(0, 1.5, (N + 1, V))
        zp = rng.normal(0, 1.5, (N, V))
        law = lawlib.exact_law(orc, zq, zp, T)
        _check_law(law, zq, zp, T)


def pin_exact_law_with_zero_mass(orc):
    """Tokens with zero probability on either side (-inf logits)."""
    zq = np.array([[0.0, -np.inf, 1.0, 0.5], [0.3, 0.2, -np.inf, -np.inf], [0.0, 0.0, 0.0, 0.0]])
    zp = np.array([[1.0, 0.0, -np.inf, 0.2], [-np.inf, 0.0, 0.0, 2.0]])
    law = lawlib.exact_law(orc, zq, zp, 1.0)
    _check_law(law, zq, zp, 1.0)
    for s in law:
        # a token the verifier gives zero mass is never emitted
        for k, t in enumerate(s):
            assert np.isfinite(zq[k][t]), s


# ---------------------------------------------------------------------------
# Worked numbers from the pages
# ---------------------------------------------------------------------------

def pin_worked_accept_probability(orc):
    g = golden()
    want, tol = g["accept_prob.draft0.9.verifier0.45"]
    q = np.array([0.45, 0.55])
    p = np.array([0.9, 0.1])
    bb = lawlib.BlackBox(orc, _log([q, q]), _log([p]), 1.0)
    edge = lawlib._accept_edge(bb, [0], 0)
    assert abs(edge - want) < tol, edge


def pin_worked_tokens_per_call(orc):
    g = golden()
    q, p = np.array([0.75, 0.25]), np.array([0.5, 0.5])  # alpha = 0.75
    assert abs(_alpha(q, p) - 0.75) < 1e-15
    zq, zp = _fixed_positions(q, p, 5)
    law = lawlib.exact_law(orc, zq, zp)
    e = lawlib.expected_tokens(law)
    want, tol = g["tokens_per_call.a0.75.N5"]
    assert abs(e - want) < tol, e
    rounded, rtol = g["tokens_per_call.a0.75.N5.page_rounded"]
    assert abs(e - rounded) < rtol


def pin_worked_survival(orc):
    g = golden()
    q, p = np.array([0.8, 0.2]), np.array([0.5, 0.5])  # alpha = 0.7
    N = 4
    zq, zp = _fixed_positions(q, p, N)
    law = lawlib.exact_law(orc, zq, zp)
    for k in range(1, N + 1):
        surv = sum(pr for s, pr in law.items() if len(s) - 1 >= k)
        assert abs(surv - 0.7 ** k) < 1e-10, (k, surv)
        want, tol = g[f"survival.a0.7.k{k}"]
        assert abs(surv - want) < tol, (k, surv, want)


def pin_worked_ten_drafts(orc):
    """alpha = 0.7 and ten drafts: three or four tokens per round (page 4)."""
    g = golden()
    q, p = np.array([0.8, 0.2]), np.array([0.5, 0.5])
    N = 10
    B = 40000
    zq, zp = _fixed_positions(q, p, N)
    rng = np.random.default_rng(3)
    d = (rng.random((B, N)) >= 0.5).astype(np.int32)  # d_i ~ p = (0.5, 0.5)
    u = rng.random((B, N + 1))
    r = orc.verify(np.broadcast_to(zq, (B,) + zq.shape).copy(),
                   np.broadcast_to(zp, (B,) + zp.shape).copy(), d, u, np.ones(B),
                   dtype="f64", diagnostics=False)
    mean = float((r["num_accepted"] + 1).mean())
    closed = (1 - 0.7 ** (N + 1)) / 0.3
    sd = float((r["num_accepted"] + 1).std()) / math.sqrt(B)
    assert abs(mean - closed) < 4 * sd, (mean, closed, sd)
    assert g["emitted.a0.7.N10.low"][0] <= mean <= g["emitted.a0.7.N10.high"][0]


def pin_worked_alpha_0_4(orc):
    g = golden()
    q, p = np.array([0.8, 0.2]), np.array([0.2, 0.8])  # alpha = 0.4
    e = {}
    for N in (3, 7):
        zq, zp = _fixed_positions(q, p, N)
        e[N] = lawlib.expected_tokens(lawlib.exact_law(orc, zq, zp))
        closed = (1 - 0.4 ** (N + 1)) / 0.6
        assert abs(e[N] - closed) < 1e-9, (N, e[N], closed)
    assert e[7] / e[3] <= g["tokens_per_call.a0.4.N7_over_N3.max"][0]


def pin_worked_all_accepted(orc):
    """p == q at every draft position: all N accepted and a bonus, N + 1 tokens."""
    g = golden()
    rng = np.random.default_rng(8)
    N, V, B = 5, 9, 200
    zq = rng.normal(0, 2, (B, N + 1, V))
    zp = zq[:, :N].copy()
    d = rng.integers(0, V, (B, N)).astype(np.int32)
    u = rng.random((B, N + 1))
    u[:, 0] = np.nextafter(1.0, 0.0)  # even the largest uniform accepts
    r = orc.verify(zq, zp, d, u, np.full(B, 0.9), dtype="f64")
    assert (r["num_accepted"] == N).all()
    assert ((r["out_tokens"] >= 0).sum(axis=1) == g["all_accepted.N5.tokens"][0]).all()
    assert (r["out_tokens"][:, :N] == d).all()


def pin_tokens_per_call_range(orc):
    g = golden()
    rng = np.random.default_rng(9)
    B, N, V = 500, 4, 12
    zq = rng.normal(0, 2, (B, N + 1, V))
    zp = rng.normal(0, 2, (B, N, V))
    d = rng.integers(0, V, (B, N)).astype(np.int32)
    u = rng.random((B, N + 1))
    r = orc.verify(zq, zp, d, u, np.full(B, 1.0), dtype="f64")
    n_emit = (r["out_tokens"] >= 0).sum(axis=1)
    assert (n_emit >= g["tokens_per_call.min"][0]).all()
    assert (n_emit <= N + g["tokens_per_call.max_minus_N"][0]).all()
    assert (n_emit == r["num_accepted"] + 1).all()
    for b in range(B):
        j = r["num_accepted"][b]
        assert (r["out_tokens"][b, :j] == d[b, :j]).all()
        assert (r["out_tokens"][b, j + 1:] == -1).all()


# ---------------------------------------------------------------------------
# Invariants and exact boundary semantics
# ---------------------------------------------------------------------------

def pin_disjoint_one_hot(orc):
    """p one-hot on x, q one-hot on y != x: reject at the first position and
    emit y (q(d) = 0 makes the ratio 0, and u < 0 never holds)."""
    V, N = 6, 3
    for x, y in [(0, 5), (4, 1), (2, 3)]:
        zq = np.full((1, N + 1, V), NEG_INF)
        zq[0, :, y] = 0.0
        zp = np.full((1, N, V), NEG_INF)
        zp[0, :, x] = 0.0
        for u0 in (0.0, 0.3, np.nextafter(1.0, 0.0)):
            u = np.array([[u0, 0.5, 0.5, 0.7]])
            r = orc.verify(zq, zp, np.full((1, N), x, np.int32), u, np.ones(1), dtype="f64")
            assert r["num_accepted"][0] == 0
            assert list(r["out_tokens"][0]) == [y, -1, -1, -1]


def pin_strict_comparison(orc):
    """Exact ratio 0.5: u = 0.5 rejects, the next double below accepts."""
    zq = np.zeros((1, 2, 4))                       # q = 1/4 each, exactly
    zp = np.array([[[0.0, 0.0, NEG_INF, NEG_INF]]])  # p = (1/2, 1/2, 0, 0)
    d = np.array([[0]], np.int32)
    r = orc.verify(zq, zp, d, np.array([[0.5, 0.1]]), np.ones(1), dtype="f64")
    assert r["num_accepted"][0] == 0
    r = orc.verify(zq, zp, d, np.array([[np.nextafter(0.5, 0.0), 0.1]]), np.ones(1), dtype="f64")
    assert r["num_accepted"][0] == 1


def pin_inverse_cdf_edges(orc):
    """Residual (q - p)_+ = (0, 0, 1/4, 1/4): u*R below 1/4 gives token 2,
    exactly 1/4 gives token 3 (strict comparison with the cumulative)."""
    zq = np.zeros((1, 2, 4))
    zp = np.array([[[0.0, 0.0, NEG_INF, NEG_INF]]])
    d = np.array([[0]], np.int32)
    for uN, want in [(0.0, 2), (np.nextafter(0.5, 0.0), 2), (0.5, 3), (np.nextafter(1.0, 0.0), 3)]:
        r = orc.verify(zq, zp, d, np.array([[0.75, uN]]), np.ones(1), dtype="f64")
        assert r["num_accepted"][0] == 0
        assert r["out_tokens"][0, 0] == want, (uN, r["out_tokens"][0])
    # bonus from q_N: four equal quarters
    for uN, want in [(0.0, 0), (0.25, 1), (np.nextafter(0.5, 0.0), 1), (0.5, 2), (0.75, 3)]:
        r = orc.verify(zq, zp, d, np.array([[0.1, uN]]), np.ones(1), dtype="f64")
        assert r["num_accepted"][0] == 1
        assert r["out_tokens"][0, 1] == want, (uN, r["out_tokens"][0])


def pin_accept_margin_is_the_distance_to_a_flip(orc):
    """The margin of an accept test is how far the ratio q(d)/p(d) would have
    to move for the decision u < min(1, ratio) to change: |u - ratio| below 1,
    and ratio - u at or above 1 (the threshold is then 1, and the decision
    changes only once the ratio has fallen to u).  Exact cases with dyadic
    probabilities: ratio 1 (identical rows), ratio 2 and ratio 1/2."""
    eps = 2.0 ** -24
    zq = np.zeros((1, 2, 4))                              # q = 1/4 each
    # identical rows: ratio exactly 1; u one float32 step below 1
    for u0, want in [(1.0 - eps, eps), (0.5, 0.5), (0.0, 1.0)]:
        r = orc.verify(zq, zq[:, :1].copy(), np.array([[2]], np.int32), np.array([[u0, 0.3]]), np.ones(1),
                       dtype="f64")
        assert r["num_accepted"][0] == 1
        assert r["ratio_at_d"][0, 0] == 1.0
        assert r["accept_margin"][0, 0] == want, (u0, r["accept_margin"][0, 0])
    # q(d) = 1/2, p(d) = 1/4: ratio 2, always accepted, margin 2 - u
    zq2 = np.array([[[0.0, 0.0, NEG_INF, NEG_INF]] * 2])
    for u0 in (0.0, 0.25, 1.0 - eps):
        r = orc.verify(zq2, np.zeros((1, 1, 4)), np.array([[0]], np.int32), np.array([[u0, 0.3]]), np.ones(1),
                       dtype="f64")
        assert r["num_accepted"][0] == 1 and r["ratio_at_d"][0, 0] == 2.0
        assert r["accept_margin"][0, 0] == 2.0 - u0
    # q(d) = 1/4, p(d) = 1/2: ratio 1/2, margin |u - 1/2| on both sides
    zp = np.array([[[0.0, 0.0, NEG_INF, NEG_INF]]])
    for u0, acc in [(0.1, 1), (0.75, 0)]:
        r = orc.verify(zq, zp, np.array([[0]], np.int32), np.array([[u0, 0.3]]), np.ones(1), dtype="f64")
        assert r["num_accepted"][0] == acc and r["ratio_at_d"][0, 0] == 0.5
        assert r["accept_margin"][0, 0] == abs(u0 - 0.5)
    # a zero draft probability: ratio +inf, accepted whatever u, margin +inf
    zp0 = np.array([[[NEG_INF, 0.0, 0.0, 0.0]]])
    r = orc.verify(zq, zp0, np.array([[0]], np.int32), np.array([[1.0 - eps, 0.3]]), np.ones(1), dtype="f64")
    assert r["num_accepted"][0] == 1 and r["ratio_at_d"][0, 0] == np.inf and r["accept_margin"][0, 0] == np.inf


def pin_zero_draft_probability_accepts(orc):
    """p_i(d_i) == 0 accepts whatever the uniform (ratio taken as +inf)."""
    zq = np.zeros((1, 2, 3))
    zp = np.array([[[0.0, NEG_INF, 0.0]]])
    for u0 in (0.0, 0.5, np.nextafter(1.0, 0.0)):
        r = orc.verify(zq, zp, np.array([[1]], np.int32), np.array([[u0, 0.2]]), np.ones(1), dtype="f64")
        assert r["num_accepted"][0] == 1, u0
        assert r["out_tokens"][0, 0] == 1


def pin_zero_residual_samples_q(orc):
    """q_j == p_j and a forced rejection (u = 1): the residual has no mass and
    the token is drawn from q_j itself."""
    zq = np.log(np.array([[[0.1, 0.2, 0.3, 0.4]] * 2]))
    zp = zq[:, :1].copy()
    for uN, want in [(0.05, 0), (0.2, 1), (0.5, 2), (0.95, 3)]:
        r = orc.verify(zq, zp, np.array([[2]], np.int32), np.array([[1.0, uN]]), np.ones(1), dtype="f64")
        assert r["num_accepted"][0] == 0
        assert r["out_tokens"][0, 0] == want, (uN, r["out_tokens"][0])


def pin_accept_when_verifier_not_below(orc):
    """q(d) >= p(d) always accepts (page 3 and page 4)."""
    rng = np.random.default_rng(13)
    B, N, V = 400, 3, 10
    zq = rng.normal(0, 1.5, (B, N + 1, V))
    zp = rng.normal(0, 1.5, (B, N, V))
    d = rng.integers(0, V, (B, N)).astype(np.int32)
    u = rng.random((B, N + 1))
    r = orc.verify(zq, zp, d, u, np.full(B, 1.0), dtype="f64")
    seen = 0
    for b in range(B):
        j = r["num_accepted"][b]
        for i in range(min(j + 1, N)):
            if r["q_at_d"][b, i] >= r["p_at_d"][b, i]:
                assert i < j, (b, i, j)
                seen += 1
    assert seen > 50


def pin_greedy_rule(orc):
    """Greedy: accept while d_i is the argmax (lowest index on ties, as
    numpy.argmax), emit the argmax at the first mismatch or as the bonus."""
    rng = np.random.default_rng(17)
    B, N, V = 300, 4, 7
    zq = rng.integers(-2, 3, (B, N + 1, V)).astype(np.float64)  # many ties
    a = zq.argmax(axis=2)
    d = a[:, :N].copy().astype(np.int32)
    flip = rng.random((B, N)) < 0.3
    d[flip] = rng.integers(0, V, flip.sum())
    u = rng.random((B, N + 1))
    r = orc.verify(zq, None, d, u, None, greedy=True, dtype="f64")
    for b in range(B):
        j = 0
        while j < N and d[b, j] == a[b, j]:
            j += 1
        assert r["num_accepted"][b] == j
        assert list(r["out_tokens"][b, :j]) == list(d[b, :j])
        assert r["out_tokens"][b, j] == a[b, j]
    # per-sequence greedy through T <= 0
    T = np.where(rng.random(B) < 0.5, 0.0, -1.0)
    r2 = orc.verify(zq, np.zeros((B, N, V)), d, u, T, dtype="f64")
    assert (r2["out_tokens"] == r["out_tokens"]).all()


def pin_greedy_is_zero_temperature_limit(orc):
    """With greedy drafts and well-separated logits, sampling at T -> 0 gives
    the greedy output for any uniforms."""
    rng = np.random.default_rng(19)
    B, N, V = 200, 3, 12
    # logits on a 0.05 grid without ties: exp(-0.05 / T) vanishes at T = 1e-4
    zq = np.stack([np.stack([rng.permutation(V) * 0.05 for _ in range(N + 1)]) for _ in range(B)])
    zp = np.stack([np.stack([rng.permutation(V) * 0.05 for _ in range(N)]) for _ in range(B)])
    d = zp.argmax(axis=2).astype(np.int32)
    same = rng.random((B, N)) < 0.6
    zp[same] = zq[:, :N][same]  # make many drafts agree with the verifier
    d = zp.argmax(axis=2).astype(np.int32)
    u = rng.random((B, N + 1)) * 0.999
    rs = orc.verify(zq, zp, d, u, np.full(B, 1e-4), dtype="f64")
    rg = orc.verify(zq, zp, d, u, None, greedy=True, dtype="f64")
    assert (rs["out_tokens"] == rg["out_tokens"]).all()
    assert (rs["num_accepted"] == rg["num_accepted"]).all()
    assert 0 < rg["num_accepted"].mean() < N


def pin_temperature_divides(orc):
    """softmax(z/T): temperature 2 on z equals temperature 1 on z/2."""
    rng = np.random.default_rng(23)
    B, N, V = 50, 2, 16
    zq = rng.normal(0, 3, (B, N + 1, V))
    zp = rng.normal(0, 3, (B, N, V))
    d = rng.integers(0, V, (B, N)).astype(np.int32)
    u = rng.random((B, N + 1))
    r1 = orc.verify(zq, zp, d, u, np.full(B, 2.0), dtype="f64")
    r2 = orc.verify(zq / 2.0, zp / 2.0, d, u, np.full(B, 1.0), dtype="f64")
    assert np.allclose(r1["q_at_d"], r2["q_at_d"], rtol=1e-13)
    assert np.allclose(r1["p_at_d"], r2["p_at_d"], rtol=1e-13)
    assert np.allclose(r1["q_at_d"], [[softmax(zq[b, i] / 2.0)[d[b, i]] for i in range(N)] for b in range(B)],
                       rtol=1e-13)


def pin_invalid_inputs(orc):
    """Out-of-range drafts and non-finite rows or temperatures give -1."""
    rng = np.random.default_rng(29)
    B, N, V = 8, 2, 5
    zq = rng.normal(0, 1, (B, N + 1, V))
    zp = rng.normal(0, 1, (B, N, V))
    d = rng.integers(0, V, (B, N)).astype(np.int32)
    T = np.ones(B)
    d[0, 1] = V          # bad token
    d[1, 0] = -1         # bad token
    zq[2, 2, 3] = np.nan  # NaN in a target row
    zp[3, 0, 0] = np.inf  # +inf in a draft row
    zq[4, 1, :] = NEG_INF  # a row without mass
    T[5] = np.nan
    T[6] = np.inf
    u = rng.random((B, N + 1))
    r = orc.verify(zq, zp, d, u, T, dtype="f64")
    for b in range(7):
        assert r["num_accepted"][b] == -1 and (r["out_tokens"][b] == -1).all(), b
        assert r["seq_status"][b] != 0
    assert r["seq_status"][0] == 1 and r["seq_status"][1] == 1
    assert r["seq_status"][2] == 2
    assert r["num_accepted"][7] >= 0 and r["seq_status"][7] == 0


def pin_degenerate_sizes(orc):
    # V = 1: every distribution is the point mass on token 0
    r = orc.verify(np.zeros((2, 4, 1)), np.zeros((2, 3, 1)), np.zeros((2, 3), np.int32),
                   np.full((2, 4), 0.99), np.ones(2), dtype="f64")
    assert (r["num_accepted"] == 3).all() and (r["out_tokens"] == 0).all()
    # N = 0: only the bonus token, drawn from q_0 by inverse CDF
    zq = np.log(np.array([[[0.5, 0.25, 0.25]]]))
    for uN, want in [(0.1, 0), (0.6, 1), (0.8, 2)]:
        r = orc.verify(zq, None, np.zeros((1, 0), np.int32), np.array([[uN]]), np.ones(1), dtype="f64")
        assert r["num_accepted"][0] == 0 and r["out_tokens"][0, 0] == want
    # B = 0
    r = orc.verify(np.zeros((0, 3, 4)), np.zeros((0, 2, 4)), np.zeros((0, 2), np.int32),
                   np.zeros((0, 3)), np.zeros(0), dtype="f64")
    assert r["out_tokens"].shape == (0, 3)


def pin_storage_types(orc):
    """bf16 and float32 logits are widened exactly: same result as the
    float64 copy of the same values."""
    import torch
    rng = np.random.default_rng(31)
    B, N, V = 20, 3, 33
    zq = torch.tensor(rng.normal(0, 3, (B, N + 1, V)), dtype=torch.float32)
    zp = torch.tensor(rng.normal(0, 3, (B, N, V)), dtype=torch.float32)
    d = rng.integers(0, V, (B, N)).astype(np.int32)
    u = rng.random((B, N + 1)).astype(np.float32)
    T = np.full(B, 0.8, np.float32)
    for tdt, name in [(torch.float32, "f32"), (torch.bfloat16, "bf16")]:
        a, b_ = zq.to(tdt), zp.to(tdt)
        r = orc.verify(a, b_, d, u, T, dtype=name)
        r64 = orc.verify(a.double().numpy(), b_.double().numpy(), d, u, T, dtype="f64")
        for k in ("out_tokens", "num_accepted"):
            assert (r[k] == r64[k]).all()
        assert np.array_equal(r["q_at_d"], r64["q_at_d"])


# ---- KV-cache commit / rollback ---------------------------------------------

def _kv_row(plane, pos, tok, row_bytes):
    """Bytes that identify (plane, position, token): a stand-in KV entry."""
    r = (np.arange(row_bytes, dtype=np.int64) * 7 + plane * 31 + pos * 13 + tok * 3) % 251
    r[:4] = (plane, pos, tok & 0xFF, (tok >> 8) & 0xFF)
    return r.astype(np.uint8)


def _kv_state(tokens_per_seq, P, max_len, row_bytes, fill=0xEE):
    cache = np.full((P, len(tokens_per_seq), max_len, row_bytes), fill, np.uint8)
    for b, toks in enumerate(tokens_per_seq):
        for p in range(P):
            for pos, t in enumerate(toks):
                cache[p, b, pos] = _kv_row(p, pos, t, row_bytes)
    return cache


def _kv_scratch(drafts_per_seq, starts, P, N, row_bytes):
    s = np.zeros((P, len(drafts_per_seq), N, row_bytes), np.uint8)
    for b, (ds, L) in enumerate(zip(drafts_per_seq, starts)):
        for p in range(P):
            for k, t in enumerate(ds):
                s[p, b, k] = _kv_row(p, L + k, t, row_bytes)
    return s


def _rejection_at(orc, N, reject_1based, V=8):
    """num_accepted from the verify oracle for drafts whose first
    reject_1based - 1 positions have p == q (ratio 1: always accepted) and
    whose next position has disjoint one-hot p and q (ratio 0: always
    rejected), whatever the uniforms."""
    rng = np.random.default_rng(0)
    zq = rng.normal(0, 1, (1, N + 1, V))
    zp = zq[:, :N].copy()
    j = reject_1based - 1
    zq[0, j] = NEG_INF
    zq[0, j, 1] = 0.0
    zp[0, j] = NEG_INF
    zp[0, j, 2] = 0.0
    d = np.zeros((1, N), np.int32)
    for i in range(N):
        d[0, i] = int(np.argmax(zp[0, i]))
    u = np.full((1, N + 1), 0.999, np.float32)
    r = orc.verify(zq, zp, d, u, np.ones(1), dtype="f64")
    return int(r["num_accepted"][0]), d[0]


def pin_kv_exercise_rollback(orc):
    """The lesson's rollback exercise: prefix 10, 5 drafts, rejection at the
    third draft; the cache then reads prefix + the first 2 drafts."""
    g = golden()
    L0 = int(g["kv_rollback.prefix"][0])
    N = int(g["kv_rollback.drafts"][0])
    rej = int(g["kv_rollback.rejected_draft_1based"][0])
    want_acc = int(g["kv_rollback.accepted"][0])
    acc, _ = _rejection_at(orc, N, rej)
    assert acc == want_acc, (acc, want_acc)
    P, row, max_len = 4, 32, 24
    rng = np.random.default_rng(1)
    prefixes = [list(rng.integers(0, 50000, L0)) for _ in range(3)]
    drafts = [list(rng.integers(0, 50000, N)) for _ in range(3)]
    cache = _kv_state(prefixes, P, max_len, row)
    scratch = _kv_scratch(drafts, [L0] * 3, P, N, row)
    nacc = np.array([acc, N, 0], np.int32)
    c2, ln, st = orc.kv_commit(scratch, cache, np.full(3, L0, np.int32), nacc)
    assert st == 0
    assert list(ln) == [L0 + acc, L0 + N, L0]
    for b in range(3):
        seq = prefixes[b] + drafts[b][: nacc[b]]
        assert np.array_equal(c2[:, b, : ln[b]], _kv_state([seq], P, ln[b], row)[:, 0])
        # the rolled-back drafts never reach the cache
        assert (c2[:, b, ln[b]:] == 0xEE).all()
    # next iteration: three more entries land right after the committed ones
    more = [list(rng.integers(0, 50000, N)) for _ in range(3)]
    scratch2 = _kv_scratch(more, list(ln), P, N, row)
    c3, ln3, st = orc.kv_commit(scratch2, c2, ln, np.array([3, 1, 5], np.int32))
    assert st == 0 and list(ln3) == [L0 + acc + 3, L0 + N + 1, L0 + 5]
    for b, k in enumerate([3, 1, 5]):
        seq = prefixes[b] + drafts[b][: nacc[b]] + more[b][:k]
        assert np.array_equal(c3[:, b, : ln3[b]], _kv_state([seq], P, ln3[b], row)[:, 0])


def pin_kv_bad_counts_and_overflow(orc):
    P, B, N, row, max_len = 2, 6, 4, 16, 12
    rng = np.random.default_rng(2)
    cache = rng.integers(0, 256, (P, B, max_len, row), dtype=np.uint8)
    scratch = rng.integers(0, 256, (P, B, N, row), dtype=np.uint8)
    lens = np.array([3, 3, 10, 8, -1, 5], np.int32)
    nacc = np.array([-1, N + 1, 3, 4, 0, 2], np.int32)
    c2, ln, st = orc.kv_commit(scratch, cache, lens, nacc)
    assert st == (1 | 2), st
    # -1: an invalid verify commits nothing and is not an error here
    # N+1: a count the verify cannot produce; 10+3 > 12: overflow; -1 length: bad
    for b in (0, 1, 2, 4):
        assert ln[b] == lens[b] and np.array_equal(c2[:, b], cache[:, b])
    # exactly filling the cache is fine; the others still commit
    assert ln[3] == 12 and np.array_equal(c2[:, 3, 8:12], scratch[:, 3, :4])
    assert ln[5] == 7 and np.array_equal(c2[:, 5, 5:7], scratch[:, 5, :2])
    assert np.array_equal(c2[:, 5, :5], cache[:, 5, :5]) and np.array_equal(c2[:, 5, 7:], cache[:, 5, 7:])
    _, _, st = orc.kv_commit(scratch[:, :1], cache[:, :1], np.array([0], np.int32), np.array([N], np.int32))
    assert st == 0


def pin_kv_planes_and_sequences_stay_apart(orc):
    """Every plane gets its own rows at the sequence's shared length; nothing
    outside [len, len + a) moves (random bytes, several layouts)."""
    rng = np.random.default_rng(3)
    for P, B, N, row, max_len in [(1, 1, 1, 16, 1), (3, 5, 7, 48, 20), (6, 2, 3, 1024, 9)]:
        cache = rng.integers(0, 256, (P, B, max_len, row), dtype=np.uint8)
        scratch = rng.integers(0, 256, (P, B, N, row), dtype=np.uint8)
        nacc = rng.integers(0, N + 1, B).astype(np.int32)
        lens = np.array([rng.integers(0, max_len - a + 1) for a in nacc], np.int32)
        c2, ln, st = orc.kv_commit(scratch, cache, lens, nacc)
        assert st == 0 and np.array_equal(ln, lens + nacc)
        for p in range(P):
            for b in range(B):
                L, a = lens[b], nacc[b]
                assert np.array_equal(c2[p, b, L:L + a], scratch[p, b, :a])
                assert np.array_equal(c2[p, b, :L], cache[p, b, :L])
                assert np.array_equal(c2[p, b, L + a:], cache[p, b, L + a:])
    # no sequences, no drafts
    c2, ln, st = orc.kv_commit(np.zeros((2, 0, 3, 16), np.uint8), np.zeros((2, 0, 4, 16), np.uint8),
                               np.zeros(0, np.int32), np.zeros(0, np.int32))
    assert st == 0 and ln.size == 0
    cache = rng.integers(0, 256, (2, 2, 4, 16), dtype=np.uint8)
    c2, ln, st = orc.kv_commit(np.zeros((2, 2, 0, 16), np.uint8), cache, np.array([1, 4], np.int32),
                               np.zeros(2, np.int32))
    assert st == 0 and list(ln) == [1, 4] and np.array_equal(c2, cache)


# ---- tree verification ---------------------------------------------------------

def _prefix_model(seed, V, scale=1.5, mask=False):
    """Logits after every token prefix, drawn once per prefix (a stand-in for a
    language model); with mask, one token per prefix gets -inf."""
    cache = {}

    def f(prefix):
        key = tuple(int(t) for t in prefix)
        if key not in cache:
            g = np.random.default_rng([seed, len(key)] + [t + 1 for t in key])
            z = g.normal(0.0, scale, V)
            if mask:
                z[g.integers(V)] = NEG_INF
            cache[key] = z
        return cache[key]
    return f


def pin_tree_exact_law(orc):
    """Children drawn independently from their parent's draft distribution,
    every assignment and every uniform: the emitted sequence is distributed as
    ancestral sampling from the verifier, prefix by prefix."""
    cases = [([-1, 0, 0, 1, 1], 3, 1.0, False), ([-1, 0, 0, 0], 3, 0.8, False),
             ([-1, 0, 1, 1, 0], 2, 1.3, False), ([-1, 0, 0, 1], 3, 1.0, True)]
    for i, (parent, V, T, mask) in enumerate(cases):
        mq, mp = _prefix_model(100 + i, V, mask=mask), _prefix_model(200 + i, V, mask=mask)
        law = treelaw.exact_tree_law(orc, parent, V, mq, mp, T)
        treelaw.check_ancestral(law, mq, T)
        depth = max(len(s) for s in law)
        assert depth >= 2, law  # some draft is accepted with positive probability


def pin_tree_chain_is_the_chain_verify(orc):
    """A tree whose nodes form one chain gives the chain verify's outputs
    (uniforms mapped: node n+1 <- u[n], the final sample <- u[N]); the draft
    row of the last node (a leaf) is not read."""
    rng = np.random.default_rng(31)
    B, N, V, T = 60, 4, 6, 0.9
    zq = rng.normal(0, 1.2, (B, N + 1, V))
    zp = rng.normal(0, 1.2, (B, N, V))
    d = rng.integers(0, V, (B, N)).astype(np.int32)
    u = rng.random((B, N + 1))
    parent = np.arange(-1, N, dtype=np.int32)
    tok = np.concatenate([np.zeros((B, 1), np.int32), d], axis=1)
    ut = np.concatenate([u[:, N:], u[:, :N]], axis=1)
    zpt = np.concatenate([zp, np.full((B, 1, V), np.nan)], axis=1)
    for greedy in (False, True):
        c = orc.verify(zq, None if greedy else zp, d, u, None if greedy else np.full(B, T), greedy=greedy, dtype="f64")
        t = orc.tree_verify(zq, None if greedy else zpt, parent, tok, ut, None if greedy else np.full(B, T),
                            greedy=greedy, dtype="f64")
        assert (t["seq_status"] == 0).all()
        sure = (c["sample_margin"] > 1e-12) | greedy
        assert sure.sum() >= B - 2
        assert np.array_equal(c["num_accepted"], t["num_accepted"])
        assert np.array_equal(c["out_tokens"][sure], t["out_tokens"][sure])
        for b in range(B):
            a = c["num_accepted"][b]
            assert list(t["path_nodes"][b][:a]) == list(range(1, a + 1)) and (t["path_nodes"][b][a:] == -1).all()
            if not greedy:
                np.testing.assert_allclose(t["accept_margin"][b, 1:a + 2][: min(a + 1, N)],
                                           c["accept_margin"][b, : min(a + 1, N)], rtol=1e-12)


def pin_tree_worked_siblings(orc):
    """Two children at the root, q_0 = (1/2, 1/2), p_0 = (0.9, 0.1), V = 2.
    The first child (token 0) passes with probability (1/2)/0.9 = 5/9.  After
    its rejection the residual is (0, 1): a second child with token 0 has
    ratio 0 and always fails (the token is then 1), one with token 1 has ratio
    10 and always passes."""
    zq = np.log(np.array([[0.5, 0.5], [0.5, 0.5], [0.5, 0.5]]))[None]
    zp = np.log(np.array([[0.9, 0.1], [0.5, 0.5], [0.5, 0.5]]))[None]
    parent = [-1, 0, 0]
    for toks, u1, want_path, want_first in [((0, 0), 0.6, [], 1), ((0, 1), 0.6, [2], 1), ((0, 1), 0.5, [1], 0),
                                            ((0, 0), 0.5, [1], 0)]:
        r = orc.tree_verify(zq, zp, parent, np.array([[0, *toks]]), np.array([[0.3, u1, 0.99]]), np.ones(1),
                            dtype="f64")
        path = list(r["path_nodes"][0][: r["num_accepted"][0]])
        assert path == want_path, (toks, u1, path)
        assert r["out_tokens"][0][0] == want_first
        assert abs(r["accept_margin"][0][1] - abs(u1 - 5.0 / 9.0)) < 1e-15
        if toks == (0, 0) and u1 > 5.0 / 9.0:
            assert abs(r["accept_margin"][0][2] - 0.99) < 1e-15  # |u - 0|
            assert r["sample_margin"][0] > 0.3 - 1e-15  # the residual is all on token 1
        assert abs(r["ratio_at"][0][1] - 5.0 / 9.0) < 1e-15
        if toks == (0, 1) and u1 > 5.0 / 9.0:
            # ratio r(1)/p(1) = 1/0.1 = 10: accepted, and the ratio would have
            # to fall by 10 - 0.99 to change that
            assert abs(r["ratio_at"][0][2] - 10.0) < 1e-12
            assert abs(r["accept_margin"][0][2] - (10.0 - 0.99)) < 1e-12
    # a child whose token the draft gives probability 0 is accepted (ratio +inf),
    # as in the chain verify, whatever its uniform
    zp0 = np.array([[[0.0, -np.inf], [0.0, 0.0], [0.0, 0.0]]])
    for u1 in (0.0, 0.5, ONE_MINUS):
        r = orc.tree_verify(zq, zp0, parent, np.array([[0, 1, 0]]), np.array([[0.3, u1, 0.5]]), np.ones(1),
                            dtype="f64")
        assert list(r["path_nodes"][0][:1]) == [1] and r["accept_margin"][0][1] == np.inf


def pin_tree_greedy_rule(orc):
    """Greedy: accept the first child (in index order) whose token is the
    verifier's argmax at its parent; emit the argmax where no child matches."""
    V = 6
    zq = np.zeros((1, 6, V))
    zq[0, 0, 3] = 2.0  # root argmax 3
    zq[0, 2, 4] = 1.0  # node 2 argmax 4
    zq[0, 5, 1] = 3.0  # node 5 argmax 1
    zq[0, 3, 0] = 9.0  # node 3 (never reached) argmax 0
    parent = [-1, 0, 0, 0, 2, 2]
    tok = np.array([[0, 1, 3, 3, 2, 4]])
    for greedy, T in [(True, None), (False, np.zeros(1))]:
        r = orc.tree_verify(zq, None if greedy else np.zeros_like(zq), parent, tok, np.full((1, 6), 0.5), T,
                            greedy=greedy, dtype="f64")
        assert list(r["path_nodes"][0][:2]) == [2, 5] and r["num_accepted"][0] == 2
        assert list(r["out_tokens"][0][:3]) == [3, 4, 1] and (r["out_tokens"][0][3:] == -1).all()
    # ties go to the lowest index, as in the chain verify
    zq2 = np.zeros((1, 2, V))
    r = orc.tree_verify(zq2, None, [-1, 0], np.array([[0, 0]]), np.zeros((1, 2)), None, greedy=True, dtype="f64")
    assert r["num_accepted"][0] == 1 and list(r["out_tokens"][0]) == [0, 0]


def pin_tree_invalid_inputs(orc):
    V, M = 5, 3
    rng = np.random.default_rng(41)
    good_parent = np.array([-1, 0, 0, 1], np.int32)
    base = dict(zq=rng.normal(0, 1, (1, M + 1, V)), zp=rng.normal(0, 1, (1, M + 1, V)),
                parent=good_parent, tok=np.array([[0, 1, 2, 3]], np.int32), T=np.ones(1))

    def run(**kw):
        a = {**base, **kw}
        return orc.tree_verify(a["zq"], a["zp"], a["parent"], a["tok"], np.full((1, M + 1), 0.4), a["T"], dtype="f64")

    assert run()["seq_status"][0] == 0
    for bad_parent in ([0, 0, 0, 1], [-1, 0, 2, 1], [-1, 0, 0, -1], [-1, 0, 0, 4]):
        r = run(parent=np.array(bad_parent, np.int32))
        assert r["seq_status"][0] & 4 and r["num_accepted"][0] == -1 and (r["out_tokens"] == -1).all()
    assert run(tok=np.array([[0, 1, V, 3]], np.int32))["seq_status"][0] == 1
    zp = base["zp"].copy()
    zp[0, 1, 2] = np.nan  # node 1 has a child: its draft row is read
    assert run(zp=zp)["seq_status"][0] == 2
    zp = base["zp"].copy()
    zp[0, 3, :] = np.nan  # leaves' draft rows are not read
    zp[0, 2, :] = np.nan
    assert run(zp=zp)["seq_status"][0] == 0
    zq = base["zq"].copy()
    zq[0, 2, 0] = np.inf  # every verifier row is read
    assert run(zq=zq)["seq_status"][0] == 2
    assert run(T=np.array([np.nan]))["seq_status"][0] == 2
    # a root alone: the bonus token from q_0
    r = orc.tree_verify(base["zq"][:, :1], base["zp"][:, :1], [-1], np.zeros((1, 1), np.int32),
                        np.array([[0.25]]), np.ones(1), dtype="f64")
    q0 = softmax(base["zq"][0, 0])
    assert r["num_accepted"][0] == 0 and r["out_tokens"][0][0] == int(np.searchsorted(np.cumsum(q0), 0.25, side="right"))


# ---- the LM-head product ----------------------------------------------------------

def pin_lm_head_definition(orc):
    """logits[r, v] = sum_k hidden[r, k] weight[v, k]: an identity weight
    returns the hidden states, a one-hot hidden row selects a weight column,
    and a tiny case equals the sum written out."""
    import oracle
    rng = np.random.default_rng(51)
    h = rng.normal(size=(3, 4))
    assert np.array_equal(oracle.lm_head_logits(h, np.eye(4)), h)
    w = rng.normal(size=(5, 4))
    e = np.zeros((1, 4))
    e[0, 2] = 1.0
    assert np.array_equal(oracle.lm_head_logits(e, w)[0], w[:, 2])
    got = oracle.lm_head_logits(h, w)
    for r in range(3):
        for v in range(5):
            assert abs(got[r, v] - sum(h[r, k] * w[v, k] for k in range(4))) < 1e-12


ALL_PINS = [
    pin_softmax_matches_scipy,
    pin_exact_law_small,
    pin_exact_law_with_zero_mass,
    pin_worked_accept_probability,
    pin_worked_tokens_per_call,
    pin_worked_survival,
    pin_worked_ten_drafts,
    pin_worked_alpha_0_4,
    pin_worked_all_accepted,
    pin_tokens_per_call_range,
    pin_disjoint_one_hot,
    pin_strict_comparison,
    pin_inverse_cdf_edges,
    pin_accept_margin_is_the_distance_to_a_flip,
    pin_zero_draft_probability_accepts,
    pin_zero_residual_samples_q,
    pin_accept_when_verifier_not_below,
    pin_greedy_rule,
    pin_greedy_is_zero_temperature_limit,
    pin_temperature_divides,
    pin_invalid_inputs,
    pin_degenerate_sizes,
    pin_storage_types,
    pin_kv_exercise_rollback,
    pin_kv_bad_counts_and_overflow,
    pin_kv_planes_and_sequences_stay_apart,
    pin_tree_exact_law,
    pin_tree_chain_is_the_chain_verify,
    pin_tree_worked_siblings,
    pin_tree_greedy_rule,
    pin_tree_invalid_inputs,
    pin_lm_head_definition,
]
