"""Exact law of the oracle's output, found by treating the oracle as a black box.

The verify step reads each uniform exactly once: u[i] decides the accept test
at position i, u[N] drives the final sample.  For fixed logits and drafts the
output is therefore a step function of each uniform separately:
  * position i is accepted for u[i] in [0, a_i) and rejected on [a_i, 1);
  * at the stopping position the emitted token is a non-decreasing step
    function of u[N] (inverse CDF in ascending token order).
Bisection on the oracle's own outputs finds every step edge to the last bit,
so integrating over the uniforms is exact up to double rounding.  Summing over
all draft tuples d, weighted by prod_i p_i(d_i) (p from scipy's softmax, not
from the oracle), gives the exact probability of every emitted sequence.
Nothing here re-implements the accept rule, the residual or the sampler.
"""
from __future__ import annotations

import ctypes
import itertools

import numpy as np
from scipy.special import softmax

ONE_MINUS = np.nextafter(1.0, 0.0)


class BlackBox:
    """B=1 calls of an oracle library with preallocated buffers."""

    def __init__(self, orc, zq, zp, T, dtype="f64", greedy=False):
        self.orc = orc
        self.zq = np.ascontiguousarray(zq, dtype=np.float64)[None]
        self.N = self.zq.shape[1] - 1
        self.V = self.zq.shape[2]
        self.zp = (np.ascontiguousarray(zp, dtype=np.float64)[None]
                   if self.N > 0 else np.zeros((1, 0, self.V)))
        self.T = np.array([T], np.float64)
        self.greedy = int(greedy)
        self.tok = np.zeros((1, self.N), np.int32)
        self.u = np.zeros((1, self.N + 1), np.float64)
        self.out = np.zeros((1, self.N + 1), np.int32)
        self.acc = np.zeros((1,), np.int32)
        self.st = np.zeros((1,), np.int32)
        self.calls = 0

    def run(self, d, u):
        self.tok[0, :] = d
        self.u[0, :] = u
        rc = self.orc.lib.orc_verify(
            self.zq.ctypes.data, self.zp.ctypes.data, 2, self.tok.ctypes.data,
            self.u.ctypes.data, self.T.ctypes.data, self.greedy, 1, self.N, self.V,
            self.out.ctypes.data, self.acc.ctypes.data, None, None, None, None,
            None, None, self.st.ctypes.data, None, 1)
        assert rc == 0
        self.calls += 1
        return self.out[0].copy(), int(self.acc[0])


def _accept_edge(bb, d, j):
    """a_j: position j (reached by accepting 0..j-1 at u=0) is accepted
    exactly for u[j] < a_j."""
    N = bb.N

    def accepted(x):
        u = np.zeros(N + 1)
        u[j] = x
        return bb.run(d, u)[1] > j

    if not accepted(0.0):
        return 0.0
    if accepted(ONE_MINUS):
        return 1.0
    lo, hi = 0.0, ONE_MINUS
    while True:
        mid = 0.5 * (lo + hi)
        if mid <= lo or mid >= hi:
            return hi
        if accepted(mid):
            lo = mid
        else:
            hi = mid


def _sample_steps(bb, d, j, u_reject):
    """[(token, measure)] of the emitted token at stop position j over u[N]."""
    N = bb.N

    def token(x):
        u = np.zeros(N + 1)
        if j < N:
            u[j] = u_reject
        u[N] = x
        out, acc = bb.run(d, u)
        assert acc == j, (acc, j)
        return int(out[j])

    steps = []
    x0 = 0.0
    t0 = token(x0)
    while True:
        t_end = token(ONE_MINUS)
        if t_end == t0:
            steps.append((t0, 1.0 - x0))
            return steps
        lo, hi = x0, ONE_MINUS  # token(lo) == t0, token(hi) != t0
        while True:
            mid = 0.5 * (lo + hi)
            if mid <= lo or mid >= hi:
                break
            if token(mid) == t0:
                lo = mid
            else:
                hi = mid
        steps.append((t0, hi - x0))
        x0 = hi
        t0 = token(x0)


def exact_law(orc, zq, zp, T=1.0):
    """{emitted tuple: probability} and {(j, emitted tuple): probability}
    when d_i ~ p_i independently (context-free distributions)."""
    bb = BlackBox(orc, zq, zp, T)
    N, V = bb.N, bb.V
    p = [softmax(np.asarray(zp[i], np.float64) / T) for i in range(N)]
    law = {}
    for d in itertools.product(range(V), repeat=N):
        w = 1.0
        for i in range(N):
            w *= p[i][d[i]]
        if w == 0.0:
            continue
        reach = 1.0
        for j in range(N + 1):
            if j < N:
                a = _accept_edge(bb, d, j)
                stop = reach * (1.0 - a)
                u_rej = 0.5 * (a + 1.0)
            else:
                a = None
                stop = reach
                u_rej = None
            if stop > 0.0:
                for t, meas in _sample_steps(bb, d, j, u_rej):
                    key = tuple(d[:j]) + (t,)
                    law[key] = law.get(key, 0.0) + w * stop * meas
            if j < N:
                reach *= a
                if reach == 0.0:
                    break
    return law


def target_dists(zq, T=1.0):
    return [softmax(np.asarray(z, np.float64) / T) for z in zq]


def draft_dists(zp, T=1.0):
    return [softmax(np.asarray(z, np.float64) / T) for z in zp]


def expected_tokens(law):
    return sum(pr * len(s) for s, pr in law.items())
