"""Exact law of the tree oracle's output, found by treating it as a black box.

As in the chain case (lawlib.py), every uniform is read by at most one
decision: u[c] by the accept test of node c, u[0] by the final sample.  For
fixed logits and drafts the walk is a step function of each uniform, so the
law over the uniforms is found by bisection on the oracle's own outputs.
Which node is tested next is read off the oracle's outputs too: a node was
tested iff its accept margin is not NaN, and the walk tests the children of
each path node in index order.  The draft tokens are summed over every
assignment, each child drawn independently from its parent's draft
distribution (scipy softmax of the model's logits), with the verifier and
draft logits of every node given by a model of the whole prefix.  Nothing
here re-implements the accept rule, the residual or the sampler.
"""
from __future__ import annotations

import itertools

import numpy as np
from scipy.special import softmax

ONE_MINUS = np.nextafter(1.0, 0.0)


class TreeBox:
    def __init__(self, orc, parent, V, T):
        self.orc = orc
        self.parent = np.asarray(parent, np.int32)
        self.M = len(parent) - 1
        self.V = V
        self.T = T
        self.calls = 0

    def set_logits(self, zq, zp):
        self.zq = np.asarray(zq, np.float64)[None]
        self.zp = np.asarray(zp, np.float64)[None]

    def run(self, tokens, u):
        r = self.orc.tree_verify(self.zq, self.zp, self.parent, np.asarray(tokens, np.int32)[None],
                                 np.asarray(u, np.float64)[None], np.array([self.T]), dtype="f64")
        self.calls += 1
        n = int(r["num_accepted"][0])
        assert n >= 0
        return r["out_tokens"][0], list(r["path_nodes"][0][:n]), r["accept_margin"][0]


def _test_order(parent, path, margin):
    tested = [c for c in range(1, len(parent)) if not np.isnan(margin[c])]
    order, n = [], 0
    for nxt in list(path) + [None]:
        order += sorted(c for c in tested if parent[c] == n)
        if nxt is None:
            break
        n = nxt
    return order


def _edge(box, tokens, u, c):
    """Node c (tested with the other uniforms fixed) is accepted exactly for
    u[c] below the returned value."""
    def accepted(x):
        v = u.copy()
        v[c] = x
        return c in box.run(tokens, v)[1]

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


def _sample_steps(box, tokens, u):
    """[(emitted tuple, measure)] over u[0] with every tested node fixed."""
    def emitted(x):
        v = u.copy()
        v[0] = x
        out, path, _ = box.run(tokens, v)
        return tuple(int(t) for t in out[: len(path) + 1])

    steps, x0 = [], 0.0
    s0 = emitted(x0)
    while True:
        if emitted(ONE_MINUS) == s0:
            steps.append((s0, 1.0 - x0))
            return steps
        lo, hi = x0, ONE_MINUS
        while True:
            mid = 0.5 * (lo + hi)
            if mid <= lo or mid >= hi:
                break
            if emitted(mid) == s0:
                lo = mid
            else:
                hi = mid
        steps.append((s0, hi - x0))
        x0 = hi
        s0 = emitted(x0)


def _explore(box, tokens, fixed, w, law):
    u = np.zeros(box.M + 1)
    for c, x in fixed.items():
        u[c] = x
    _, path, margin = box.run(tokens, u)
    pending = [c for c in _test_order(box.parent, path, margin) if c not in fixed]
    if not pending:
        for s, meas in _sample_steps(box, tokens, u):
            law[s] = law.get(s, 0.0) + w * meas
        return
    c = pending[0]
    a = _edge(box, tokens, u, c)
    if a > 0.0:
        _explore(box, tokens, {**fixed, c: 0.0}, w * a, law)
    if a < 1.0:
        _explore(box, tokens, {**fixed, c: 0.5 * (a + 1.0)}, w * (1.0 - a), law)


def node_prefixes(parent, tokens):
    """Token prefix (path from the root, root excluded) of every node."""
    pre = [()]
    for n in range(1, len(parent)):
        pre.append(pre[parent[n]] + (int(tokens[n]),))
    return pre


def exact_tree_law(orc, parent, V, model_q, model_p, T=1.0):
    """{emitted tuple: probability}; model_q / model_p map a prefix tuple to
    the verifier / draft logits after it."""
    box = TreeBox(orc, parent, V, T)
    M = len(parent) - 1
    law = {}
    for assign in itertools.product(range(V), repeat=M):
        tokens = (0,) + assign
        pre = node_prefixes(parent, tokens)
        w = 1.0
        for c in range(1, M + 1):
            w *= softmax(np.asarray(model_p(pre[parent[c]]), np.float64) / T)[tokens[c]]
        if w == 0.0:
            continue
        box.set_logits([model_q(pre[n]) for n in range(M + 1)], [model_p(pre[n]) for n in range(M + 1)])
        _explore(box, np.array(tokens), {}, w, law)
    return law


def check_ancestral(law, model_q, T, tol=1e-10):
    """The emitted sequence has the law of ancestral sampling from the
    verifier: given an emitted prefix x that the sequence continues past,
    the next token is distributed as softmax(model_q(x) / T)."""
    total = sum(law.values())
    assert abs(total - 1.0) < tol, total
    depth = max(len(s) for s in law)
    for k in range(depth):
        joint = {}
        for s, pr in law.items():
            if len(s) >= k + 1:
                x = s[:k]
                if x not in joint:
                    joint[x] = np.zeros(len(model_q(x)))
                joint[x][s[k]] += pr
        for x, row in joint.items():
            mass = row.sum()
            if mass > 1e-9:
                want = softmax(np.asarray(model_q(x), np.float64) / T)
                assert np.allclose(row / mass, want, atol=tol / mass, rtol=0), (k, x, row / mass, want)
