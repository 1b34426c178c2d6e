"""Statistical checks of the oracle (CPU only), as the pages prescribe them:
  * chi-square of the emitted tokens against direct sampling from the
    verifier, 50 000 tokens, p > 0.05 (page 1, Step 5 and exercise 1);
  * mean tokens per verify call against (1 - a^(N+1)) / (1 - a),
    a = sum_k min(p, q) (page 1, "What determines speedup" and exercise 2);
  * acceptance rate falls as KL(draft || verifier) grows (page 1, Step 4).
Drafts are drawn from p with the Gumbel-max trick, uniforms from numpy.
"""
import math

import numpy as np
from scipy.special import softmax
from scipy.stats import chisquare

import oracle


def _fixed_batch(zq, zp, B):
    return (np.broadcast_to(zq, (B,) + zq.shape).copy(),
            np.broadcast_to(zp, (B,) + zp.shape).copy())


def _draw_drafts(rng, zp, B, T=1.0):
    N, V = zp.shape
    g = rng.gumbel(size=(B, N, V))
    return np.argmax(zp[None] / T + g, axis=2).astype(np.int32)


def test_chi_square_emitted_tokens_match_verifier():
    orc = oracle.Oracle()
    pvals = []
    for seed in range(5):
        rng = np.random.default_rng(100 + seed)
        N, V, B = 3, 16, 50_000
        zq = rng.normal(0, 1.5, (N + 1, V))
        zp = zq[:N] + rng.normal(0, 1.0, (N, V))
        d = _draw_drafts(rng, zp, B)
        u = rng.random((B, N + 1))
        ZQ, ZP = _fixed_batch(zq, zp, B)
        r = orc.verify(ZQ, ZP, d, u, np.ones(B), dtype="f64", diagnostics=False, threads=4)
        first = r["out_tokens"][:, 0]
        q0 = softmax(zq[0])
        obs = np.bincount(first, minlength=V)
        pvals.append(chisquare(obs, q0 * B).pvalue)
        # second emitted token, among rounds that emitted at least two
        keep = r["num_accepted"] >= 1
        second = r["out_tokens"][keep, 1]
        obs2 = np.bincount(second, minlength=V)
        pvals.append(chisquare(obs2, softmax(zq[1]) * keep.sum()).pvalue)
    print("chi-square p-values:", ["%.3f" % p for p in pvals])
    assert min(pvals) > 0.001, pvals
    assert np.mean(np.array(pvals) > 0.05) >= 0.8, pvals


def test_mean_tokens_per_call_matches_closed_form():
    orc = oracle.Oracle()
    rng = np.random.default_rng(7)
    N, V, B = 4, 6, 200_000
    zq1 = rng.normal(0, 1.0, V)
    zp1 = rng.normal(0, 1.0, V)
    q, p = softmax(zq1), softmax(zp1)
    alpha = float(np.minimum(p, q).sum())
    zq = np.stack([zq1] * (N + 1))
    zp = np.stack([zp1] * N)
    d = _draw_drafts(rng, zp, B)
    u = rng.random((B, N + 1))
    ZQ, ZP = _fixed_batch(zq, zp, B)
    r = orc.verify(ZQ, ZP, d, u, np.ones(B), dtype="f64", diagnostics=False, threads=4)
    emitted = r["num_accepted"] + 1
    closed = (1 - alpha ** (N + 1)) / (1 - alpha)
    se = emitted.std() / math.sqrt(B)
    print(f"alpha={alpha:.4f} mean={emitted.mean():.5f} closed={closed:.5f} se={se:.5f}")
    assert abs(emitted.mean() - closed) < 4 * se
    # per-position acceptance rate equals alpha
    acc0 = (r["num_accepted"] >= 1).mean()
    assert abs(acc0 - alpha) < 4 * math.sqrt(alpha * (1 - alpha) / B)


def test_acceptance_falls_as_kl_grows():
    orc = oracle.Oracle()
    rng = np.random.default_rng(12)
    N, V, B = 4, 32, 10_000
    zq1 = rng.normal(0, 2.0, V)
    noise = rng.normal(0, 1.0, V)
    rates, kls = [], []
    for lam in (0.0, 0.5, 1.0, 2.0, 4.0):
        zp1 = zq1 + lam * noise
        q, p = softmax(zq1), softmax(zp1)
        kls.append(float(np.sum(p * (np.log(p) - np.log(q)))))
        zq = np.stack([zq1] * (N + 1))
        zp = np.stack([zp1] * N)
        d = _draw_drafts(rng, zp, B)
        u = rng.random((B, N + 1))
        ZQ, ZP = _fixed_batch(zq, zp, B)
        r = orc.verify(ZQ, ZP, d, u, np.ones(B), dtype="f64", diagnostics=False, threads=4)
        # acceptance rate over all evaluated accept tests
        acc = r["num_accepted"]
        tests = np.minimum(acc + 1, N).sum()
        rates.append(acc.sum() / tests)
    print("KL:", kls, "acceptance:", rates)
    assert all(np.diff(kls) > 0)
    assert all(np.diff(rates) < 0)
    assert rates[0] == 1.0
