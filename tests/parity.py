"""GPU-vs-oracle comparison used by the -m gpu tests, the smoke check and the
benchmark's self-check.

Decision rule: tokens and accept counts must match the float64 oracle
exactly, except in sequences where one of the oracle's decisions had a margin
below BAND (|u - ratio| for an accept test, the distance of u to the chosen
token's CDF edge for the final sample).  Those are counted and must stay
below 1e-4 of all decisions.  Normalised probabilities (q(d), p(d)) and the
normaliser S must agree to 1e-5 relative for float32 logits and 2e-3 for
bf16 logits.  The ratio each of the GPU's accept tests compared its uniform
with must lie within BAND of the oracle's (on min(1, ratio)), which is what
makes the band sufficient: outside it, a decision cannot flip.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle

BAND = 1e-6
PROB_RTOL = {"f32": 1e-5, "bf16": 2e-3}


def run_gpu(ctx, w, debug=True, greedy=None, seqs=None):
    greedy = w.greedy if greedy is None else greedy
    dbg = ctx.debug_buffers(w.B, w.N, device=w.target.device) if debug else None
    out, nacc = ctx.run(w.target, None if greedy else w.draft, w.draft_tokens,
                        None if greedy else w.uniforms, None if greedy else w.temperature,
                        greedy=greedy, debug=dbg)
    torch.cuda.synchronize()
    res = {"out_tokens": out.cpu().numpy(), "num_accepted": nacc.cpu().numpy()}
    if dbg:
        res.update({k: v.cpu().numpy() for k, v in dbg.items()})
    if seqs is not None:
        res = {k: v[seqs] for k, v in res.items()}
    return res


def run_oracle(w, seqs=None, threads=8, greedy=None):
    greedy = w.greedy if greedy is None else greedy
    sel = (lambda t: t) if seqs is None else (lambda t: t[torch.as_tensor(seqs, device=t.device)])
    return oracle.verify(sel(w.target), None if greedy else sel(w.draft), sel(w.draft_tokens),
                         sel(w.uniforms).double(), None if greedy else sel(w.temperature).double(),
                         greedy=greedy, dtype=w.dtype, threads=threads)


def compare(w, gpu, orc, check_probs=True):
    """Returns a report dict; raises AssertionError on a mismatch outside the
    margin band or a probability outside tolerance."""
    out_g, acc_g = gpu["out_tokens"], gpu["num_accepted"]
    out_o, acc_o = orc["out_tokens"], orc["num_accepted"]
    B = out_o.shape[0]
    am, sm = orc["accept_margin"], orc["sample_margin"]
    decisions = int(np.isfinite(am).sum() + np.isinf(am).sum() + (~np.isnan(sm)).sum())
    band_dec = int((am < BAND).sum() + (sm < BAND).sum())
    in_band = (np.nan_to_num(am, nan=np.inf) < BAND).any(axis=1) | (np.nan_to_num(sm, nan=np.inf) < BAND)
    same = (out_g == out_o).all(axis=1) & (acc_g == acc_o)
    bad = np.nonzero(~same & ~in_band)[0]
    assert bad.size == 0, (
        f"{bad.size} sequences differ outside the margin band, first b={bad[0]}: "
        f"gpu {out_g[bad[0]].tolist()}/{acc_g[bad[0]]} oracle {out_o[bad[0]].tolist()}/{acc_o[bad[0]]} "
        f"margins {am[bad[0]].tolist()} {sm[bad[0]]}")
    rep = {"sequences": B, "exact": int(same.sum()), "band_sequences": int(in_band.sum()),
           "band_mismatch": int((~same & in_band).sum()), "decisions": decisions,
           "band_decisions": band_dec}
    if check_probs and "q_at_draft" in gpu:
        tol = PROB_RTOL[w.dtype]
        ok = (orc["seq_status"] == 0)[:, None] & np.isfinite(orc["q_at_d"])
        qrel = np.abs(gpu["q_at_draft"] - orc["q_at_d"]) / np.maximum(orc["q_at_d"], 1e-300)
        prel = np.abs(gpu["p_at_draft"] - orc["p_at_d"]) / np.maximum(orc["p_at_d"], 1e-300)
        # probabilities below float32's normal range are compared absolutely
        tiny_q = orc["q_at_d"] < 1e-30
        tiny_p = orc["p_at_d"] < 1e-30
        qrel = np.where(tiny_q, np.abs(gpu["q_at_draft"] - orc["q_at_d"]) / 1e-30, qrel)
        prel = np.where(tiny_p, np.abs(gpu["p_at_draft"] - orc["p_at_d"]) / 1e-30, prel)
        q_max = float(np.max(qrel[ok], initial=0.0))
        p_max = float(np.max(prel[ok], initial=0.0))
        assert q_max <= tol, f"q(d) relative error {q_max:.3g} > {tol}"
        assert p_max <= tol, f"p(d) relative error {p_max:.3g} > {tol}"
        ts_ok = (orc["seq_status"] == 0)[:, None] & np.isfinite(orc["tstats"][..., 1])
        m_diff = np.abs(gpu["target_row_stats"][..., 0] - orc["tstats"][..., 0])[ts_ok]
        assert (m_diff == 0).all(), "row max differs"
        s_rel = (np.abs(gpu["target_row_stats"][..., 1] - orc["tstats"][..., 1]) / orc["tstats"][..., 1])[ts_ok]
        s_max = float(np.max(s_rel, initial=0.0))
        assert s_max <= tol, f"S relative error {s_max:.3g} > {tol}"
        ds_ok = (orc["seq_status"] == 0)[:, None] & np.isfinite(orc["dstats"][..., 1])
        d_rel = (np.abs(gpu["draft_row_stats"][..., 1] - orc["dstats"][..., 1]) / orc["dstats"][..., 1])[ds_ok]
        d_max = float(np.max(d_rel, initial=0.0))
        assert d_max <= tol, f"draft S relative error {d_max:.3g} > {tol}"
        # accept-test ratio error, where both sides evaluated it
        ratio_o = orc["q_at_d"] / np.where(orc["p_at_d"] > 0, orc["p_at_d"], np.nan)
        ratio_g = gpu["q_at_draft"].astype(np.float64) / np.where(gpu["p_at_draft"] > 0, gpu["p_at_draft"], np.nan)
        rr = np.abs(np.minimum(ratio_g, 1.0) - np.minimum(ratio_o, 1.0))[ok]
        rep.update(q_rel_max=q_max, p_rel_max=p_max, S_rel_max=max(s_max, d_max),
                   ratio_abs_max=float(np.nanmax(rr, initial=0.0)))
    if "ratio_at_draft" in gpu and "ratio_at_d" in orc:
        err = decision_ratio_error(gpu["ratio_at_draft"], orc["ratio_at_d"], orc["seq_status"])
        assert err <= BAND, f"decision ratio differs from the oracle's by {err:.3g} > {BAND}"
        rep["decision_ratio_err_max"] = err
    return rep


def decision_ratio_error(ratio_gpu, ratio_orc, seq_status, rows=None):
    """max |min(1, ratio_gpu) - min(1, ratio_orc)| over the accept tests the
    oracle made in valid sequences (the GPU makes every one of them too)."""
    ro = np.asarray(ratio_orc, np.float64)
    rg = np.asarray(ratio_gpu, np.float64)
    ev = (np.asarray(seq_status) == 0)[:, None] & ~np.isnan(ro)
    if rows is not None:
        ev &= np.asarray(rows)[:, None]
    assert not np.isnan(rg[ev]).any(), "the GPU left an accept test the oracle made without a ratio"
    return float(np.max(np.abs(np.minimum(rg, 1.0) - np.minimum(ro, 1.0))[ev], initial=0.0))


# ---- tree verification ----------------------------------------------------------

# Band of a tree decision taken against a residual (a sibling after k >= 1
# rejections, or a token drawn from such a residual): r_k = (q - c p)+ / Z is
# evaluated from float32 probabilities, and q - c p loses relative precision
# where the two are close, so these decisions are compared outside a band of
# k * TREE_BAND_PER_STEP.  Measured over every tree test (316 sibling tests):
# the ratio such a test compares u with differs from the
# oracle's by at most 5.8e-7 per rejection (1.16e-6 at k = 2); the band is
# about four times that, and each test checks that its ratios stay inside it.
TREE_BAND_PER_STEP = 2.5e-6


def run_gpu_tree(ctx, w, greedy=None, seqs=None, stats=True):
    greedy = w.greedy if greedy is None else greedy
    st = None
    if stats:
        st = {k: torch.full((w.B, w.M + 1, 2), float("nan"), device=w.target.device)
              for k in ("target_row_stats", "draft_row_stats")}
        st["ratio_at_node"] = torch.full((w.B, w.M + 1), float("nan"), device=w.target.device)
    out, path, nacc = ctx.tree_run(w.target, None if greedy else w.draft, w.parent, w.tokens,
                                   None if greedy else w.uniforms, None if greedy else w.temperature,
                                   greedy=greedy, stats=st)
    torch.cuda.synchronize()
    res = {"out_tokens": out.cpu().numpy(), "path_nodes": path.cpu().numpy(), "num_accepted": nacc.cpu().numpy()}
    if st:
        res.update({k: v.cpu().numpy() for k, v in st.items()})
    if seqs is not None:
        res = {k: v[seqs] for k, v in res.items()}
    return res


def run_oracle_tree(w, seqs=None, threads=8, greedy=None):
    greedy = w.greedy if greedy is None else greedy
    sel = (lambda t: t) if seqs is None else (lambda t: t[torch.as_tensor(seqs, device=t.device)])
    return oracle.tree_verify(sel(w.target), None if greedy else sel(w.draft), sel(w.parent), sel(w.tokens),
                              sel(w.uniforms).double(), None if greedy else sel(w.temperature).double(),
                              greedy=greedy, dtype=w.dtype, threads=threads)


def _sibling_steps(parent, margin):
    """Per tested node: how many siblings were rejected before it (k)."""
    k = np.zeros(margin.shape, np.int64)
    for b in range(margin.shape[0]):
        seen = {}
        for c in range(1, margin.shape[1]):
            if not np.isnan(margin[b, c]):
                p = int(parent[b, c])
                k[b, c] = seen.get(p, 0)
                seen[p] = k[b, c] + 1
    return k


def compare_tree(w, gpu, orc, seqs=None, check_stats=True):
    """Report dict; AssertionError on a mismatch outside the margin bands or a
    normaliser outside tolerance."""
    parent = w.parent.cpu().numpy() if seqs is None else w.parent.cpu().numpy()[seqs]
    am, sm = orc["accept_margin"], orc["sample_margin"]
    k = _sibling_steps(parent, am)
    band = np.where(k == 0, BAND, TREE_BAND_PER_STEP * np.maximum(k, 1))
    in_band_acc = (np.nan_to_num(am, nan=np.inf) < band).any(axis=1)
    # the final draw comes from a residual when the last tested node was rejected
    kmax = np.where(np.isnan(am), -1, k).max(axis=1, initial=-1)
    sband = np.where(kmax >= 0, TREE_BAND_PER_STEP * (kmax + 1), BAND)
    in_band = in_band_acc | (np.nan_to_num(sm, nan=np.inf) < sband)
    same = ((gpu["out_tokens"] == orc["out_tokens"]).all(axis=1) & (gpu["path_nodes"] == orc["path_nodes"]).all(axis=1)
            & (gpu["num_accepted"] == orc["num_accepted"]))
    bad = np.nonzero(~same & ~in_band)[0]
    assert bad.size == 0, (
        f"{bad.size} trees differ outside the margin band, first b={bad[0]}: gpu {gpu['out_tokens'][bad[0]].tolist()} "
        f"{gpu['path_nodes'][bad[0]].tolist()} oracle {orc['out_tokens'][bad[0]].tolist()} "
        f"{orc['path_nodes'][bad[0]].tolist()} margins {am[bad[0]].tolist()} {sm[bad[0]]}")
    tested = int((~np.isnan(am)).sum())
    rep = {"sequences": int(len(same)), "exact": int(same.sum()), "band_sequences": int(in_band.sum()),
           "band_mismatch": int((~same & in_band).sum()), "tests": tested,
           "sibling_tests": int(((k > 0) & ~np.isnan(am)).sum())}
    if "ratio_at_node" in gpu and "ratio_at" in orc:
        # the ratio each tested child's uniform was compared with, in trees
        # that took the oracle's path (there both tested the same children):
        # before any rejection at the parent (k = 0) and against a residual
        ro, rg = orc["ratio_at"], gpu["ratio_at_node"].astype(np.float64)
        ev = same[:, None] & (orc["seq_status"] == 0)[:, None] & ~np.isnan(ro)
        assert not np.isnan(rg[ev]).any(), "the walk left a tested child without a ratio"
        assert np.isnan(rg[same & (orc["seq_status"] == 0)][np.isnan(ro[same & (orc["seq_status"] == 0)])]).all(), \
            "the walk reports a ratio for a child the oracle did not test"
        err = np.abs(np.minimum(rg, 1.0) - np.minimum(ro, 1.0))
        e0 = float(np.max(err[ev & (k == 0)], initial=0.0))
        assert e0 <= BAND, f"first-child decision ratio differs from the oracle's by {e0:.3g} > {BAND}"
        rep["ratio_err_first"] = e0
        rep["k_max"] = int(np.max(np.where(ev, k, 0), initial=0))
        rep["ratio_err_sibling"] = float(np.max(err[ev & (k > 0)], initial=0.0))
        rep["ratio_err_sibling_per_step"] = float(np.max((err / np.maximum(k, 1))[ev & (k > 0)], initial=0.0))
        assert rep["ratio_err_sibling_per_step"] <= TREE_BAND_PER_STEP, \
            f"sibling decision ratio differs by {rep['ratio_err_sibling_per_step']:.3g} per rejection"
    if check_stats and "target_row_stats" in gpu:
        tol = PROB_RTOL[w.dtype]
        ok = (orc["seq_status"] == 0)[:, None] & np.isfinite(orc["tstats"][..., 1])
        assert (gpu["target_row_stats"][..., 0][ok] == orc["tstats"][..., 0][ok]).all(), "row max differs"
        s_rel = (np.abs(gpu["target_row_stats"][..., 1] - orc["tstats"][..., 1]) / orc["tstats"][..., 1])[ok]
        okd = (orc["seq_status"] == 0)[:, None] & np.isfinite(orc["dstats"][..., 1])
        d_rel = (np.abs(gpu["draft_row_stats"][..., 1] - orc["dstats"][..., 1]) / orc["dstats"][..., 1])[okd]
        s_max = float(max(np.max(s_rel, initial=0.0), np.max(d_rel, initial=0.0)))
        assert s_max <= tol, f"S relative error {s_max:.3g} > {tol}"
        rep["S_rel_max"] = s_max
    return rep


# ---- the fused LM-head path ----------------------------------------------------------

# The fused path decides on float32 logits accumulated on the tensor cores from
# bf16 products; the oracle on the float64 products.  A logit of the fused path
# differs from the float64 product by at most LOGIT_ERR_FACTOR * sqrt(K) 2^-24
# sum_j |h_j w_jk| (the LM-head tests measure at most 0.31 of that scale, and
# the fused tests' row maxima at most 0.17), so a row maximum by at most delta =
# that bound's largest value over the row, a normaliser S by a factor within
# exp(+-2 delta / T) on top of its own float32 evaluation (1e-5 relative), and
# a greedy argmax only where the two largest logits are within 2 delta.  The
# ratio an accept test compares u with differs from the oracle's by at most
# FUSED_BAND on min(1, ratio) (measured at most 2.2e-6 over every fused test),
# so decisions whose margin is below FUSED_BAND may differ.
LOGIT_ERR_FACTOR = 2.0
FUSED_BAND = 1e-5


def run_gpu_fused(ctx, w, greedy=None, seqs=None):
    greedy = w.greedy if greedy is None else greedy
    st = {"target_row_stats": torch.full((w.B, w.N + 1, 2), float("nan"), device=w.target_hidden.device),
          "draft_row_stats": torch.full((w.B, w.N, 2), float("nan"), device=w.target_hidden.device),
          "ratio_at_draft": torch.full((w.B, w.N), float("nan"), device=w.target_hidden.device)}
    out, nacc = ctx.run_fused(w.target_hidden, w.target_weight, None if greedy else w.draft_hidden,
                              None if greedy else w.draft_weight, w.draft_tokens,
                              None if greedy else w.uniforms, None if greedy else w.temperature,
                              greedy=greedy, stats=st)
    torch.cuda.synchronize()
    res = {"out_tokens": out.cpu().numpy(), "num_accepted": nacc.cpu().numpy()}
    res.update({k: v.cpu().numpy() for k, v in st.items()})
    if seqs is not None:
        res = {k: v[seqs] for k, v in res.items()}
    return res


def run_oracle_fused(w, seqs=None, threads=8, greedy=None):
    """Float64 logits (the plain product) of the selected sequences, then the
    verify oracle on them."""
    greedy = w.greedy if greedy is None else greedy
    B, N = w.B, w.N
    sel = np.arange(B) if seqs is None else np.asarray(seqs)
    rt = (sel[:, None] * (N + 1) + np.arange(N + 1)[None, :]).ravel()
    rd = (sel[:, None] * N + np.arange(N)[None, :]).ravel()
    th = w.target_hidden[torch.as_tensor(rt, device=w.target_hidden.device)]
    zt = oracle.lm_head_logits(th, w.target_weight).reshape(len(sel), N + 1, w.V)
    # bound on the float32 product's error per row: the largest of
    # LOGIT_ERR_FACTOR sqrt(K) 2^-24 sum_j |h_j w_jk| over the row
    mag = LOGIT_ERR_FACTOR * lm_head_error_scale(th, w.target_weight).max(axis=1).reshape(len(sel), N + 1)
    zd = None
    dmag = np.zeros((len(sel), N))
    if not greedy and N > 0:
        dh = w.draft_hidden[torch.as_tensor(rd, device=w.draft_hidden.device)]
        zd = oracle.lm_head_logits(dh, w.draft_weight).reshape(len(sel), N, w.V)
        dmag = LOGIT_ERR_FACTOR * lm_head_error_scale(dh, w.draft_weight).max(axis=1).reshape(len(sel), N)
    idx = torch.as_tensor(sel, device=w.draft_tokens.device)
    res = oracle.verify(zt, zd, w.draft_tokens[idx], w.uniforms[idx].double(),
                        None if greedy else w.temperature[idx].double(), greedy=greedy, dtype="f64", threads=threads)
    # greedy decisions: the gap between the two largest logits of each verifier row
    top2 = np.sort(zt, axis=-1)[..., -2:]
    res["top2_gap"] = top2[..., 1] - top2[..., 0]
    res["m_bound"] = mag
    res["dm_bound"] = dmag
    res["T"] = np.full(len(sel), np.inf) if greedy else w.temperature[idx].double().cpu().numpy()
    return res


def lm_head_error_scale(hidden, weight):
    """sqrt(K) * 2^-24 * sum_j |h_j w_jk| for every output (float64): the size of
    the rounding error of a float32 sum of K products with random signs."""
    h = np.abs(np.asarray(hidden.float().cpu().numpy() if hasattr(hidden, "float") else hidden, np.float64))
    wt = np.abs(np.asarray(weight.float().cpu().numpy() if hasattr(weight, "float") else weight, np.float64))
    return (h @ wt.T) * (math.sqrt(h.shape[1]) * 2.0 ** -24)


def compare_fused(w, gpu, orc, greedy=False):
    """Report dict of the fused path against the oracle on the float64
    products; AssertionError outside the bands and tolerances (checked after
    the report is printed)."""
    am, sm = orc["accept_margin"], orc["sample_margin"]
    in_band = (np.nan_to_num(am, nan=np.inf) < FUSED_BAND).any(axis=1) | (np.nan_to_num(sm, nan=np.inf) < FUSED_BAND)
    greedy_rows = (orc["tstats"][..., 1] != orc["tstats"][..., 1]).all(axis=1) if not greedy else np.ones(len(am), bool)
    in_band |= greedy_rows & (orc["top2_gap"] < 2.0 * orc["m_bound"]).any(axis=1)
    same = (gpu["out_tokens"] == orc["out_tokens"]).all(axis=1) & (gpu["num_accepted"] == orc["num_accepted"])
    bad = np.nonzero(~same & ~in_band)[0]
    ok = (orc["seq_status"] == 0)[:, None] & np.isfinite(orc["tstats"][..., 1])
    m_abs = np.abs(gpu["target_row_stats"][..., 0] - orc["tstats"][..., 0])
    m_err = float(np.max(m_abs[ok], initial=0.0))
    s_rel_all = np.abs(gpu["target_row_stats"][..., 1] - orc["tstats"][..., 1]) / orc["tstats"][..., 1]
    s_rel = float(np.max(s_rel_all[ok], initial=0.0))
    okd = (orc["seq_status"] == 0)[:, None] & np.isfinite(orc["dstats"][..., 1])
    d_rel_all = np.abs(gpu["draft_row_stats"][..., 1] - orc["dstats"][..., 1]) / orc["dstats"][..., 1]
    d_rel = float(np.max(d_rel_all[okd], initial=0.0))
    dm_abs = np.abs(gpu["draft_row_stats"][..., 0] - orc["dstats"][..., 0])
    # tolerances derived from the logit error bound (see LOGIT_ERR_FACTOR)
    T = orc["T"][:, None]
    s_tol = np.expm1(2.0 * orc["m_bound"] / T) + 1e-5
    d_tol = np.expm1(2.0 * orc["dm_bound"] / T) + 1e-5
    okm = (orc["seq_status"] == 0)[:, None] & np.isfinite(orc["tstats"][..., 0])
    rep = {"sequences": int(len(same)), "exact": int(same.sum()), "band_sequences": int(in_band.sum()),
           "band_mismatch": int((~same & in_band).sum()), "m_abs_max": m_err, "S_rel_max": max(s_rel, d_rel)}
    if "ratio_at_draft" in gpu:
        ro, rg = orc["ratio_at_d"], gpu["ratio_at_draft"].astype(np.float64)
        ev = (orc["seq_status"] == 0)[:, None] & ~np.isnan(ro)
        assert not np.isnan(rg[ev]).any()
        err = np.abs(np.minimum(rg, 1.0) - np.minimum(ro, 1.0))[ev]
        rel = (np.abs(rg - ro) / np.where(ro > 0, ro, 1.0))[ev & np.isfinite(ro)]
        rep["ratio_err_max"] = float(np.max(err, initial=0.0))
        rep["ratio_rel_err_max"] = float(np.max(rel, initial=0.0))
    rep["m_err_over_bound"] = float(np.max((m_abs / orc["m_bound"])[okm], initial=0.0))
    rep["S_err_over_tol"] = float(max(np.max((s_rel_all / s_tol)[ok], initial=0.0),
                                      np.max((d_rel_all / d_tol)[okd], initial=0.0)))
    print("fused parity:", rep)
    assert bad.size == 0, (f"{bad.size} sequences differ outside the band, first {bad[0]}: gpu "
                           f"{gpu['out_tokens'][bad[0]].tolist()} oracle {orc['out_tokens'][bad[0]].tolist()} "
                           f"margins {am[bad[0]].tolist()} {sm[bad[0]]}")
    assert (m_abs[okm] <= orc["m_bound"][okm]).all(), f"row max beyond the logit error bound ({rep['m_err_over_bound']:.3g})"
    assert (dm_abs[okd] <= orc["dm_bound"][okd]).all(), "draft row max beyond the logit error bound"
    assert (s_rel_all[ok] <= s_tol[ok]).all() and (d_rel_all[okd] <= d_tol[okd]).all(), \
        f"normaliser beyond its tolerance ({rep['S_err_over_tol']:.3g} of it)"
    if "ratio_err_max" in rep:
        assert rep["ratio_err_max"] <= FUSED_BAND, f"decision ratio differs by {rep['ratio_err_max']:.3g} > {FUSED_BAND}"
    return rep
