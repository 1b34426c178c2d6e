"""The synthetic inputs follow their stated recipe (CPU, reduced sizes).

Each workload is base logits ~ N(0, sigma_p^2), draft = base, target = base +
N(0, sigma_q^2), then a per-workload twist; drafts are drawn from the stored
draft logits at temperature T (argmax when T <= 0); uniforms are U[0, 1).
"""
import numpy as np
import torch

import synth
from synth.workloads import EAGLE16_PARENT


def _arr(t):
    return t.float().numpy()


def test_uniforms_and_token_ranges():
    for name, over in (("tiny", {}), ("small", {"B": 16, "V": 4096}), ("mixed", {"B": 24, "V": 4096}),
                       ("headline", {"B": 6, "V": 4096}), ("stress", {"B": 32, "V": 2048})):
        w = synth.make_workload(name, seed=1, **over)
        u = w.uniforms.numpy()
        assert u.shape == (w.B, w.N + 1) and (u >= 0).all() and (u < 1).all()
        d = w.draft_tokens.numpy()
        assert d.shape == (w.B, w.N) and (d >= 0).all() and (d < w.V).all()
        assert tuple(w.target.shape) == (w.B, w.N + 1, w.V) and tuple(w.draft.shape) == (w.B, w.N, w.V)


def test_greedy_sequences_draft_the_argmax():
    """mixed: temperatures come from {0, 0.7, 1}; at T = 0 the draft token is
    the argmax of the stored draft row."""
    w = synth.make_workload("mixed", seed=2, B=48, V=4096)
    T = w.temperature.numpy()
    assert set(np.unique(T)).issubset({0.0, np.float32(0.7), 1.0}) and (T == 0).any() and (T > 0).any()
    z = _arr(w.draft)
    d = w.draft_tokens.numpy()
    for b in np.nonzero(T == 0)[0]:
        assert (d[b] == z[b].argmax(axis=-1)).all()


def test_small_spikes_one_token_in_a_tenth_of_the_rows():
    """small: about 10 % of verifier rows (positions with a draft row) carry a
    +8 spike over the draft's logits at one token; the rest differ by noise of
    scale 0.5 only."""
    w = synth.make_workload("small", seed=3, B=64, V=4096)
    diff = _arr(w.target)[:, :w.N, :] - _arr(w.draft)
    spiked = (diff.max(axis=-1) > 5.0)
    frac = spiked.mean()
    assert 0.04 < frac < 0.18, frac
    assert (np.abs(diff[~spiked]) < 4.0).all()


def test_headline_zipf_prior_on_odd_sequences():
    """headline: odd sequences add -1.1 ln(token + 1) to both rows, so their
    mean logit falls with the token id; even sequences show no such trend."""
    w = synth.make_workload("headline", seed=4, B=8, V=8192)
    z = _arr(w.draft)
    lo, hi = slice(0, 256), slice(4096, 8192)
    for b in range(w.B):
        gap = z[b][:, lo].mean() - z[b][:, hi].mean()
        if b % 2:
            assert gap > 3.0, (b, gap)
        else:
            assert abs(gap) < 1.0, (b, gap)


def test_stress_forces_tokens_the_verifier_rules_out():
    """stress: about 5 % of draft positions are forced to a token whose
    verifier logit is set to -30."""
    w = synth.make_workload("stress", seed=5, B=128, V=2048)
    zt = _arr(w.target)
    d = w.draft_tokens.numpy()
    b, i = np.meshgrid(np.arange(w.B), np.arange(w.N), indexing="ij")
    forced = zt[b, i, d] == -30.0
    assert 0.02 < forced.mean() < 0.09, forced.mean()


def test_tree_topologies_and_greedy_children():
    """Random trees: parent[n] in [max(0, n-3), n-1] and parent[0] = -1; the
    bench tree is the fixed 16-node shape; a greedy tree's children all carry
    the argmax of their parent's draft row."""
    w = synth.make_tree_workload("tree_mixed", seed=6, B=24, V=2048)
    par = w.parent.numpy()
    n = np.arange(1, w.M + 1)
    assert (par[:, 0] == -1).all()
    assert ((par[:, 1:] >= np.maximum(0, n - 3)) & (par[:, 1:] <= n - 1)).all()
    T = w.temperature.numpy()
    assert (T == 0).any()
    zd = _arr(w.draft)
    tok = w.tokens.numpy()
    for b in np.nonzero(T == 0)[0]:
        for c in range(1, w.M + 1):
            assert tok[b, c] == zd[b, par[b, c]].argmax()
    fixed = synth.make_tree_workload("tree", seed=0, B=2, V=1024)
    assert fixed.parent.numpy().tolist() == [EAGLE16_PARENT] * 2


def test_fused_draft_model_reads_the_first_features():
    """fused: the draft head is the verifier head's first Kd features scaled by
    sqrt(Kt/Kd) (rounded to bf16); greedy drafts are the argmax of the draft
    product."""
    w = synth.make_fused_workload("fused_mixed", seed=7, B=6)
    wt, wd = w.target_weight.float(), w.draft_weight.float()
    want = (wt[:, :w.Kd] * (w.Kt / w.Kd) ** 0.5).to(torch.bfloat16).float()
    assert torch.equal(wd, want)
    T = w.temperature.numpy()
    zd = (w.draft_hidden.float() @ wd.T).view(w.B, w.N, w.V).numpy()
    d = w.draft_tokens.numpy()
    for b in np.nonzero(T <= 0)[0]:
        assert (d[b] == zd[b].argmax(axis=-1)).all()
