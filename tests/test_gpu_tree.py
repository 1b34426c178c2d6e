"""Tree verification on the GPU against the float64 tree oracle (needs a GB300).

Every call goes through the C ABI (spec_verify_tree_run).  Decisions taken
against a residual (siblings after a rejection, tokens drawn from such a
residual) are compared outside a band that grows with the number of
residual steps; everything else must match exactly.
"""
import os

import numpy as np
import pytest
import torch

import parity
import synth
import speculative_decoding_verification_49_gb300 as sv

pytestmark = pytest.mark.gpu

THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_verification_49_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _ctx(w):
    return sv.SpecVerify(w.B, w.M, w.V, w.dtype)


def _check(w, ctx=None, greedy=None, seqs=None):
    ctx = ctx or _ctx(w)
    gpu = parity.run_gpu_tree(ctx, w, greedy=greedy, seqs=seqs)
    orc = parity.run_oracle_tree(w, seqs=seqs, threads=THREADS, greedy=greedy)
    rep = parity.compare_tree(w, gpu, orc, seqs=seqs)
    print(w.name, rep)
    assert rep["band_mismatch"] <= max(1, rep["sequences"] // 50)
    assert ctx.status() == sv.SV_OK
    return rep, gpu


@pytest.mark.parametrize("name,seed,over", [
    ("tree_small", 0, {}), ("tree_small", 1, {}), ("tree_small", 2, {"B": 40}),
    ("tree_mixed", 0, {}), ("tree_mixed", 1, {}),
    ("tree", 0, {"B": 6}),
    # at least a wave of nodes (660 and 1260): kernel A runs one CTA per logit row
    ("tree_small", 3, {"B": 60}), ("tree_mixed", 2, {"B": 60}),
])
def test_tree_parity(name, seed, over):
    w = synth.make_tree_workload(name, seed=seed, device="cuda", **over)
    rep, _ = _check(w)
    assert rep["exact"] >= rep["sequences"] - rep["band_sequences"]


def test_tree_full_size_sampled():
    """The batch the benchmark times (64 trees of 16 nodes, V = 151936 bf16);
    the oracle checks a spread of its trees."""
    w = synth.make_tree_workload("tree", seed=0, device="cuda")
    seqs = np.array([0, 1, 2, 3, 17, 31, 32, 47, 62, 63])
    _check(w, seqs=seqs)


def test_tree_wide_siblings_exercise_many_residual_steps():
    """A star: 12 children of the root drawn from a draft far from the
    verifier, so that most walks reject several siblings in a row."""
    w = synth.make_tree_workload("tree_small", seed=3, device="cuda", B=24, M=12, sigma_q=3.0)
    w.parent[:] = 0
    w.parent[:, 0] = -1
    g = torch.Generator(device="cuda").manual_seed(3)
    z = w.draft[:, 0].float()
    for n in range(1, 13):
        gum = -torch.log(torch.empty_like(z).exponential_(generator=g))
        w.tokens[:, n] = torch.argmax(z + gum, dim=-1).to(torch.int32)
    rep, gpu = _check(w)
    assert rep["sibling_tests"] >= 24


@pytest.mark.parametrize("name,over,seqs", [
    # one CTA per tree (80 trees), 18 ring tiles a row
    ("tree_small", {"B": 80, "M": 12, "V": 36864}, None),
    # the benchmark's rows, two CTAs per tree (64 trees), 19-20 ring tiles a CTA
    ("tree", {"M": 12, "topology": "random"}, [0, 5, 9, 21, 33, 40, 52, 63]),
])
def test_tree_wide_siblings_at_long_rows(name, over, seqs):
    """Stars of 12 children with a draft far from the verifier, at row
    lengths where every consumer group of the walk streams six or more ring
    tiles per pass: several rejections in a row at one node, each a full
    pass over its row pair through the same ring stages."""
    w = synth.make_tree_workload(name, seed=13, device="cuda", sigma_q=3.0, **over)
    w.parent[:] = 0
    w.parent[:, 0] = -1
    g = torch.Generator(device="cuda").manual_seed(13)
    z = w.draft[:, 0].float()
    for n in range(1, w.M + 1):
        gum = -torch.log(torch.empty_like(z).exponential_(generator=g))
        w.tokens[:, n] = torch.argmax(z + gum, dim=-1).to(torch.int32)
    rep, gpu = _check(w, seqs=None if seqs is None else np.array(seqs))
    print(name, rep)
    assert rep["k_max"] >= 3  # three or more rejections at one node
    assert rep["sibling_tests"] >= rep["sequences"]


def test_tree_all_greedy_without_draft_logits():
    w = synth.make_tree_workload("tree_mixed", seed=2, device="cuda")
    rep, _ = _check(w, greedy=True)
    assert rep["exact"] == rep["sequences"]


def test_chain_shaped_tree_equals_the_chain_verify():
    """Both GPU paths on the same data: a chain of N nodes below the root."""
    cw = synth.make_workload("small", seed=5, device="cuda", B=10, N=5)
    B, N, V = cw.B, cw.N, cw.V
    tw = synth.TreeWorkload("chain", B, N, V, cw.dtype, cw.target.contiguous(),
                            torch.cat([cw.draft, cw.draft[:, :1]], dim=1).contiguous(),
                            torch.arange(-1, N, dtype=torch.int32, device="cuda").repeat(B, 1).contiguous(),
                            torch.cat([torch.zeros((B, 1), dtype=torch.int32, device="cuda"), cw.draft_tokens],
                                      dim=1).contiguous(),
                            torch.cat([cw.uniforms[:, N:], cw.uniforms[:, :N]], dim=1).contiguous(),
                            cw.temperature)
    ctx = sv.SpecVerify(B, N, V, cw.dtype)
    out_c, nacc_c = ctx.run(cw.target, cw.draft, cw.draft_tokens, cw.uniforms, cw.temperature)
    out_t, path_t, nacc_t = ctx.tree_run(tw.target, tw.draft, tw.parent, tw.tokens, tw.uniforms, tw.temperature)
    torch.cuda.synchronize()
    assert torch.equal(nacc_c, nacc_t)
    assert torch.equal(out_c, out_t)
    for b in range(B):
        a = int(nacc_t[b])
        assert path_t[b, :a].tolist() == list(range(1, a + 1))


def test_tree_invalid_inputs():
    w = synth.make_tree_workload("tree_small", seed=6, device="cuda", B=6)
    w.parent[0, 3] = 3                    # a node that is its own parent
    w.tokens[1, 2] = w.V                  # bad token
    internal = w.internal()
    n_int = int(torch.nonzero(internal[2])[0])
    w.draft[2, n_int, 7] = float("nan")   # a draft row that is read
    n_leaf = int(torch.nonzero(~internal[3])[0])
    w.draft[3, n_leaf, :] = float("nan")  # a leaf's draft row is not read
    w.temperature[4] = float("nan")
    ctx = _ctx(w)
    gpu = parity.run_gpu_tree(ctx, w)
    for b in (0, 1, 2, 4):
        assert gpu["num_accepted"][b] == -1 and (gpu["out_tokens"][b] == -1).all()
        assert (gpu["path_nodes"][b] == -1).all()
    assert gpu["num_accepted"][3] >= 0 and gpu["num_accepted"][5] >= 0
    assert ctx.status() == sv.SV_ERR_BAD_TREE
    assert ctx.status() == sv.SV_OK
    orc = parity.run_oracle_tree(w)
    assert (orc["seq_status"][[0, 1, 2, 4]] != 0).all() and orc["seq_status"][3] == 0
    assert np.array_equal(orc["num_accepted"][[0, 1, 2, 4]], gpu["num_accepted"][[0, 1, 2, 4]])
    w.parent[0, 3] = 0
    w.tokens[1, 2] = 0
    # the context is usable afterwards
    _check(synth.make_tree_workload("tree_small", seed=7, device="cuda", B=6), ctx=ctx)


@pytest.mark.parametrize("B", [6, 64])
def test_tree_invalid_trees_repeatedly_in_clustered_walks(B):
    """Invalid trees (a NaN temperature, a bad token) beside valid ones, 25
    calls in a row on one context, with the walk split over clusters of 4 CTAs
    (B = 6) and of 2 (B = 64): every call returns -1 rows for the invalid trees
    and the same tokens for the valid ones.  Every CTA of a walk cluster reads
    the sequence's error word before the leader resets it for the next call."""
    w = synth.make_tree_workload("tree_small", seed=11, device="cuda", B=B)
    bad_t = list(range(0, B, 3))
    bad_d = [b for b in range(1, B, 3)]
    for b in bad_t:
        w.temperature[b] = float("nan")
    for b in bad_d:
        w.tokens[b, 1] = w.V
    bad = sorted(bad_t + bad_d)
    good = [b for b in range(B) if b not in bad]
    ctx = _ctx(w)
    first = None
    for _ in range(25):
        gpu = parity.run_gpu_tree(ctx, w, stats=False)
        assert (gpu["num_accepted"][bad] == -1).all() and (gpu["out_tokens"][bad] == -1).all()
        assert (gpu["num_accepted"][good] >= 0).all()
        assert ctx.status() != sv.SV_OK
        if first is None:
            first = gpu
        else:
            assert np.array_equal(gpu["out_tokens"], first["out_tokens"])
            assert np.array_equal(gpu["path_nodes"], first["path_nodes"])


def _random_trees(n=6, seed=55):
    """Seeded random tree batches: bf16 or f32, V at any 16-byte multiple up to
    9600, 1-100 nodes below the root (random parents in the last three
    nodes), B 1-30, one temperature or a per-sequence mix with greedy trees."""
    rng = np.random.default_rng(seed)
    out = []
    for k in range(n):
        dtype = "bf16" if rng.random() < 0.5 else "f32"
        V = int(rng.integers(1, 1201)) * (8 if dtype == "bf16" else 4)
        M = int(rng.integers(1, 101))
        B = int(rng.integers(1, 31))
        T = (0.0, 0.7, 1.0) if rng.random() < 0.5 else float(rng.choice([0.5, 1.0, 1.5]))
        out.append((k, dtype, V, M, B, T))
    return out


@pytest.mark.parametrize("k,dtype,V,M,B,T", _random_trees())
def test_tree_random_shapes(k, dtype, V, M, B, T):
    w = synth.make_tree_workload("tree_small", seed=300 + k, device="cuda", B=B, M=M, V=V, dtype=dtype, T=T)
    _check(w)


def test_tree_with_the_most_nodes():
    """1024 nodes per tree (M = 1023, the largest tree the walk holds in shared
    memory), random topologies, against the tree oracle."""
    w = synth.make_tree_workload("tree_small", seed=21, device="cuda", B=3, M=1023, V=256)
    _check(w)


def test_tree_root_only_and_ragged_vocabularies():
    for V, dtype in [(1000, "f32"), (4104, "bf16"), (16, "f32")]:
        w = synth.make_tree_workload("tree_small", seed=8, device="cuda", B=5, M=0, V=V, dtype=dtype)
        rep, gpu = _check(w)
        assert (gpu["num_accepted"] == 0).all()
        w = synth.make_tree_workload("tree_small", seed=9, device="cuda", B=5, M=6, V=V, dtype=dtype)
        _check(w)


def test_tree_counts_path_lengths():
    w = synth.make_tree_workload("tree_small", seed=10, device="cuda", B=20)
    ctx = _ctx(w)
    ctx.acceptance_counts(reset=True)
    _, gpu = _check(w, ctx=ctx)
    counts = ctx.acceptance_counts()
    want = np.bincount(gpu["num_accepted"], minlength=w.M + 1)
    assert counts[: w.M + 1] == want.tolist() and counts[w.M + 1] == 0
