"""The verify step fused into the LM-head products, against the float64
oracle on the float64 products (needs a GB300)."""
import dataclasses
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


def _check(w, greedy=None, seqs=None, ctx=None, keep=True):
    ctx = ctx or sv.SpecVerify(w.B, w.N, w.V, "f32")
    ctx.set_fused_logits(keep)
    gpu = parity.run_gpu_fused(ctx, w, greedy=greedy, seqs=seqs)
    orc = parity.run_oracle_fused(w, seqs=seqs, threads=THREADS, greedy=greedy)
    rep = parity.compare_fused(w, gpu, orc, greedy=bool(greedy))
    print(w.name, rep)
    assert rep["band_mismatch"] <= max(1, rep["sequences"] // 20)
    assert ctx.status() == sv.SV_OK
    return rep, gpu


@pytest.mark.parametrize("keep", [True, False], ids=["kept_logits", "recomputed_rows"])
@pytest.mark.parametrize("name,seed", [("fused_small", 0), ("fused_small", 1), ("fused_mixed", 0)])
def test_fused_parity(name, seed, keep):
    w = synth.make_fused_workload(name, seed=seed, device="cuda")
    _check(w, keep=keep)


@pytest.mark.parametrize("keep", [True, False], ids=["kept_logits", "recomputed_rows"])
@pytest.mark.parametrize("V,Kt,Kd", [(4104, 200, 72), (1000, 64, 8), (20, 520, 136)])
def test_fused_ragged_vocabulary_and_depth(V, Kt, Kd, keep):
    """A last vocabulary tile shorter than 256 columns, and K not a multiple of
    the 64-wide stage (the tensor maps fill the missing columns with zeros)."""
    w = synth.make_fused_workload("fused_small", seed=V, device="cuda", V=V, Kt=Kt, Kd=Kd)
    _check(w, keep=keep)


def _random_fused_shapes(n=6, seed=77):
    """Seeded random shapes: V any multiple of 4 up to 12000 (the float32
    context's rule; most leave a ragged last 32-column box for the tensor
    stores), verifier and draft hidden sizes multiples of 8 (not of the 64-wide
    stage; the draft's no larger than the verifier's), B 1-24, N 0-6, one
    temperature or a per-sequence mix with greedy sequences."""
    rng = np.random.default_rng(seed)
    out = []
    for k in range(n):
        V = int(rng.integers(1, 3001)) * 4
        Kt = int(rng.integers(2, 129)) * 8
        Kd = int(rng.integers(1, Kt // 8 + 1)) * 8  # the draft reads the first Kd hidden features
        B = int(rng.integers(1, 25))
        N = int(rng.integers(0, 7))
        T = (0.0, 0.7, 1.0) if rng.random() < 0.5 else float(rng.choice([0.5, 1.0, 1.5]))
        out.append((k, V, Kt, Kd, B, N, T))
    return out


@pytest.mark.parametrize("k,V,Kt,Kd,B,N,T", _random_fused_shapes())
def test_fused_random_shapes(k, V, Kt, Kd, B, N, T):
    w = synth.make_fused_workload("fused_small", seed=200 + k, device="cuda", V=V, Kt=Kt, Kd=Kd, B=B, N=N, T=T)
    _check(w)


def test_fused_all_greedy_without_draft_model():
    w = synth.make_fused_workload("fused_mixed", seed=1, device="cuda")
    rep, _ = _check(w, greedy=True)
    assert rep["exact"] >= rep["sequences"] - rep["band_sequences"]


@pytest.mark.parametrize("c1,c2", [(5, 40), (100, 200), (30, 700), (255, 256)])
def test_fused_greedy_ties_take_the_lowest_column(c1, c2):
    """Two vocabulary columns with identical head rows give equal logits; the
    greedy token is the lower column (the first index of the argmax), whether
    the twins share a 128-column chunk of the epilogue, sit in two chunks of one
    tile, or in two tiles.  Position k's draft token is the higher twin, so a
    kernel that took it would accept position k instead of emitting the lower
    twin there."""
    B, N, V, K = 8, 3, 1024, 64
    w = synth.make_fused_workload("fused_small", seed=c1 + c2, device="cuda", B=B, N=N, V=V, Kt=K, Kd=K)
    wt = w.target_weight.clone()
    wt[c2] = wt[c1]
    th = (wt[c1].float() * 40.0).to(torch.bfloat16).repeat(B * (N + 1), 1).contiguous()
    toks = torch.full((B, N), c1, dtype=torch.int32, device="cuda")
    want_out = np.full((B, N + 1), -1, np.int32)
    want_nacc = np.zeros(B, np.int32)
    for b in range(B):
        k = b % (N + 1)  # the higher twin's position; k == N: every draft is the lower twin
        if k < N:
            toks[b, k] = c2
        want_out[b, :k + 1] = c1
        want_nacc[b] = k
    w2 = dataclasses.replace(w, target_weight=wt, target_hidden=th, draft_tokens=toks)
    orc = parity.run_oracle_fused(w2, threads=THREADS, greedy=True)
    assert (orc["out_tokens"] == want_out).all() and (orc["num_accepted"] == want_nacc).all()
    ctx = sv.SpecVerify(B, N, V, "f32")
    out, nacc = ctx.run_fused(th, wt, None, None, toks, None, None, greedy=True)
    torch.cuda.synchronize()
    assert (out.cpu().numpy() == want_out).all(), out.cpu().numpy().tolist()
    assert (nacc.cpu().numpy() == want_nacc).all()
    assert ctx.status() == sv.SV_OK


@pytest.mark.parametrize("keep", [True, False], ids=["kept_logits", "recomputed_rows"])
def test_fused_full_size_sampled(keep):
    """The 256-sequence batch the benchmark times (Qwen-sized heads: V = 151936,
    Kt = 3584, Kd = 896); the oracle checks a spread of sequences."""
    w = synth.make_fused_workload("fused", seed=0, device="cuda")
    _check(w, seqs=np.array([0, 1, 100, 255]), keep=keep)


def test_fused_kept_and_recomputed_rows_agree_on_one_context():
    """One context switched between the two ways of getting the sampled rows
    (its scratch is reallocated at each switch): the same tokens outside the
    band, call after call."""
    w = synth.make_fused_workload("fused_mixed", seed=3, device="cuda")
    ctx = sv.SpecVerify(w.B, w.N, w.V, "f32")
    orc = parity.run_oracle_fused(w, threads=THREADS)
    in_band = (np.nan_to_num(orc["accept_margin"], nan=np.inf) < parity.FUSED_BAND).any(axis=1) | \
        (np.nan_to_num(orc["sample_margin"], nan=np.inf) < parity.FUSED_BAND)
    runs = []
    for keep in (True, False, True):
        ctx.set_fused_logits(keep)
        out, nacc = ctx.run_fused(w.target_hidden, w.target_weight, w.draft_hidden, w.draft_weight,
                                  w.draft_tokens, w.uniforms, w.temperature)
        torch.cuda.synchronize()
        assert ctx.status() == sv.SV_OK
        runs.append((out.cpu().numpy(), nacc.cpu().numpy()))
    for out, nacc in runs[1:]:
        same = (out == runs[0][0]).all(axis=1) & (nacc == runs[0][1])
        assert (same | in_band).all()
    assert np.array_equal(runs[0][0], runs[2][0]) and np.array_equal(runs[0][1], runs[2][1])


def test_fused_matches_the_logit_path():
    """The same float32 logits through spec_verify_lm_head_logits and
    spec_verify_run give the same tokens outside the band."""
    w = synth.make_fused_workload("fused_small", seed=2, device="cuda", B=16)
    ctx = sv.SpecVerify(w.B, w.N, w.V, "f32")
    out_f, nacc_f = ctx.run_fused(w.target_hidden, w.target_weight, w.draft_hidden, w.draft_weight, w.draft_tokens,
                                  w.uniforms, w.temperature)
    zt = sv.lm_head_logits(w.target_hidden, w.target_weight).view(w.B, w.N + 1, w.V)
    zd = sv.lm_head_logits(w.draft_hidden, w.draft_weight).view(w.B, w.N, w.V)
    out_c, nacc_c = ctx.run(zt, zd, w.draft_tokens, w.uniforms, w.temperature)
    torch.cuda.synchronize()
    orc = parity.run_oracle_fused(w, threads=THREADS)
    in_band = (np.nan_to_num(orc["accept_margin"], nan=np.inf) < parity.FUSED_BAND).any(axis=1) | \
        (np.nan_to_num(orc["sample_margin"], nan=np.inf) < parity.FUSED_BAND)
    same = (out_f == out_c).all(dim=1).cpu().numpy() & (nacc_f == nacc_c).cpu().numpy()
    assert (same | in_band).all()


def test_fused_host_errors_and_bad_tokens():
    w = synth.make_fused_workload("fused_small", seed=3, device="cuda")
    bf = sv.SpecVerify(w.B, w.N, w.V, "bf16")
    with pytest.raises(sv.SpecVerifyError) as e:
        bf.run_fused(w.target_hidden, w.target_weight, w.draft_hidden, w.draft_weight, w.draft_tokens, w.uniforms,
                     w.temperature)
    assert e.value.status == sv.SV_ERR_DTYPE
    ctx = sv.SpecVerify(w.B, w.N, w.V, "f32")
    w.draft_tokens[2, 1] = w.V + 5
    out, nacc = ctx.run_fused(w.target_hidden, w.target_weight, w.draft_hidden, w.draft_weight, w.draft_tokens,
                              w.uniforms, w.temperature)
    torch.cuda.synchronize()
    assert int(nacc[2]) == -1 and (out[2] == -1).all()
    assert ctx.status() == sv.SV_ERR_BAD_TOKEN
    w.draft_tokens[2, 1] = 0
    _check(synth.make_fused_workload("fused_small", seed=4, device="cuda"), ctx=ctx)
