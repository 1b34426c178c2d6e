"""The verify step fused into the LM-head products, against the float64
oracle on the float64 products (needs a GB300)."""
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


def _check(w, greedy=None, seqs=None, ctx=None):
    ctx = ctx or sv.SpecVerify(w.B, w.N, w.V, "f32")
    gpu = parity.run_gpu_fused(ctx, w, greedy=greedy, seqs=seqs)
    orc = parity.run_oracle_fused(w, seqs=seqs, threads=THREADS, greedy=greedy)
    rep = parity.compare_fused(w, gpu, orc, greedy=bool(greedy))
    print(w.name, rep)
    assert rep["band_mismatch"] <= max(1, rep["sequences"] // 20)
    assert ctx.status() == sv.SV_OK
    return rep, gpu


@pytest.mark.parametrize("name,seed", [("fused_small", 0), ("fused_small", 1), ("fused_mixed", 0)])
def test_fused_parity(name, seed):
    w = synth.make_fused_workload(name, seed=seed, device="cuda")
    _check(w)


@pytest.mark.parametrize("V,Kt,Kd", [(4104, 200, 72), (1000, 64, 8), (20, 520, 136)])
def test_fused_ragged_vocabulary_and_depth(V, Kt, Kd):
    """A last vocabulary tile shorter than 256 columns, and K not a multiple of
    the 64-wide stage (the tensor maps fill the missing columns with zeros)."""
    w = synth.make_fused_workload("fused_small", seed=V, device="cuda", V=V, Kt=Kt, Kd=Kd)
    _check(w)


def test_fused_all_greedy_without_draft_model():
    w = synth.make_fused_workload("fused_mixed", seed=1, device="cuda")
    rep, _ = _check(w, greedy=True)
    assert rep["exact"] >= rep["sequences"] - rep["band_sequences"]


def test_fused_full_size_sampled():
    """The 256-sequence batch the benchmark times (Qwen-sized heads: V = 151936,
    Kt = 3584, Kd = 896); the oracle checks a spread of sequences."""
    w = synth.make_fused_workload("fused", seed=0, device="cuda")
    _check(w, seqs=np.array([0, 1, 100, 255]))


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
