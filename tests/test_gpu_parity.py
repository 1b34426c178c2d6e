"""CUDA path against the float64 oracle (needs a GB300).

Every call goes through the C ABI (ctypes binding of libspecverify.so).  The
five workloads run at full size, and the oracle checks every sequence of
every launch, including the full headline and stress launches the benchmark
times.
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


def _ctx(w, **kw):
    return sv.SpecVerify(w.B, w.N, w.V, w.dtype, **kw)


def _check(w, seqs=None, ctx=None, greedy=None):
    ctx = ctx or _ctx(w)
    gpu = parity.run_gpu(ctx, w, greedy=greedy, seqs=seqs)
    orc = parity.run_oracle(w, seqs=seqs, threads=THREADS, greedy=greedy)
    rep = parity.compare(w, gpu, orc, check_probs=not (greedy or w.greedy))
    print(w.name, rep)
    # sequences that differ (all inside the band): at most one a launch here;
    # their rate over many launches is checked below
    assert rep["band_mismatch"] <= max(1, 1e-4 * rep["decisions"])
    assert ctx.status() == sv.SV_OK
    return rep


@pytest.mark.parametrize("name,seed,overrides", [
    ("tiny", 0, {}),
    ("tiny", 1, {}),
    ("small", 0, {}),
    ("small", 1, {}),
    ("mixed", 0, {}),
    ("headline", 0, {"B": 12}),
    ("stress", 0, {"B": 48}),
])
def test_parity_full_oracle(name, seed, overrides):
    w = synth.make_workload(name, seed=seed, device="cuda", **overrides)
    _check(w)


def _random_shapes(n=12, seed=2026):
    """Seeded random shapes: dtype, V at every 16-byte alignment (a multiple of
    8 bf16 or 4 f32 elements, up to 9600), N 0..7, B 1..40, one temperature or a
    per-sequence mix that includes greedy sequences."""
    rng = np.random.default_rng(seed)
    out = []
    for k in range(n):
        dtype = "bf16" if rng.random() < 0.5 else "f32"
        V = int(rng.integers(1, 1201)) * (8 if dtype == "bf16" else 4)
        N = int(rng.integers(0, 8))
        B = int(rng.integers(1, 41))
        T = (0.0, 0.5, 1.0, 1.7) if rng.random() < 0.5 else float(rng.choice([0.3, 0.8, 1.0, 2.0]))
        out.append((k, dtype, V, N, B, T))
    return out


@pytest.mark.parametrize("k,dtype,V,N,B,T", _random_shapes())
def test_parity_random_shapes(k, dtype, V, N, B, T):
    w = synth.make_workload("small", seed=100 + k, device="cuda", B=B, N=N, V=V, dtype=dtype, T=T)
    _check(w)


@pytest.mark.parametrize("dtype,T", [("bf16", (0.0, 0.7, 1.0)), ("f32", 0.9)])
def test_parity_one_row_per_cta(dtype, T):
    """More than a wave of positions (320 sequences x 4 positions) makes the
    row kernel take one CTA per logit row and meet a position's two rows
    through the workspace; every sequence against the oracle, with greedy
    sequences (draft rows not read), a bad token and a NaN row among them."""
    w = synth.make_workload("small", seed=31, device="cuda", B=320, N=3, V=4096 if dtype == "f32" else 8192,
                            dtype=dtype, T=T)
    w.draft_tokens[5, 1] = w.V + 3        # bad token
    w.draft[7, 2, 11] = float("nan")      # NaN in a draft row
    if dtype == "bf16":
        w.temperature[7] = 1.0            # a sampled sequence, so that its draft rows are read
    ctx = _ctx(w)
    assert ctx.cluster_size(w.B, w.N) == 1
    gpu = parity.run_gpu(ctx, w)
    orc = parity.run_oracle(w, threads=THREADS)
    rep = parity.compare(w, gpu, orc)
    print(w.name, rep)
    assert rep["sequences"] == w.B and rep["band_mismatch"] <= 1
    assert gpu["num_accepted"][5] == -1 and gpu["num_accepted"][7] == -1
    assert ctx.status() in (sv.SV_ERR_BAD_TOKEN, sv.SV_ERR_BAD_VALUE)
    assert ctx.status() == sv.SV_OK


@pytest.mark.parametrize("dtype,T,greedy", [("bf16", (0.0, 0.7, 1.0), False), ("f32", 0.9, False),
                                             ("bf16", 1.0, True)])
def test_parity_packed_rows(dtype, T, greedy):
    """Between two CTAs per SM and a wave of positions (64 sequences x 6
    positions on 152 SMs) the row kernel takes one CTA per row and packs the
    rows it reads at the front of its grid: every target row, then the draft
    rows of the sampled sequences only.  Every sequence against the oracle:
    greedy and sampled sequences side by side with an invalid temperature, a
    bad token and a NaN among them; all sampled in float32 (more rows than a
    wave); and the greedy flag with no draft logits (no draft rows at all)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    w = synth.make_workload("mixed", seed=41, device="cuda", B=64, N=5, V=8192 if dtype == "bf16" else 4096,
                            dtype=dtype, T=T)
    assert 2 * sms <= w.B * (w.N + 1) < 4 * sms
    ctx = _ctx(w)
    assert ctx.cluster_size(w.B, w.N) == 1
    if greedy:
        rep = _check(w, ctx=ctx, greedy=True)
        assert rep["exact"] == rep["sequences"] == w.B
        return
    w.draft_tokens[5, 1] = w.V + 3        # bad token
    w.draft[9, 2, 11] = float("nan")      # NaN in a draft row
    w.temperature[9] = 1.0                # a sampled sequence, so that its draft rows are read
    w.temperature[12] = float("nan")      # invalid temperature
    gpu = parity.run_gpu(ctx, w)
    orc = parity.run_oracle(w, threads=THREADS)
    rep = parity.compare(w, gpu, orc)
    print(w.name, dtype, rep)
    assert rep["sequences"] == w.B and rep["band_mismatch"] <= 1
    assert gpu["num_accepted"][5] == -1 and gpu["num_accepted"][9] == -1 and gpu["num_accepted"][12] == -1
    assert ctx.status() in (sv.SV_ERR_BAD_TOKEN, sv.SV_ERR_BAD_VALUE)
    assert ctx.status() == sv.SV_OK


@pytest.mark.parametrize("name", ["headline", "stress"])
def test_parity_full_size_every_sequence(name):
    """The full-size launch the benchmark times (headline: 256 sequences x 15
    rows of 151936 bf16 logits; stress: 1024 x 7 rows of 128256 f32 logits),
    every sequence checked against the oracle."""
    w = synth.make_workload(name, seed=0, device="cuda")
    rep = _check(w)
    assert rep["sequences"] == w.B


def test_band_rate_over_fifty_headline_launches():
    """Every sequence of 50 full-size headline launches (seeds 100-149, about
    43 000 accept and sampling decisions) against the oracle.  Outside the
    1e-6 margin band every token and count matches, and every decision ratio
    lies within the band of the oracle's.  The sequences that differ (all
    inside the band) must be fewer than 1e-4 of the decisions.  The share of
    decisions inside the band is reported, split into accept tests and final
    samples."""
    ctx = sv.SpecVerify(256, 7, 151936, "bf16")
    tot = {"decisions": 0, "band_decisions": 0, "band_mismatch": 0, "sequences": 0, "exact": 0}
    acc_dec = acc_band = smp_dec = smp_band = 0
    worst = 0.0
    details = []
    for seed in range(100, 150):
        w = synth.make_workload("headline", seed=seed, device="cuda")
        gpu = parity.run_gpu(ctx, w)
        orc = parity.run_oracle(w, threads=THREADS)
        rep = parity.compare(w, gpu, orc)
        assert ctx.status() == sv.SV_OK
        for k in tot:
            tot[k] += rep[k]
        am, sm = orc["accept_margin"], orc["sample_margin"]
        acc_dec += int((~np.isnan(am)).sum())
        acc_band += int((am < parity.BAND).sum())
        smp_dec += int((~np.isnan(sm)).sum())
        smp_band += int((sm < parity.BAND).sum())
        worst = max(worst, rep["decision_ratio_err_max"])
        diff = np.nonzero(((gpu["out_tokens"] != orc["out_tokens"]).any(axis=1))
                          | (gpu["num_accepted"] != orc["num_accepted"]))[0]
        for b in diff:
            details.append((seed, int(b), int(orc["num_accepted"][b]), int(gpu["num_accepted"][b]),
                            float(np.nanmin(am[b], initial=np.inf)), float(sm[b])))
        del w, gpu, orc
        torch.cuda.empty_cache()
    print(f"50 headline launches: {tot}; accept tests {acc_dec} ({acc_band} in the band), "
          f"samples {smp_dec} ({smp_band} in the band); band rate {tot['band_decisions'] / tot['decisions']:.3g}; "
          f"differing sequences {tot['band_mismatch']} = {tot['band_mismatch'] / tot['decisions']:.3g} of decisions; "
          f"decision ratio error max {worst:.3g}")
    for d in details:
        print("differs (seed, b, j oracle, j gpu, min accept margin, sample margin):", d)
    assert tot["decisions"] >= 40000
    assert worst <= parity.BAND
    assert acc_band < 1e-4 * acc_dec
    assert tot["band_mismatch"] < 1e-4 * tot["decisions"]


def test_parity_all_greedy_without_draft_logits():
    w = synth.make_workload("mixed", seed=2, device="cuda", B=16)
    rep = _check(w, greedy=True)
    assert rep["exact"] == rep["sequences"]


def test_greedy_ties_take_the_lowest_index():
    g = torch.Generator(device="cuda").manual_seed(5)
    B, N, V = 6, 3, 4096
    target = torch.randint(-3, 2, (B, N + 1, V), generator=g, device="cuda").to(torch.bfloat16)
    target[:, :, V - 1] = 1.0  # ties with the first max almost everywhere
    a = target.float().argmax(dim=-1)
    tokens = a[:, :N].to(torch.int32).clone()
    tokens[1, 1] = (tokens[1, 1] + 1) % V
    T = torch.zeros(B, device="cuda")
    u = torch.rand((B, N + 1), generator=g, device="cuda")
    w = synth.Workload("ties", B, N, V, "bf16", target.contiguous(), torch.zeros((B, N, V), dtype=torch.bfloat16,
                       device="cuda"), tokens, u, T)
    rep = _check(w)
    assert rep["exact"] == B


@pytest.mark.parametrize("N", [0, 1, 2])
def test_small_N(N):
    w = synth.make_workload("small", seed=3, device="cuda", B=5, N=N)
    _check(w)


@pytest.mark.parametrize("V,dtype", [(8, "bf16"), (4, "f32"), (16, "f32"), (1000, "f32"), (4104, "bf16"),
                                     (65544, "bf16"), (262144, "bf16")])
def test_ragged_and_extreme_vocabularies(V, dtype):
    w = synth.make_workload("small", seed=4, device="cuda", B=3, N=3, V=V, dtype=dtype)
    _check(w)


@pytest.mark.parametrize("C", [1, 2, 3, 4, 5, 7, 8])
def test_every_cluster_size_matches_the_oracle(C):
    w = synth.make_workload("headline", seed=5, device="cuda", B=6)
    ctx = _ctx(w)
    ctx.set_cluster_size(C)
    assert ctx.cluster_size(w.B, w.N) == C
    _check(w, ctx=ctx)


def test_masked_vocabulary_rows():
    w = synth.make_workload("small", seed=6, device="cuda", B=6)
    g = torch.Generator(device="cuda").manual_seed(6)
    keep = torch.rand((w.B, w.N + 1, w.V), generator=g, device="cuda") < 0.1
    w.target = torch.where(keep, w.target, torch.full_like(w.target, float("-inf")))
    w.draft = torch.where(keep[:, :w.N], w.draft, torch.full_like(w.draft, float("-inf")))
    # drafts must have draft mass: re-pick them among kept tokens
    w.draft_tokens = torch.argmax(w.draft.float(), dim=-1).to(torch.int32)
    # a whole leading chunk of -inf in one row
    w.target[0, 0, : w.V // 2] = float("-inf")
    _check(w)


def test_identical_draft_accepts_everything():
    """p == q: the ratio is exactly 1, every draft is accepted, bonus emitted."""
    w = synth.make_workload("headline", seed=7, device="cuda", B=8)
    w.draft = w.target[:, : w.N].clone()
    w.uniforms[:, : w.N] = 0.99999994  # largest float32 below 1
    ctx = _ctx(w)
    gpu = parity.run_gpu(ctx, w)
    assert (gpu["num_accepted"] == w.N).all()
    assert (gpu["out_tokens"][:, : w.N] == w.draft_tokens.cpu().numpy()).all()
    _check(w, ctx=ctx)


def test_disjoint_one_hot_rejects_first():
    B, N, V = 4, 3, 2048
    target = torch.full((B, N + 1, V), float("-inf"), device="cuda")
    draft = torch.full((B, N, V), float("-inf"), device="cuda")
    y, x = 1234, 77
    target[:, :, y] = 0.0
    draft[:, :, x] = 0.0
    tokens = torch.full((B, N), x, dtype=torch.int32, device="cuda")
    u = torch.rand((B, N + 1), device="cuda")
    w = synth.Workload("onehot", B, N, V, "f32", target, draft, tokens, u, torch.ones(B, device="cuda"))
    gpu = parity.run_gpu(_ctx(w), w)
    assert (gpu["num_accepted"] == 0).all()
    assert (gpu["out_tokens"][:, 0] == y).all() and (gpu["out_tokens"][:, 1:] == -1).all()


def test_invalid_inputs_give_minus_one_and_status():
    w = synth.make_workload("small", seed=8, device="cuda", B=6)
    w.draft_tokens[0, 1] = w.V           # bad token
    w.target[1, 2, 5] = float("nan")     # NaN logit
    w.draft[2, 0, :] = float("-inf")     # draft row without mass
    w.temperature[3] = float("nan")      # bad temperature
    ctx = _ctx(w)
    gpu = parity.run_gpu(ctx, w, debug=False)
    for b in range(4):
        assert gpu["num_accepted"][b] == -1 and (gpu["out_tokens"][b] == -1).all()
    assert (gpu["num_accepted"][4:] >= 0).all()
    st = ctx.status()
    assert st in (sv.SV_ERR_BAD_TOKEN, sv.SV_ERR_BAD_VALUE)
    assert ctx.status() == sv.SV_OK  # read-and-clear
    orc = parity.run_oracle(w)
    assert (orc["out_tokens"] == gpu["out_tokens"]).all()


def test_repeated_calls_reuse_the_workspace():
    ctx = sv.SpecVerify(64, 7, 151936, "bf16")
    for seed, B in [(10, 5), (11, 7), (12, 3), (13, 7)]:
        w = synth.make_workload("headline", seed=seed, device="cuda", B=B)
        _check(w, ctx=ctx)


def test_host_errors():
    w = synth.make_workload("small", seed=9, device="cuda", B=2)
    ctx = _ctx(w)
    out = torch.empty((w.B, w.N + 1), dtype=torch.int32, device="cuda")
    acc = torch.empty((w.B,), dtype=torch.int32, device="cuda")
    base = (ctx.ctx, w.target.data_ptr(), w.draft.data_ptr(), w.draft_tokens.data_ptr(),
            w.uniforms.data_ptr(), w.temperature.data_ptr(), 0)
    tail = (out.data_ptr(), acc.data_ptr(), None)
    assert sv.spec_verify_run(*base, w.B + 1, w.N, *tail) == sv.SV_ERR_INVALID_ARG
    assert sv.spec_verify_run(*base, w.B, w.N + 1, *tail) == sv.SV_ERR_INVALID_ARG
    mis = (ctx.ctx, w.target.data_ptr() + 2) + base[2:]
    assert sv.spec_verify_run(*mis, w.B, w.N, *tail) == sv.SV_ERR_INVALID_ARG
    assert sv.spec_verify_run(*base, 0, w.N, *tail) == sv.SV_OK
    assert sv.spec_verify_run(ctx.ctx, w.target.data_ptr(), None, w.draft_tokens.data_ptr(),
                              w.uniforms.data_ptr(), w.temperature.data_ptr(), 0, w.B, w.N,
                              *tail) == sv.SV_ERR_INVALID_ARG


def test_profiling_hook_times_both_kernels():
    w = synth.make_workload("headline", seed=14, device="cuda", B=8)
    ctx = _ctx(w)
    ctx.profile(True)
    for _ in range(3):
        ctx.run(w.target, w.draft, w.draft_tokens, w.uniforms, w.temperature)
    ms_rows, ms_sample, n = ctx.profile_read()
    assert n == 3 and ms_rows > 0.0 and ms_sample > 0.0
    ctx.profile(False)
    with pytest.raises(sv.SpecVerifyError):
        ctx.profile_read()
    _check(w, ctx=ctx)  # profiling left the results alone


def test_acceptance_counts_match_the_oracle_histogram():
    """The counters kernel C keeps equal the histogram of the oracle's
    num_accepted over every run since the last reset (invalid sequences in
    the last slot)."""
    ctx = sv.SpecVerify(16, 5, 32000, "bf16")
    assert ctx.acceptance_counts() == [0] * 7
    want = np.zeros(7, dtype=np.int64)
    for seed, B in [(20, 16), (21, 9)]:
        w = synth.make_workload("small", seed=seed, device="cuda", B=B)
        if seed == 21:
            w.draft_tokens[3, 0] = -2  # one invalid sequence
        parity.run_gpu(ctx, w, debug=False)
        orc = parity.run_oracle(w, threads=THREADS)
        for a in orc["num_accepted"]:
            want[a if a >= 0 else 6] += 1
    ctx.status()
    got = ctx.acceptance_counts(reset=True)
    assert sum(got) == 25 and got[6] == 1
    # a sampled decision inside the margin band may move one sequence
    assert np.abs(np.array(got) - want).sum() <= 2
    assert ctx.acceptance_counts() == [0] * 7


def test_bounded_wait_gives_up_and_reports():
    """Failure detection without a fault: a kernel wait that nothing ever
    satisfies gives up after its limit and reports it; the GPU and a context
    stay usable afterwards."""
    import time
    t0 = time.perf_counter()
    assert sv.selftest_timeout(20000)  # 20 ms
    dt = time.perf_counter() - t0
    assert 0.015 < dt < 2.0, dt
    w = synth.make_workload("tiny", seed=11, device="cuda")
    _check(w)
