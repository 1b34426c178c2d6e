"""spec_verify_run_noalloc against spec_verify_run and the oracle (needs a GB300).

Some callers cannot allocate device memory while they run: an inference
engine that gave all free memory to its KV cache at start-up, or a plug-in
whose host framework owns every allocation.  spec_verify_run_noalloc serves
them with a fixed scratch array built into the library instead of a context
workspace.  Here it must give the same tokens and accept counts as the
context entry point, call after call on the one shared scratch (batches of
different sizes and dtypes in a row, the full 256-sequence headline batch, the
mixed greedy/sampled batch, and a batch exactly at the scratch's slice limit),
and agree with the float64 oracle outside its margin band.  The file name makes pytest collect it last.
"""
import os

import pytest
import torch

import parity
import synth
import speculative_decoding_verification_49_gb300 as sv

pytestmark = pytest.mark.gpu

THREADS = max(1, min(16, os.cpu_count() or 1))


def _ptr(t):
    return t.data_ptr()


def _run_noalloc(w, stream):
    out = torch.full((w.B, w.N + 1), -9, dtype=torch.int32, device=w.target.device)
    acc = torch.full((w.B,), -9, dtype=torch.int32, device=w.target.device)
    st = sv.spec_verify_run_noalloc(_ptr(w.target), _ptr(w.draft), _ptr(w.draft_tokens), _ptr(w.uniforms),
                                    _ptr(w.temperature), 0, w.B, w.N, w.V,
                                    sv.SV_BF16 if w.dtype == "bf16" else sv.SV_F32,
                                    _ptr(out), _ptr(acc), stream.cuda_stream)
    assert st == sv.SV_OK, sv.spec_verify_error_string(st)
    return out, acc


def _against_oracle(w, out, acc, seqs=None):
    """The oracle's tokens and counts, exact outside the margin band."""
    orc = parity.run_oracle(w, seqs=seqs, threads=THREADS)
    gpu = {"out_tokens": out.cpu().numpy(), "num_accepted": acc.cpu().numpy()}
    if seqs is not None:
        gpu = {k: v[seqs] for k, v in gpu.items()}
    rep = parity.compare(w, gpu, orc, check_probs=False)
    assert rep["band_decisions"] <= max(1, 1e-4 * rep["decisions"]) or rep["band_mismatch"] == 0
    return rep


def test_noalloc_matches_the_context_entry_point_call_after_call():
    from speculative_decoding_verification_49_gb300 import build
    build.build()
    stream = torch.cuda.current_stream()
    # calls in a row on the same scratch: a larger batch, then a smaller one,
    # then float32 logits, then the full 256-sequence headline batch
    # (256 x 75 residual slices), then the mixed greedy/sampled batch (one
    # CTA per row, the rows read packed into one wave), then the first again
    cases = [("headline", 21, {"B": 24}), ("headline", 22, {"B": 9}), ("stress", 23, {"B": 40}),
             ("headline", 24, {}), ("mixed", 26, {}), ("headline", 21, {"B": 24})]
    for name, seed, over in cases:
        w = synth.make_workload(name, seed=seed, device="cuda", **over)
        ctx = sv.SpecVerify(w.B, w.N, w.V, w.dtype)
        ref_out, ref_acc = ctx.run(w.target, w.draft, w.draft_tokens, w.uniforms, w.temperature,
                                   stream=stream)
        out, acc = _run_noalloc(w, stream)
        torch.cuda.synchronize()
        assert ctx.status() == sv.SV_OK
        # same kernels and cluster size on the same device: identical decisions
        assert torch.equal(out, ref_out), (name, w.B)
        assert torch.equal(acc, ref_acc), (name, w.B)
        assert (acc >= 0).all() and (acc <= w.N).all()
        rep = _against_oracle(w, out, acc)
        print(name, w.B, rep)
        ctx.close()
        del w
        torch.cuda.empty_cache()


def test_noalloc_at_the_slice_limit():
    """B * ceil(V*elt / 4 KiB) exactly at the scratch's 32768 residual slices
    (512 sequences of 131072 bf16 logits, 64 slices a row): accepted, and
    equal to the context entry point and to the oracle."""
    stream = torch.cuda.current_stream()
    w = synth.make_workload("headline", seed=25, device="cuda", B=512, N=3, V=131072)
    ctx = sv.SpecVerify(w.B, w.N, w.V, w.dtype)
    ref_out, ref_acc = ctx.run(w.target, w.draft, w.draft_tokens, w.uniforms, w.temperature, stream=stream)
    out, acc = _run_noalloc(w, stream)
    torch.cuda.synchronize()
    assert ctx.status() == sv.SV_OK
    assert torch.equal(out, ref_out) and torch.equal(acc, ref_acc)
    _against_oracle(w, out, acc, seqs=list(range(0, 512, 8)) + [511])
    ctx.close()


def test_noalloc_rejects_batches_beyond_its_scratch():
    st = sv.spec_verify_run_noalloc(16, 16, 16, 16, 16, 0, 2049, 3, 1024, sv.SV_F32, 16, 16, None)
    assert st == sv.SV_ERR_TOO_LARGE
    st = sv.spec_verify_run_noalloc(16, 16, 16, 16, 16, 0, 1024, 32, 1024, sv.SV_F32, 16, 16, None)
    assert st == sv.SV_ERR_TOO_LARGE
    # one slice past the limit: 513 sequences of 64 slices
    st = sv.spec_verify_run_noalloc(16, 16, 16, 16, 16, 0, 513, 3, 131072, sv.SV_BF16, 16, 16, None)
    assert st == sv.SV_ERR_TOO_LARGE
    assert "2048" in sv.spec_verify_error_string(sv.SV_ERR_TOO_LARGE)
