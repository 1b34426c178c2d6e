"""spec_verify_run_noalloc against spec_verify_run (needs a GB300).

Some callers cannot allocate device memory while they run: an inference
engine that gave all free memory to its KV cache at start-up, or a plug-in
whose host framework owns every allocation.  spec_verify_run_noalloc serves
them with a fixed scratch array built into the library instead of a context
workspace.  Here it must give the same tokens and accept counts as the
context entry point, call after call, while its scratch carries over from one
call to the next.  The file name makes pytest collect it last.
"""
import pytest
import torch

import synth
import speculative_decoding_verification_49_gb300 as sv

pytestmark = pytest.mark.gpu


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


def test_noalloc_matches_the_context_entry_point_call_after_call():
    from speculative_decoding_verification_49_gb300 import build
    build.build()
    stream = torch.cuda.current_stream()
    # three calls in a row on the same scratch: a larger batch, then a smaller
    # one (slots of the first call are left behind), then float32 logits
    cases = [("headline", 21, {"B": 24}), ("headline", 22, {"B": 9}), ("stress", 23, {"B": 40})]
    for name, seed, over in cases:
        w = synth.make_workload(name, seed=seed, device="cuda", **over)
        ctx = sv.SpecVerify(w.B, w.N, w.V, w.dtype)
        ref_out, ref_acc = ctx.run(w.target, w.draft, w.draft_tokens, w.uniforms, w.temperature,
                                   stream=stream)
        out, acc = _run_noalloc(w, stream)
        torch.cuda.synchronize()
        assert ctx.status() == sv.SV_OK
        # same kernel and cluster size on the same device: identical decisions
        assert torch.equal(out, ref_out), name
        assert torch.equal(acc, ref_acc), name
        assert (acc >= 0).all() and (acc <= w.N).all()
        ctx.close()


def test_noalloc_rejects_batches_beyond_its_scratch():
    st = sv.spec_verify_run_noalloc(16, 16, 16, 16, 16, 0, 2049, 3, 1024, sv.SV_F32, 16, 16, None)
    assert st == sv.SV_ERR_TOO_LARGE
    st = sv.spec_verify_run_noalloc(16, 16, 16, 16, 16, 0, 1024, 32, 1024, sv.SV_F32, 16, 16, None)
    assert st == sv.SV_ERR_TOO_LARGE
    assert "2048" in sv.spec_verify_error_string(sv.SV_ERR_TOO_LARGE)
