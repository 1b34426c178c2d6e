"""KV-cache commit/rollback on the GPU against the oracle (needs a GB300).

The CUDA path (spec_verify_kv_commit through the C ABI) and the oracle's
plain row-by-row copy see the same seeded bytes; the cache, the lengths and
the status bits must agree exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import pins
import synth
import speculative_decoding_verification_49_gb300 as sv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_verification_49_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _random_case(rng, P, B, N, row, max_len, invalid=False):
    scratch = rng.integers(0, 256, (P, B, N, row), dtype=np.uint8)
    cache = rng.integers(0, 256, (P, B, max_len, row), dtype=np.uint8)
    nacc = rng.integers(0, N + 1, B).astype(np.int32)
    lens = np.array([rng.integers(0, max(1, max_len - a + 1)) for a in nacc], np.int32)
    if invalid and B >= 4:
        nacc[0] = -1                  # invalid verify: nothing
        nacc[1] = N + 1               # bad count
        lens[2] = max_len - nacc[2] + 1 if nacc[2] > 0 else max_len + 1  # overflow
        lens[3] = -5
    return scratch, cache, lens, nacc


def _gpu_commit(scratch, cache, lens, nacc):
    s = torch.from_numpy(scratch).cuda()
    c = torch.from_numpy(cache).cuda()
    ln = torch.from_numpy(lens).cuda()
    a = torch.from_numpy(nacc).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sv.kv_commit(s, c, ln, a, status=st)
    torch.cuda.synchronize()
    return c.cpu().numpy(), ln.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("P,B,N,row,max_len", [
    (1, 1, 1, 16, 1),        # smallest
    (3, 5, 7, 48, 20),       # ragged rows, many segments per CTA
    (4, 3, 5, 32, 24),       # the rollback exercise's shape
    (2, 9, 4, 4096, 11),     # a segment per CTA, chunks of whole rows
    (2, 3, 6, 40960, 9),     # one segment spans several 32 KiB chunks
    (56, 37, 7, 1024, 64),   # 7B-class GQA entry, ragged batch
    (2, 300, 1, 16, 3),      # many tiny segments (32 per CTA, ragged last CTA)
])
def test_kv_commit_matches_the_oracle(P, B, N, row, max_len):
    rng = np.random.default_rng(P * 1000 + B)
    case = _random_case(rng, P, B, N, row, max_len, invalid=True)
    want = oracle.kv_commit(*case)
    got = _gpu_commit(*case)
    assert got[2] == want[2]
    assert np.array_equal(got[1], want[1])
    assert np.array_equal(got[0], want[0])


def _random_layouts(n=10, seed=31):
    """Seeded random layouts: planes 1-12, B 1-60, N 1-8, rows a multiple of
    16 bytes up to 5 KiB (units that end inside a row and rows that span
    units), cache lengths 1-40; invalid, bad and overflowing counts mixed in."""
    rng = np.random.default_rng(seed)
    return [(k, int(rng.integers(1, 13)), int(rng.integers(1, 61)), int(rng.integers(1, 9)),
             int(rng.integers(1, 321)) * 16, int(rng.integers(1, 41))) for k in range(n)]


@pytest.mark.parametrize("k,P,B,N,row,max_len", _random_layouts())
def test_kv_commit_random_layouts(k, P, B, N, row, max_len):
    rng = np.random.default_rng(900 + k)
    case = _random_case(rng, P, B, N, row, max_len, invalid=True)
    want = oracle.kv_commit(*case)
    got = _gpu_commit(*case)
    assert got[2] == want[2]
    assert np.array_equal(got[1], want[1])
    assert np.array_equal(got[0], want[0])


def test_kv_commit_without_drafts_only_checks_lengths():
    rng = np.random.default_rng(5)
    cache = rng.integers(0, 256, (2, 4, 6, 16), dtype=np.uint8)
    scratch = np.zeros((2, 4, 0, 16), np.uint8)
    lens = np.array([0, 6, 3, 7], np.int32)
    nacc = np.array([0, 0, 1, 0], np.int32)
    want = oracle.kv_commit(scratch, cache, lens, nacc)
    got = _gpu_commit(scratch, cache, lens, nacc)
    assert got[2] == want[2] == (sv.SV_KV_BAD_COUNT | sv.SV_KV_OVERFLOW)
    assert np.array_equal(got[1], want[1]) and np.array_equal(got[0], cache)


def test_rollback_exercise_after_a_gpu_verify():
    """The lesson's exercise 4 end to end on the GPU: the verify kernel
    rejects the third draft of a 5-draft step over a 10-token prefix, and the
    commit leaves the cache reading the prefix plus the first 2 drafts."""
    N, V, L0, P, row = 5, 4096, 10, 4, 32
    B = 3
    g = torch.Generator(device="cpu").manual_seed(7)
    zq = torch.randn((B, N + 1, V), generator=g)
    zp = zq[:, :N].clone()
    zq[:, 2] = float("-inf")
    zq[:, 2, 11] = 0.0
    zp[:, 2] = float("-inf")
    zp[:, 2, 12] = 0.0
    d = zp.argmax(dim=-1).to(torch.int32)
    u = torch.full((B, N + 1), 0.5)
    T = torch.ones(B)
    w = synth.Workload("rollback", B, N, V, "f32", zq.cuda(), zp.cuda(), d.cuda(), u.cuda(), T.cuda())
    ctx = sv.SpecVerify(B, N, V, "f32")
    out, nacc = ctx.run(w.target, w.draft, w.draft_tokens, w.uniforms, w.temperature)
    assert nacc.cpu().tolist() == [2] * B
    rng = np.random.default_rng(8)
    prefixes = [list(rng.integers(0, V, L0)) for _ in range(B)]
    drafts = d.numpy().tolist()
    cache = torch.from_numpy(pins._kv_state(prefixes, P, 24, row)).cuda()
    scratch = torch.from_numpy(pins._kv_scratch(drafts, [L0] * B, P, N, row)).cuda()
    lens = torch.full((B,), L0, dtype=torch.int32, device="cuda")
    sv.kv_commit(scratch, cache, lens, nacc)
    torch.cuda.synchronize()
    assert lens.cpu().tolist() == [L0 + 2] * B
    c = cache.cpu().numpy()
    for b in range(B):
        seq = prefixes[b] + drafts[b][:2]
        assert np.array_equal(c[:, b, :L0 + 2], pins._kv_state([seq], P, L0 + 2, row)[:, 0])
        assert (c[:, b, L0 + 2:] == 0xEE).all()
    # and the verify's own emitted tokens agree: accepted drafts, then the correction
    o = out.cpu().numpy()
    assert (o[:, :2] == d.numpy()[:, :2]).all() and (o[:, 2] == 11).all()


def test_kv_commit_at_full_size_sampled():
    """A 7B-class cache (28 layers x K,V = 56 planes, 4 KV heads x 128 bf16 =
    1 KiB rows, 2048 positions) for the 256-sequence, 7-draft batch, with the
    accepted counts of a real verify launch.  Lengths and status are checked
    for every sequence, the bytes for a sample of (plane, sequence) slabs."""
    w = synth.make_workload("headline", seed=0, device="cuda")
    ctx = sv.SpecVerify(w.B, w.N, w.V, w.dtype)
    _, nacc = ctx.run(w.target, w.draft, w.draft_tokens, w.uniforms, w.temperature)
    del w
    P, B, N, max_len, heads, dim = 56, nacc.shape[0], 7, 2048, 4, 128
    gen = torch.Generator(device="cuda").manual_seed(3)
    scratch = torch.randn((P, B, N, heads, dim), generator=gen, device="cuda").to(torch.bfloat16)
    cache = torch.empty((P, B, max_len, heads, dim), dtype=torch.bfloat16, device="cuda")
    cache.view(torch.uint8).random_(0, 256, generator=gen)  # 30 GB: filled in place
    lens0 = torch.randint(0, max_len - N + 1, (B,), generator=gen, device="cuda", dtype=torch.int32)
    lens0[0] = max_len - N            # fills to the end when all drafts are accepted
    lens = lens0.clone()
    rng = np.random.default_rng(4)
    sample = [(0, 0), (P - 1, B - 1)] + [(int(rng.integers(P)), int(rng.integers(B))) for _ in range(30)]
    before = {(p, b): cache[p, b].view(torch.uint8).cpu().numpy() for p, b in sample}
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sv.kv_commit(scratch, cache, lens, nacc, status=st)
    torch.cuda.synchronize()
    a = nacc.cpu().numpy()
    # lengths and status for every sequence (row content does not matter for them)
    _, want_len, want_st = oracle.kv_commit(np.zeros((1, B, N, 16), np.uint8), np.zeros((1, B, max_len, 16), np.uint8),
                                            lens0.cpu().numpy(), a)
    assert int(st.item()) == want_st == 0
    assert np.array_equal(lens.cpu().numpy(), want_len)
    l0 = lens0.cpu().numpy()
    for p, b in sample:
        s_np = scratch[p, b].view(torch.uint8).cpu().numpy().reshape(1, 1, N, -1)
        c_np = before[(p, b)].reshape(1, 1, max_len, -1)
        want_c, _, _ = oracle.kv_commit(s_np, c_np, l0[b:b + 1], a[b:b + 1])
        got = cache[p, b].view(torch.uint8).cpu().numpy().reshape(1, 1, max_len, -1)
        assert np.array_equal(got, want_c), (p, b)


def test_kv_commit_twice_in_a_row_appends():
    rng = np.random.default_rng(9)
    P, B, N, row, max_len = 3, 6, 4, 64, 16
    scratch, cache, lens, nacc = _random_case(rng, P, B, N, row, max_len)
    lens[:] = rng.integers(0, 5, B)
    c1, l1, s1 = oracle.kv_commit(scratch, cache, lens, nacc)
    scratch2 = rng.integers(0, 256, scratch.shape, dtype=np.uint8)
    nacc2 = rng.integers(0, N + 1, B).astype(np.int32)
    c2, l2, s2 = oracle.kv_commit(scratch2, c1, l1, nacc2)
    s = torch.from_numpy(scratch).cuda()
    c = torch.from_numpy(cache).cuda()
    ln = torch.from_numpy(lens).cuda()
    sv.kv_commit(s, c, ln, torch.from_numpy(nacc).cuda())
    s.copy_(torch.from_numpy(scratch2))
    sv.kv_commit(s, c, ln, torch.from_numpy(nacc2).cuda())
    torch.cuda.synchronize()
    assert s1 == s2 == 0
    assert np.array_equal(ln.cpu().numpy(), l2) and np.array_equal(c.cpu().numpy(), c2)
