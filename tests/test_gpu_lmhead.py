"""The tensor-core LM-head product against its float64 definition (needs a GB300)."""
import numpy as np
import pytest
import torch

import oracle
import parity
import speculative_decoding_verification_49_gb300 as sv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from speculative_decoding_verification_49_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _case(M, V, K, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    h = (torch.randn((M, K), generator=g) * 0.5).to(torch.bfloat16)
    w = (torch.randn((V, K), generator=g) * 0.05).to(torch.bfloat16)
    return h, w


def _bound(h, w):
    """Bound on the float32 product's error: LOGIT_ERR_FACTOR (2) times the
    size of a float32 sum of K products with random signs, sqrt(K) 2^-24
    sum_k |h_k w_k| (every case below measures at most 0.31 of that size).
    A product that dropped one term of its sum misses it by |h_k w_k|, far
    above the bound (checked on each case)."""
    return parity.LOGIT_ERR_FACTOR * parity.lm_head_error_scale(h, w) + 1e-30


def _report(err, h, w):
    """Largest error over the random-sign scale sqrt(K) 2^-24 sum_k |h_k w_k|."""
    r = float((err / (parity.lm_head_error_scale(h, w) + 1e-300)).max())
    print(f"lm-head error over sqrt(K) 2^-24 sum|hw|: {r:.3g} (K = {h.shape[1]})")
    return r


def _dropped_term_fails(want, h, w, bound):
    """The float64 product without its middle term lies outside the bound for
    most outputs (over 80 %): the bound can tell a missing product term apart."""
    k = h.shape[1] // 2
    term = np.outer(h[:, k].double().numpy(), w[:, k].double().numpy())
    off = np.abs(term) > bound
    assert off.mean() > 0.8, off.mean()


@pytest.mark.parametrize("M,V,K", [(128, 256, 64), (300, 1000, 72), (1, 17, 8), (257, 2304, 896),
                                   (130, 4099, 3584), (520, 40000, 136)])
def test_lm_head_logits_match_the_definition(M, V, K):
    h, w = _case(M, V, K, seed=M + V + K)
    got = sv.lm_head_logits(h.cuda(), w.cuda()).cpu().double().numpy()
    want = oracle.lm_head_logits(h, w)
    err = np.abs(got - want)
    _report(err, h, w)
    bound = _bound(h, w)
    assert (err <= bound).all(), float((err / bound).max())
    _dropped_term_fails(want, h, w, bound)


def test_lm_head_logits_sampled_at_vocabulary_size():
    """A Qwen-sized head (V = 151936, K = 3584) for 256 rows; 16 rows checked."""
    M, V, K = 256, 151936, 3584
    g = torch.Generator(device="cuda").manual_seed(1)
    h = (torch.randn((M, K), generator=g, device="cuda") * 0.5).to(torch.bfloat16)
    w = (torch.randn((V, K), generator=g, device="cuda") * 0.05).to(torch.bfloat16)
    got = sv.lm_head_logits(h, w)
    rows = torch.tensor([0, 1, 63, 64, 127, 128, 200, 255, 5, 77, 99, 150, 180, 222, 240, 254])
    want = oracle.lm_head_logits(h[rows].cpu(), w.cpu())
    err = np.abs(got[rows.cuda()].cpu().double().numpy() - want)
    _report(err, h[rows].cpu(), w.cpu())
    bound = _bound(h[rows].cpu(), w.cpu())
    assert (err <= bound).all()
    _dropped_term_fails(want, h[rows].cpu(), w.cpu(), bound)


def test_lm_head_logits_into_an_unaligned_output():
    """An output buffer that starts 4 bytes past a 16-byte boundary (no tensor
    map: the epilogue's warp stores) gives the same logits as an aligned one
    (tensor stores), and neither writes outside its [M, V] block."""
    M, V, K = 200, 2048, 128
    h, w = _case(M, V, K, seed=11)
    h, w = h.cuda(), w.cuda()
    want = sv.lm_head_logits(h, w).cpu()
    flat = torch.full((M * V + 8,), -7.0, dtype=torch.float32, device="cuda")
    out = flat[1:1 + M * V].view(M, V)
    assert out.data_ptr() % 16 == 4
    got = sv.lm_head_logits(h, w, out=out)
    torch.cuda.synchronize()
    assert torch.equal(got.cpu(), want)
    assert flat[0].item() == -7.0 and (flat[1 + M * V:] == -7.0).all()


def test_lm_head_logits_long_hidden_size():
    """A 70B-class hidden size (K = 8192: 128 stages per tile, the ring wrapping
    many times within each tile) for 512 rows of a 32768-entry head; 16 rows
    checked against the float64 product within the accumulation bound."""
    M, V, K = 512, 32768, 8192
    g = torch.Generator(device="cuda").manual_seed(3)
    h = (torch.randn((M, K), generator=g, device="cuda") * 0.5).to(torch.bfloat16)
    w = (torch.randn((V, K), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    got = sv.lm_head_logits(h, w)
    rows = torch.tensor([0, 1, 31, 32, 127, 128, 255, 256, 300, 383, 384, 400, 450, 500, 510, 511])
    want = oracle.lm_head_logits(h[rows].cpu(), w.cpu())
    err = np.abs(got[rows.cuda()].cpu().double().numpy() - want)
    _report(err, h[rows].cpu(), w.cpu())
    bound = _bound(h[rows].cpu(), w.cpu())
    assert (err <= bound).all()
    _dropped_term_fails(want, h[rows].cpu(), w.cpu(), bound)
