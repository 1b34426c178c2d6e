"""The row kernel's branch-free online normaliser, emulated on the host (CPU).

Per ring stage a thread folds its vectors into (m, s): M = max(m, tile max),
s <- s * r + sum_k 2^((z_k - M') c) with r = 2^((m - M) c) when the max grew
(else 1), and M' = M, or 0 while M is still -inf, so an all -inf prefix
leaves s = 0 and a NaN makes s NaN; columns past the row's end enter as -inf.
For bf16 the argument is z c - M' c in one rounding (fma).  Here that
recurrence runs in float32 (fma emulated in float64, then rounded)
over random tilings of a row, and its result, merged over threads as the
kernel merges them, is compared with sum_k exp((z_k - max z)/T) in float64.
"""
import numpy as np
import pytest

LOG2E = 1.4426950408889634074


def f32(x):
    return np.float32(x)


def fold_tile(m, s, tile, cf, bf16):
    """One stage: m, s float32 state; tile float32 values (-inf padded)."""
    with np.errstate(invalid="ignore", over="ignore"):
        vmax = f32(np.nanmax(tile)) if not np.all(np.isnan(tile)) else f32(np.nan)
        M = f32(np.fmax(m, vmax))                       # fmaxf: NaN is never the max
        r = f32(np.exp2(f32(f32(m - vmax) * cf))) if vmax > m else f32(1.0)
        Ms = f32(0.0) if M == -np.inf else M
        if bf16:
            nmc = -f32(Ms * cf)
            args = [f32(float(z) * float(cf) + float(nmc)) for z in tile]   # one rounding
        else:
            args = [f32(f32(z - Ms) * cf) for z in tile]
        e = f32(0.0)
        for a in args:  # the order of the partial sums does not matter at this tolerance
            e = f32(e + f32(np.exp2(a)))
        s = f32(float(s) * float(r) + float(e))  # fma(s, r, e)
    return M, s


def merge(a, b, cf):
    (ma, sa), (mb, sb) = a, b
    m = f32(np.fmax(ma, mb))
    with np.errstate(invalid="ignore", over="ignore"):
        xa = sa if ma == m else f32(sa * f32(np.exp2(f32(f32(ma - m) * cf))))
        xb = sb if mb == m else f32(sb * f32(np.exp2(f32(f32(mb - m) * cf))))
    return m, f32(xa + xb)


def kernel_normaliser(z, T, threads, tile_len, bf16, rng):
    cf = f32(LOG2E / float(T))
    parts = np.array_split(z.astype(np.float32), threads)
    states = []
    for p in parts:
        m, s = f32(-np.inf), f32(0.0)
        for k in range(0, len(p), tile_len):
            tile = p[k:k + tile_len]
            if len(tile) < tile_len:  # ragged end: -inf fill
                tile = np.concatenate([tile, np.full(tile_len - len(tile), -np.inf, np.float32)])
            m, s = fold_tile(m, s, tile, cf, bf16)
        states.append((m, s))
    out = states[0]
    for st in states[1:]:
        out = merge(out, st, cf)
    return out


@pytest.mark.parametrize("bf16", [False, True])
def test_normaliser_matches_the_definition(bf16):
    rng = np.random.default_rng(12 + bf16)
    for _ in range(40):
        V = int(rng.integers(5, 3000))
        T = float(10.0 ** rng.uniform(-1, 0.5))
        z = (rng.standard_normal(V) * rng.uniform(0.5, 8)).astype(np.float32)
        if rng.random() < 0.3:
            z[rng.random(V) < 0.5] = -np.inf  # masked vocabulary
        if not np.isfinite(z).any():
            z[0] = 0.0
        m, s = kernel_normaliser(z, T, int(rng.integers(1, 9)), int(rng.integers(1, 33)), bf16, rng)
        zf = z[np.isfinite(z)].astype(np.float64)
        assert m == np.float32(zf.max())
        ref = np.exp((zf - zf.max()) / np.float64(np.float32(T)) * 1.0).sum()
        # float32 exp2 arguments and sums; for bf16 the one rounding of M c in
        # z c - M c scales every term of a thread's sum by up to 2^(|M c| 2^-24)
        cf = float(np.float32(LOG2E / T))
        tol = 2e-6 + (abs(float(m)) * cf * 2.0 ** -24 * np.log(2) if bf16 else 0.0)
        assert abs(float(s) / ref - 1.0) < tol, (float(s), ref, tol)


def test_all_minus_inf_row_gives_zero_sum():
    z = np.full(100, -np.inf, np.float32)
    m, s = kernel_normaliser(z, 1.0, 4, 8, True, None)
    assert m == -np.inf and s == 0.0  # the kernel flags S == 0 as invalid


def test_nan_poisons_the_sum():
    rng = np.random.default_rng(3)
    z = rng.standard_normal(200).astype(np.float32)
    z[57] = np.nan
    m, s = kernel_normaliser(z, 0.8, 3, 16, True, rng)
    assert np.isnan(s)


def test_padding_does_not_change_the_sum():
    rng = np.random.default_rng(4)
    z = rng.standard_normal(96).astype(np.float32)
    a = kernel_normaliser(z, 0.7, 1, 32, True, rng)   # three full tiles
    b = kernel_normaliser(z, 0.7, 1, 40, True, rng)   # a ragged last tile padded with -inf
    assert a[0] == b[0]
    assert abs(float(a[1]) / float(b[1]) - 1.0) < 1e-6
