"""The row kernel's branch-free online normaliser, emulated on the host (CPU).

Per ring stage a thread folds its vectors into (m, s): M = max(m, tile max),
s <- s * r + sum_k 2^((z_k - M') c) with r = 2^((m - M) c) when the max grew
(else 1), and M' = M, or 0 while M is still -inf, so an all -inf prefix
leaves s = 0 and a NaN makes s NaN; columns past the row's end enter as -inf.
For bf16 the argument is z c - K in one rounding (fma), K = fl(M' c), which
shifts every term by e = M c - K; the rescale is then 2^(K_old - K_new), and
the thread's final sum is multiplied by 1 - e ln 2 (e = fma(m, c, -fl(m c))).
Here that recurrence runs in float32 (fma emulated in float64, then rounded)
over random tilings of a row, and its result, merged over threads as the
kernel merges them, is compared with sum_k exp((z_k - max z)/T) in float64.
"""
import numpy as np
import pytest

LOG2E = 1.4426950408889634074


def f32(x):
    return np.float32(x)


def fma32(a, b, c):
    """float32 fma: the exact a*b + c (float64 holds the product of two
    float32 exactly), rounded once."""
    return f32(float(a) * float(b) + float(c))


def fold_tile(m, s, tile, cf, bf16, shift_fix=True):
    """One stage: m, s float32 state; tile float32 values (-inf padded).
    shift_fix=False keeps the rescale 2^((m - M) c) with the bf16 arguments
    (the form before the common shift was taken out)."""
    with np.errstate(invalid="ignore", over="ignore"):
        vmax = f32(np.nanmax(tile)) if not np.all(np.isnan(tile)) else f32(np.nan)
        M = f32(np.fmax(m, vmax))                       # fmaxf: NaN is never the max
        Ms = f32(0.0) if M == -np.inf else M
        Kn, Ko = f32(Ms * cf), f32(m * cf)
        if bf16 and shift_fix:
            r = f32(np.exp2(f32(Ko - Kn))) if vmax > m else f32(1.0)
        else:
            r = f32(np.exp2(f32(f32(m - vmax) * cf))) if vmax > m else f32(1.0)
        if bf16:
            args = [fma32(z, cf, -Kn) for z in tile]   # one rounding
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


def fold_thread(m, s, cf, bf16, shift_fix=True):
    """A thread's final (m, s): for bf16 the common shift is taken out."""
    if bf16 and shift_fix and np.isfinite(m):
        e = fma32(m, cf, -f32(m * cf))                  # exactly m c - fl(m c)
        s = fma32(s, -f32(e * f32(0.6931471805599453)), s)
    return m, s


def kernel_normaliser(z, T, threads, tile_len, bf16, rng, shift_fix=True):
    cf = f32(LOG2E / float(T))
    parts = np.array_split(z.astype(np.float32), threads)
    states = []
    for p in parts:
        m, s = f32(-np.inf), f32(0.0)
        for k in range(0, len(p), tile_len):
            tile = p[k:k + tile_len]
            if len(tile) < tile_len:  # ragged end: -inf fill
                tile = np.concatenate([tile, np.full(tile_len - len(tile), -np.inf, np.float32)])
            m, s = fold_tile(m, s, tile, cf, bf16, shift_fix)
        states.append(fold_thread(m, s, cf, bf16, shift_fix))
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
        # float32 exp2 arguments and sums (the bf16 arguments' common shift
        # is taken out, so both forms meet the same bound)
        assert abs(float(s) / ref - 1.0) < 2e-6, (float(s), ref)


def test_bf16_common_shift_is_taken_out():
    """Logits near 60 at T = 0.3 (|M c| about 290, half an ulp of which is
    7.6e-6 in log2 units): without taking the common shift out, the sum is off
    by up to 5e-6 relative, more than the accept test's 1e-6 band can absorb
    in a ratio of two such sums; with it, within 2e-6 on every row."""
    rng = np.random.default_rng(21)
    worst_fixed = worst_plain = 0.0
    for _ in range(30):
        V = int(rng.integers(200, 2000))
        z = (60.0 + rng.standard_normal(V) * 2.0).astype(np.float32)
        z = z.astype(np.float32)
        T = 0.3
        zf = z.astype(np.float64)
        ref = np.exp((zf - zf.max()) / np.float64(np.float32(T))).sum()
        _, s_fix = kernel_normaliser(z, T, 4, 16, True, rng, shift_fix=True)
        _, s_plain = kernel_normaliser(z, T, 4, 16, True, rng, shift_fix=False)
        worst_fixed = max(worst_fixed, abs(float(s_fix) / ref - 1.0))
        worst_plain = max(worst_plain, abs(float(s_plain) / ref - 1.0))
    assert worst_fixed < 2e-6, worst_fixed
    assert worst_plain > 1e-6, worst_plain  # the shift the fix removes is really there


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
