"""The warp total the mass pass and the tree walk store (a xor butterfly) is
bit for bit the value the pick's warp-inclusive scan (shift-up, Kogge-Stone)
leaves in lane 31, so the pick finds the warp shares the mass pass wrote.

Both shuffle patterns are emulated lane by lane in float32 (round to nearest,
as __fadd_rn), on random, cancelling, tiny and huge values (CPU).
"""
import numpy as np
import pytest


def scan_last_lane(x):
    """Inclusive scan over 32 lanes: at step o, lane l >= o adds lane l - o."""
    v = np.array(x, dtype=np.float32)
    o = 1
    while o < 32:
        up = v.copy()
        for lane in range(31, -1, -1):
            if lane >= o:
                v[lane] = np.float32(up[lane] + up[lane - o])
        o <<= 1
    return v[31]


def butterfly_total(x):
    """Xor butterfly: at step o, every lane adds lane (l xor o); returns lane 31."""
    v = np.array(x, dtype=np.float32)
    o = 1
    while o < 32:
        prev = v.copy()
        for lane in range(32):
            v[lane] = np.float32(prev[lane] + prev[lane ^ o])
        o <<= 1
    return v[31]


def _cases():
    rng = np.random.default_rng(11)
    out = [rng.random(32, dtype=np.float32) for _ in range(200)]
    out += [(rng.standard_normal(32) * 10.0 ** rng.integers(-30, 30, 32)).astype(np.float32) for _ in range(200)]
    # the residual masses: many exact zeros, a few spikes
    for _ in range(100):
        v = np.zeros(32, dtype=np.float32)
        idx = rng.choice(32, size=rng.integers(1, 6), replace=False)
        v[idx] = rng.random(idx.size, dtype=np.float32) * np.float32(1e-3)
        out.append(v)
    out.append(np.full(32, np.float32(1e-45)))  # subnormals
    out.append(np.array([3e38] * 2 + [0] * 30, dtype=np.float32))  # overflow to inf in one add
    return out


@pytest.mark.parametrize("chunk", range(5))
def test_butterfly_equals_scan_lane_31(chunk):
    cases = _cases()
    for x in cases[chunk::5]:
        with np.errstate(over="ignore"):  # one case overflows to inf on purpose
            a, b = scan_last_lane(x), butterfly_total(x)
        assert a.tobytes() == b.tobytes(), (x, a, b)


def test_the_check_sees_order():
    """A different summation order (sequential) does differ on some input, so
    the equality above is not vacuous."""
    rng = np.random.default_rng(3)
    differs = False
    for _ in range(200):
        x = (rng.standard_normal(32) * 10.0 ** rng.integers(-8, 8, 32)).astype(np.float32)
        seq = np.float32(0)
        for v in x:
            seq = np.float32(seq + v)
        if seq.tobytes() != scan_last_lane(x).tobytes():
            differs = True
            break
    assert differs
