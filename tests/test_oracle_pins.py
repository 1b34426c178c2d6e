"""The oracle against the pins (CPU only)."""
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=[p.__name__ for p in pins.ALL_PINS])
def test_pin(orc, pin):
    pin(orc)


def test_golden_file_parses():
    g = pins.golden()
    assert g["tokens_per_call.a0.75.N5"][0] == pytest.approx((1 - 0.75 ** 6) / 0.25, abs=1e-12)
    assert len(g) >= 10
