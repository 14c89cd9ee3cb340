"""The CPU oracle against its pins (CPU only)."""

import pytest

from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(orc, pin):
    pin(orc)


def test_oracle_threads(orc):
    assert orc.num_threads() >= 1
