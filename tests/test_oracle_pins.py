"""The CPU oracle against its pins (see ``oracle_pins``)."""
import pytest

from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(oracle, pin):
    pin(oracle)
