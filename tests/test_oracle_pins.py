"""The oracle against its pins (worked examples, closed forms, library
routines, invariants, brute force).  CPU only."""
import pytest

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_oracle_pin(oracle, pin):
    pin(oracle)
