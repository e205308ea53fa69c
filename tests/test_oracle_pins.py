"""The CPU oracle against closed forms, brute force, torch fp64 routines,
hand-worked values and the invariants the pages state (no GPU needed)."""
import pytest

from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__[4:])
def test_pin(orc, pin):
    pin(orc)
