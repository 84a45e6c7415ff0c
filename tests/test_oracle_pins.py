"""CPU tier: the fp64 oracle against its pins (closed forms, invariants,
finite differences, a library rounding routine). See tests/oracle_pins.py."""
import pytest

import oracle
from tests import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)
