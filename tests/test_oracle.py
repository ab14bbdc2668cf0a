"""The CPU oracle against its pins (closed forms, a library routine,
invariants).  CPU only."""
import pytest

import oracle
from tests import oracle_pins as pins


@pytest.fixture(scope="module")
def ol():
    return oracle.OracleLib(oracle.build())


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=[p.__name__ for p in pins.ALL_PINS])
def test_oracle_pin(ol, pin):
    pin(ol)
