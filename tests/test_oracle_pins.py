"""The oracle against its pins (closed forms, lfilter, brute force, the
parity example, superposition and split/carry identities)."""
import pytest

import oracle
import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.load())
