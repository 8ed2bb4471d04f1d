"""The tied-covariance oracle against its pins (CPU only)."""
import pytest

import oracle
import oracle_tied_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_tied_oracle_pin(pin):
    pin(oracle.tied)
