"""The fp64 oracle against facts other than itself (CPU only)."""
import pytest

import oracle
import oracle_pins as P


@pytest.fixture(scope="module")
def o():
    return oracle.Oracle()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(o, pin):
    pin(o)
