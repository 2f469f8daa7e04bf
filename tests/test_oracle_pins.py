"""The CPU oracle against facts it does not compute itself (-m "not gpu")."""
import pytest

import oracle as ora
from pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(ora.load())
