"""The oracle against its pins (see tests/pins.py for what each pin holds it to)."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(ora, pin):
    pin(ora)
