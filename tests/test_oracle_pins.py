"""The oracle against outside facts: library routines, the format definition,
closed forms, a hand-worked example and invariants of the method."""
import pytest

import _pins
import oracle as O


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(O.Oracle())
