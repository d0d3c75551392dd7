"""The oracle against its pins (closed forms, invariants, brute force, the
pages' printed numbers). No GPU involved."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)
