"""The CPU oracle against its pins (closed forms, invariants, brute force, golden files).

Every check lives in ``tests/oracle_pins.py``; this module runs each one.
"""

import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()
