"""The CPU oracle against its pins (closed forms, invariants, library routines
on special cases, brute force on tiny inputs, the pages' worked example)."""

import pytest

import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)
