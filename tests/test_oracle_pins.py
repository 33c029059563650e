"""The oracle against closed forms, invariants, torch's CPU AdamW, brute-force sums and page values."""

import inspect

import pytest

import pins
from conftest import read_golden


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    if "golden" in inspect.signature(pin).parameters:
        pin(oracle_lib, read_golden("stats_plan.txt"))
    else:
        pin(oracle_lib)
