"""The oracle against facts fixed outside itself (CPU only).

Each pin lives in ``oracle_pins.py``; see that module for the source of every fact.
"""
import pytest

import oracle
import oracle_pins as pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)
