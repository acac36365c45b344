"""The float64 oracle against what the pages and the mathematics fix.

Each pin lives in ``oracle_pins.py``; see that module for the facts and their
sources. These run on the CPU only.
"""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(orc, pin):
    pin(orc)
