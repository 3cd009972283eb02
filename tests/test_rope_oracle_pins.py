"""The rotary-embedding + cache-write oracle against its pins (CPU only)."""

import pytest

import rope_pins
from oracle import rope_cache


@pytest.mark.parametrize("pin", rope_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(rope_cache)
