"""The fp64 oracle against what the pages and the mathematics fix (CPU)."""
import pytest

import oracle_pins

FAST = [p for p in oracle_pins.ALL_PINS
        if p not in (oracle_pins.pin_output_distribution,
                     oracle_pins.pin_expected_tokens)]


@pytest.mark.parametrize("pin", FAST, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


@pytest.mark.slow
def test_pin_output_distribution(orc):
    oracle_pins.pin_output_distribution(orc)


@pytest.mark.slow
def test_pin_expected_tokens(orc):
    oracle_pins.pin_expected_tokens(orc)
