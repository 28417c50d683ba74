"""The oracle against what the pages and the mathematics fix (no GPU)."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(oracle, pin):
    pin(oracle)


def test_oracle_reports_no_plant(oracle):
    assert oracle.plant == 0
