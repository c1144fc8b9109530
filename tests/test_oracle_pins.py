"""The CPU oracle against its pins (no GPU)."""
import pytest

from oracle import wise_oracle
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    fails = pin(wise_oracle)
    assert not fails, "\n".join(fails[:20])
