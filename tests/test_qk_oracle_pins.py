"""The score-step oracle against its pins (CPU only)."""
import pytest

from oracle import gqa_qk
from qk_oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_qk_oracle_pin(pin):
    pin(gqa_qk)
