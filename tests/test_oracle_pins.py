"""The CPU oracle against independent pins (no GPU)."""
import pytest

import oracle.sinkattn_ref as ref
from tests import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    msg = check(ref)
    assert msg is None, msg
