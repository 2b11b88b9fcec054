"""The fp64 oracle against closed forms, brute force and invariances (CPU)."""
import pytest

import oracle_pins

pytestmark = pytest.mark.timeout(600) if hasattr(pytest.mark, "timeout") else []


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)
