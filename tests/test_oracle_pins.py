"""The oracle against facts the pages and mathematics fix (CPU only)."""
import pytest

import oracle as ora
import pins


@pytest.fixture(scope="module")
def be():
    return ora.load()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(be, pin):
    pin(be)
