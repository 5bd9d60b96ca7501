"""The oracle against what the mathematics and hand-worked fixtures fix (CPU only)."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_dense_bruteforce_fp8():
    pins.pin_dense_bruteforce(fp8=True)
