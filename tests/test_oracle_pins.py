"""The oracle against facts other than itself (no GPU): hand-derived tables
under tests/golden/, closed forms, exact-rational evaluation of the fp64 term
sequence, brute-force 2-D convolution and an fp64 textbook VIF."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)
