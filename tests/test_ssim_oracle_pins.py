"""The float_ssim decimation oracle against facts other than itself (no
GPU): the page's auto scales, hand-derived sizes, repeated reflection,
exact-rational window sums, closed forms and the page's in-place finding."""
import pytest

import ssim_pins


@pytest.mark.parametrize("pin", ssim_pins.ALL_SSIM_PINS,
                         ids=lambda p: p.__name__)
def test_ssim_pin(pin, oracle_lib):
    pin(oracle_lib)
