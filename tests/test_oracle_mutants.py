"""Each planted mistake in the oracle (a transposed operand, a flipped sign,
crossed axes, a dropped term, wrong rounding or clamping, an off-by-one
extent) must fail at least one pin.  The mistakes live in the oracle source
behind ORACLE_MUTATION and are compiled only here, on the CPU."""
import pytest

import oracle
from tests import oracle_pins

MUTATIONS = {
    1: "filter taps transposed / columns mirrored",
    2: "padding sign flipped",
    3: "dilation axes crossed",
    4: "column stride ignored",
    5: "rint ties away from zero",
    6: "symmetric clamp range",
    7: "last input channel dropped",
    8: "output extent off by one dilation",
    9: "bias added before the per-channel scale",
    11: "per-channel scale indexed by the image",
    12: "fused multiply-add in the per-channel epilogue",
    13: "bias ignored in the fp32 direct convolution",
    14: "column dilation ignored in the fp32 direct convolution",
    15: "row stride ignored in the fp32 direct convolution",
    16: "bias indexed by the image in the fp32 direct convolution",
    17: "fp32 error bound with the unit roundoff 2^-23",
    18: "fp32 error bound gamma_n with n the product count (bias not counted)",
}


@pytest.mark.parametrize("mutation", sorted(MUTATIONS), ids=lambda m: MUTATIONS[m])
def test_pins_catch_mutation(mutation):
    orc = oracle.Oracle(mutation)
    assert orc.lib.oracle_mutation_id() == mutation
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, OverflowError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutation {mutation}: {MUTATIONS[mutation]}"
