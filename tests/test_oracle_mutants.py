"""Each deliberately broken copy of the oracle must fail at least one pin.

The mistakes are planted in the C oracle (compile-time ORACLE_MUTANT switch) and
run on the CPU only.  This shows the pins are sensitive to a dropped term, a wrong
sign, a wrong index, swapped operands, the wrong rounding rule and a wrong scale.
"""
import pytest

import oracle
import oracle_pins

MUTANTS = {
    1: "zero-point term dropped",
    2: "zero-point sign flipped",
    3: "nibble order swapped",
    4: "row sum skips one element",
    5: "ties rounded to even",
    6: "scale uses 128 instead of 127",
    7: "activation scale not applied",
    8: "high nibble treated as unsigned",
    9: "scale and zero swapped",
    10: "bias dropped",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda i: MUTANTS[i].replace(" ", "_"))
def test_mutant_is_caught(mutant):
    tag = f"oracle_mutant{mutant}"
    oracle.lib(tag=tag, defines=(f"ORACLE_MUTANT={mutant}",))
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(tag)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"
