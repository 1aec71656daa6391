"""Each planted mistake in the oracle must be caught by at least one pin.

The mutants are built from the same C source with -DSSM_ORACLE_PLANT=k into a
temporary directory: 1 drops the D skip, 2 flips the exponent's sign, 3 swaps B and C,
4 adds the bias after the softplus, 5 gates with sigmoid instead of SiLU, 6 drops Delta
from B-bar, 7 reads out before the state update, 8 reads A transposed, 9 skips softplus;
in the backward pass 10 drops the A a h_{t-1} term of d(dt), 11 carries g to step t-1
before using it at step t, 12 takes dC from h_{t-1}; in the SSD recurrence 13 assigns
heads to groups round-robin, 14 decays the new input with the state; 15 reverses the
conv taps; 16 drops the 1 / a of the zero-order hold.
"""
import pytest

import oracle
import pins

PLANTS = list(range(1, 17))


@pytest.mark.parametrize("plant", PLANTS)
def test_mutant_is_caught(plant, tmp_path):
    mutant = oracle.Oracle(oracle.build(out_dir=str(tmp_path), plant=plant, force=True))
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, FloatingPointError, OverflowError):
            caught.append(pin.__name__)
    assert caught, f"planted mistake {plant} passed every pin"
