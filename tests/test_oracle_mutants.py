"""Each planted mistake in the oracle must be caught by at least one pin.

The mutants are built from the same C source with -DSSM_ORACLE_PLANT=k into a
temporary directory: 1 drops the D skip, 2 flips the exponent's sign, 3 swaps B and C,
4 adds the bias after the softplus, 5 gates with sigmoid instead of SiLU, 6 drops Delta
from B-bar, 7 reads out before the state update, 8 reads A transposed, 9 skips softplus.
"""
import pytest

import oracle
import pins

PLANTS = [1, 2, 3, 4, 5, 6, 7, 8, 9]


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
