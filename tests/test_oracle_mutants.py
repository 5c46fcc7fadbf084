"""Mutation tests: each build plants one plausible mistake in the oracle (a wrong
exponent bias, truncation instead of round-to-nearest-even, one scale for every K
block, a transposed scale grid, W read as [K][N], a dropped last term) and at
least one pin of tests/test_oracle_pins.py must fail on it. The mistakes live
behind ORACLE_MUTANT in oracle/w8a16_oracle.c and are compiled only here, into
a temporary directory. The seventh plants a wrong range in the weight block
quantiser (scale = amax / 447); the eighth reads the W8A8 activation scales in the
wrong layout."""
import pytest

import oracle
from test_oracle_pins import PINS

MUTANTS = {
    1: "E4M3 exponent bias off by one",
    2: "BF16 rounding truncates",
    3: "first K block's scale used for every K block",
    4: "scale grid read transposed",
    5: "W read as [K][N]",
    6: "last term of the sum dropped",
    7: "block scale uses 447 instead of 448",
    8: "W8A8 activation scales read token-major",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m])
def test_some_pin_catches_mutant(mutant, tmp_path_factory):
    o = oracle.Oracle(mutant, outdir=tmp_path_factory.mktemp(f"mutant{mutant}"))
    caught = []
    for pin in PINS:
        try:
            pin(o)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin detects mutant {mutant}: {MUTANTS[mutant]}"
