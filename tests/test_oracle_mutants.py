"""Mutation tests: each build plants one plausible mistake in the oracle (a wrong
exponent bias, truncation instead of round-to-nearest-even, one scale for every K
block, a transposed scale grid, W read as [K][N], a dropped last term) and at
least one pin of tests/test_oracle_pins.py must fail on it. The mistakes live
behind ORACLE_MUTANT in oracle/w8a16_oracle.c and are compiled only here, into
a temporary directory. The seventh plants a wrong range in the weight block
quantiser (scale = amax / 447); the eighth reads the W8A8 activation scales in the
wrong layout. The rest cover the number formats (E4M3 subnormals given a leading
one, the sign bit dropped, encoder ties away from zero, out-of-range values
encoded as NaN, BF16 ties away from zero), the row pitch, the precision of the
sum, the activation quantiser's group and the W8A8 activation scale."""
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
    9: "E4M3 subnormals decoded with an implicit leading one",
    10: "A row pitch ignored (rows read K apart)",
    11: "E4M3 encoder rounds ties away from zero",
    12: "E4M3 encoder turns out-of-range values into NaN",
    13: "activation quantiser takes one amax over the whole row",
    14: "E4M3 sign bit dropped",
    15: "BF16 rounding ties away from zero",
    16: "W8A8 activation scale ignored",
    17: "sum carried in FP32",
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
