"""Mutation tests: each case plants one plausible mistake in a copy of the oracle's
C source (oracle/w8a16_oracle.c itself holds none), compiles that copy into a
temporary directory, and checks that at least one pin of tests/test_oracle_pins.py
fails on it. The mistakes cover the number formats (E4M3 exponent bias,
subnormals given a leading one, the sign bit dropped, BF16 rounding that
truncates or breaks ties away from zero, an encoder that breaks ties away from
zero or turns out-of-range values into NaN), the layouts (one scale for every K
block, a transposed scale grid, W read as [K][N], the A row pitch ignored, the
W8A8 activation scales read token-major), the arithmetic (the last term dropped,
the sum carried in FP32, the W8A8 activation scale ignored) and the quantisers
(a range of 447, one activation amax per row).

Each patch is a literal text substitution; `count` is how many occurrences it
must replace (None: every occurrence, at least one), so a patch that no longer
matches the source fails loudly instead of testing an unmutated oracle."""
import pytest

import oracle
from test_oracle_pins import PINS

W_TERMS = ("        const double a = oracle_bf16_to_double(arow[k]);\n"
           "        const double w = j->dec[wrow[k]];\n"
           "        const double s = (double)srow[k / 128];\n")

MUTANTS = {
    1: ("E4M3 exponent bias off by one",
        [("mag = ldexp(8.0 + m, e - 7 - 3);", "mag = ldexp(8.0 + m, e - 7 - 2);", 1)]),
    2: ("BF16 rounding truncates",
        [("const double r = nearbyint(ldexp(a, -q));", "const double r = floor(ldexp(a, -q));", 1)]),
    3: ("first K block's scale used for every K block",
        [("const double s = (double)srow[k / 128];", "const double s = (double)srow[0];", None)]),
    4: ("scale grid read transposed",
        [("const double s = (double)srow[k / 128];",
          "const double s = (double)j->scale[(uint64_t)(k / 128) * ((j->N + 127) / 128) + n / 128];", None)]),
    5: ("W read as [K][N]",
        [("const double w = j->dec[wrow[k]];", "const double w = j->dec[j->W[(uint64_t)k * j->N + n]];", None)]),
    6: ("last term of the sum dropped",
        [("        const double t = a * (w * s);\n",
          "        if (k == j->K - 1)\n            continue;\n        const double t = a * (w * s);\n", None)]),
    7: ("block scale uses 447 instead of 448",
        [("const float scale = amax / 448.0f;\n            scales[(size_t)nb * kb_cols + kb] = scale;",
          "const float scale = amax / 447.0f;\n            scales[(size_t)nb * kb_cols + kb] = scale;", 1)]),
    8: ("W8A8 activation scales read token-major",
        [("j->a_scale[(uint64_t)(k / 128) * j->M + m]", "j->a_scale[(uint64_t)m * (j->K / 128) + k / 128]", 1)]),
    9: ("E4M3 subnormals decoded with an implicit leading one",
        [("mag = ldexp((double)m, -9);", "mag = ldexp(8.0 + m, -10);", 1)]),
    10: ("A row pitch ignored (rows read K apart)",
         [("const uint16_t *arow = j->A + (uint64_t)m * j->a_row_stride;",
           "const uint16_t *arow = j->A + (uint64_t)m * j->K;", 1)]),
    11: ("E4M3 encoder rounds ties away from zero",
         [("code = (lo & 1) ? hi : lo;", "code = hi;", 1)]),
    12: ("E4M3 encoder turns out-of-range values into NaN",
         [("    if (a >= 448.0)\n        return sign | 0x7E;\n",
           "    if (a > 448.0)\n        return sign | 0x7F;\n    if (a >= 448.0)\n        return sign | 0x7E;\n", 1)]),
    13: ("activation quantiser takes one amax over the whole row",
         [("            for (uint32_t k = g * 128; k < g * 128 + 128; ++k) {\n"
           "                const float v = fabsf(",
           "            for (uint32_t k = 0; k < K; ++k) {\n"
           "                const float v = fabsf(", 1)]),
    14: ("E4M3 sign bit dropped",
         [("return sign ? -mag : mag;", "(void)sign;\n    return mag;", 1)]),
    15: ("BF16 rounding ties away from zero",
         [("const double r = nearbyint(ldexp(a, -q));", "const double r = round(ldexp(a, -q));", 1)]),
    16: ("W8A8 activation scale ignored",
         [("const double a = j->dec[arow[k]] * (double)j->a_scale[(uint64_t)(k / 128) * j->M + m];",
           "const double a = j->dec[arow[k]];", 1)]),
    17: ("sum carried in FP32",
         [(W_TERMS, W_TERMS, 1),   # anchors the W8A16 loop (must still be there)
          ("    double sum = 0.0, asum = 0.0;\n", "    float sum = 0.0f;\n    double asum = 0.0;\n", None)]),
}


def mutated_source(patches) -> str:
    text = oracle.source_text()
    for old, new, count in patches:
        n = text.count(old)
        assert n >= 1 and (count is None or n == count), \
            f"mutation anchor found {n} times (want {count or '>= 1'}): {old!r}"
        text = text.replace(old, new)
    return text


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m][0])
def test_some_pin_catches_mutant(mutant, tmp_path_factory):
    desc, patches = MUTANTS[mutant]
    src = mutated_source(patches)
    assert src != oracle.source_text()
    o = oracle.Oracle(outdir=tmp_path_factory.mktemp(f"mutant{mutant}"), source=src)
    caught = []
    for pin in PINS:
        try:
            pin(o)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin detects mutant {mutant}: {desc}"


def test_oracle_source_holds_no_mutants():
    text = oracle.source_text()
    assert "MUTANT" not in text and "mutant" not in text
