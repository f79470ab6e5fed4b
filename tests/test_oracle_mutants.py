"""Each planted mistake in the oracle (a mutant build of oracle.c) fails at
least one pin, and the real build fails none: the pins can see the kind of
mistake a restatement of the pages could plausibly contain."""
import pytest

import oracle
import pins

MUTANTS = {
    1: "E2M1 nibble order", 2: "gate/up swapped", 3: "requant scale rounded down", 4: "top-k weight dropped",
    5: "W2 read transposed", 6: "activation scale dropped", 7: "combine drops a slot", 8: "SiLU sign",
    9: "unstable routing order", 10: "per-128 scale granularity", 11: "BF16 truncation", 12: "E4M3 truncation",
    13: "FP8 weights read as E2M1", 14: "L2-only rows drop the activation scale",
    15: "float recipe: weight block scale dropped", 16: "float recipe: L2-activation scale from the wrong maximum",
}


def test_real_oracle_passes_every_pin(orc):
    fails = {k: v for k, v in pins.all_pins(orc).items() if v}
    assert fails == {}


@pytest.mark.parametrize("m", sorted(MUTANTS))
def test_mutant_is_caught(m):
    o = oracle.Oracle(mutant=m)
    fails = {k: v for k, v in pins.all_pins(o).items() if v}
    assert fails, f"mutant {m} ({MUTANTS[m]}) passed every pin"
