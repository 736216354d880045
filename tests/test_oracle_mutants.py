"""Every planted mistake in the oracle (a dropped term, a wrong sign, index or operand, a
missing rescale, a missing -inf guard, a wrong head map, ignored key lengths) must fail at least
one pin.  The mistakes are planted
in copies of the oracle built on the CPU with -DORACLE_MUTANT=k; the real oracle has none."""
import pytest

import oracle
import oracle_pins

MUTANTS = {
    1: "row softmax forgets the max in the sum",
    2: "causal mask j < i instead of j <= i",
    3: "drops the last allowed key",
    4: "reads K transposed",
    5: "forgets the scale",
    6: "sign error in the exponent",
    7: "log base 2 in the log-sum-exp",
    8: "streaming state drops the rescale of l",
    9: "streaming state computes p against the old max",
    10: "streaming state has no -inf guard",
    11: "merge weighs both sides by one factor",
    12: "grouped heads dealt round-robin to the key/value heads",
    13: "per-sequence key lengths ignored",
    14: "top-k ties go to the larger column",
    15: "top-k skips the largest entry",
    16: "backward drops the D term of dS",
    17: "backward flips the sign of dS",
    18: "backward forgets the scale in dQ and dK",
    19: "explicit mask ignored",
    20: "explicit mask read transposed",
    21: "backward keeps only the last query head's part of a shared head's gradients",
    22: "backward ignores the key lengths",
}


@pytest.mark.parametrize("k", sorted(MUTANTS), ids=lambda k: f"mutant{k}")
def test_pins_catch_planted_mistake(k):
    orc = oracle.load(mutant=k)
    assert orc.mutant == k
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            with __import__("numpy").errstate(all="ignore"):
                pin(orc)
        except (AssertionError, ValueError, FloatingPointError, OverflowError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {k}: {MUTANTS[k]}"
