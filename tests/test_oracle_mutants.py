"""Planted mistakes in the oracle must be caught by the pins (CPU, no GPU).

oracle.c carries ORACLE_MUTANT blocks, each a plausible slip: a mis-decoded
e2m1 subnormal, an off-by-one e4m3 bias, swapped nibbles, a wrong scale
block, a reversed tie rule, no renormalisation, gate/up swapped, SiLU lost,
the shared expert dropped, the router or down matrix read transposed, and in
the pre-norm step of a stack a sum instead of a mean, eps outside the root
and truncation instead of rounding to bf16; in the dense GEMV the tensor
scale left out and the last column dropped; in expert-sink routing the
sinks left out of the denominator and the sinks taken as top-k candidates.
Each variant is compiled here; at least one pin must fail on it.
"""
import os

import pytest

import oracle
from tests import pins

MUTANTS = list(range(1, 19))


@pytest.mark.parametrize("mutant", MUTANTS)
def test_pins_catch_planted_mistake(mutant, tmp_path):
    path = os.path.join(str(tmp_path), f"liboracle_m{mutant}.so")
    oracle.build(mutant=mutant, out_path=path, openmp=False)
    lib = oracle.load(path)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
        except ValueError:
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} passed every pin"
