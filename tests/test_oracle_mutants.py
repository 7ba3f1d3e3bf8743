"""Pin strength: every planted mistake in the oracle is caught by some pin.

Each mutant is the oracle's C source built with -DORACLE_MUTANT=n, which turns
on exactly one plausible slip (wrong exponent bias, dropped scale, strict
causal mask, K/V halves swapped, wrong group or request index, unrounded or
mis-indexed gate, wrong split boundaries, sliding-window start or
position off by one, region selection that drops the current region or
keeps the lowest scores, indexer scores without the ReLU, with
rotated head weights, without the current region, from the wrong group or
with the token position off by one, ...).  The pins must reject each.
"""
import os
import tempfile

import pytest

import oracle
from _pins import ALL_PINS

MUTANTS = list(range(1, 27))


@pytest.fixture(scope="module")
def mutant_dir():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("mutant", MUTANTS)
def test_pins_catch_mutant(mutant, mutant_dir):
    path = oracle.build(os.path.join(mutant_dir, f"m{mutant}.so"), mutant=mutant, force=True)
    lib = oracle.load(path)
    for pin in ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, oracle.OracleError):
            return
    pytest.fail(f"no pin caught planted mistake {mutant}")
