"""CPU pins of the fp64 oracle (no GPU)."""
import pytest

import oracle
import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(0)


@pytest.mark.parametrize("mutant", sorted(P.MUTANTS), ids=lambda m: f"mutant{m}")
def test_planted_mistake_is_caught(mutant):
    """Each deliberately broken oracle build fails at least one pin."""
    assert oracle.load(mutant).mla_oracle_mutant() == mutant
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, oracle.OracleError):
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} ({P.MUTANTS[mutant]}) passed every pin"
