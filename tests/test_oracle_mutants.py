"""Every planted mistake in the oracle must be caught by some pin.

Each mutant is the oracle source compiled with -DORACLE_PLANT=n (one
deliberate error: a dropped term, a wrong sign or index, a transposed operand,
a wrong tie or boundary convention).  If a pin suite let one of them through,
the pins would not be strong enough to trust the oracle.
"""
import numpy as np
import pytest

import oracle as O
import oracle_pins as P


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return str(tmp_path_factory.mktemp("oracle_mutants"))


@pytest.mark.parametrize("name,plant", sorted(O.PLANTS.items(), key=lambda kv: kv[1]))
def test_mutant_is_caught(mutant_dir, name, plant):
    o = O.load(plant, out_dir=mutant_dir)
    assert o.plant == plant
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake '{name}'"


def test_wrong_rule_reproduces_page_numbers(mutant_dir):
    """The tutorial page (section 7) prints [0.44, 0.42, 0.14] for the wrong rule
    'redraw from p after a reject'; the planted variant must reproduce it."""
    o = O.load(O.PLANTS["resample_from_p"], out_dir=mutant_dir)
    want = P.golden("worked_example.json")["wrong_rule_resample_from_p_final"]
    np.testing.assert_allclose(P.wrong_rule_final(o), want, atol=1e-12)
