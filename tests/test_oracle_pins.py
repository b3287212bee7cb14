"""The CPU oracle against its pins (brute force, closed forms, analytic law,
library routines, greedy identity); see ``oracle_pins.py`` for what each pin
ties the oracle to."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_analytic_law_at_single_sequence_workload(orc):
    """600 rounds at V=32000, K=4 (the single-sequence workload): the accepted
    length tracks the exact per-round law; the measured alpha is reported."""
    got, law, alpha = oracle_pins.pin_analytic_length_law(orc, rounds=600, V=32000)
    assert 0.55 < alpha < 0.8, alpha
