"""The pages' printed figures, read as context (tests/golden/page_figures.json)."""
import json
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "page_figures.json")


def test_printed_analytic_mean_is_not_the_constant_alpha_law():
    """'spec-verify', section 'Measured': 1.86 is printed as sum_i alpha^i at
    alpha = 0.678, K = 4.  The constant-alpha sum is 1.661 (i = 1..4) or 2.661
    (i = 0..4), so the printed figure cannot pin the oracle; the exact
    per-round law is pinned instead (oracle_pins.pin_analytic_length_law)."""
    g = json.load(open(GOLDEN))["accepted_length_600_rounds"]
    a, K = g["alpha"], g["K"]
    s1 = sum(a ** i for i in range(1, K + 1))
    s0 = sum(a ** i for i in range(0, K + 1))
    assert abs(s1 - 1.661) < 1e-3 and abs(s0 - 2.661) < 1e-3
    assert abs(s1 - g["mean_analytic_printed"]) > 0.1
    assert abs(s0 - g["mean_analytic_printed"]) > 0.1
