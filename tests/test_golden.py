"""The tail-rate closed form and test thresholds against the numbers the pages print.

Megatron-LM PR 8370, "Problem": a draw from a row [0, -D, ..., -D] misses token 0 with
probability (V-1) r / (1 + (V-1) r), r = e^-D; the table's "expected" column and the "Tests"
section's "expected 34" at 262k draws follow from it.  The printed draw counts carry two
significant digits, so each expected count must be reproduced by some draw count that
rounds to the printed one.
"""
import math

from scipy import stats


def miss_prob(V, r):
    return (V - 1) * r / (1 + (V - 1) * r)


def test_closed_form_reproduces_page_expected_column(golden):
    tab = golden["tail_table"]
    V = tab["V"]
    for row in tab["rows"]:
        p = miss_prob(V, row["r"])
        n_lo = row["draws_printed"] * 0.975          # counts printed as 2.0e5 / 1.0e6
        n_hi = row["draws_printed"] * 1.025
        assert n_lo * p - 0.5 <= row["expected_printed"] <= n_hi * p + 0.5
        # and the fp64-noise column is inside the two-sided 1e-6 Poisson interval around it
        lo = stats.poisson.ppf(5e-7, row["expected_printed"])
        hi = stats.poisson.isf(5e-7, row["expected_printed"])
        assert lo <= row["fp64_noise_observed"] <= hi


def test_closed_form_reproduces_expected_34(golden):
    t = golden["tail_test"]
    mu = t["draws"] * miss_prob(golden["tail_table"]["V"], t["nonvacuity_r"])
    assert round(mu) == t["nonvacuity_expected_printed"]
    # observed 0 lies below the interval: the fp32 non-vacuity check has power
    assert stats.poisson.ppf(t["interval_two_sided_alpha"] / 2, mu) > 0


def test_chi_square_threshold(golden):
    c = golden["chi_square"]
    assert round(stats.chi2.isf(1e-6, c["dof"]), 1) == c["threshold_printed"]
    assert c["dof"] == c["tokens"] - 1


def test_wide_range_constants(golden):
    w = golden["wide_noise_range"]
    assert f"{-math.log1p(-2.0 ** -53):.1e}" == f"{w['E_min_printed']:.1e}"
    assert f"{53 * math.log(2):.1f}" == f"{w['E_max_printed']:.1f}"
