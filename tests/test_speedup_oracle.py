"""Pins of the operating-point oracle (oracle/speedup_model.py) against the
blog's worked values (tests/golden/speedup_worked.json) and closed forms that
the oracle does not use (it sums and enumerates)."""
import json
import math
import os

import numpy as np
import pytest

from oracle import speedup_model as M

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = json.load(open(os.path.join(HERE, "golden", "speedup_worked.json")))["cases"]


def test_golden_worked_operating_points():
    for case in GOLD:
        a, c = case["alpha"], case["c"]
        if "s_max" in case:
            g, s = M.optimal_gamma(a, c, 400)
            assert abs(s - case["s_max"]) <= case["s_tol"], case
            if "gamma_star" in case:
                assert g == case["gamma_star"], (g, case)
        if "flat_range" in case:
            _, s_best = M.optimal_gamma(a, c, 400)
            lo, hi = case["flat_range"]
            for g in range(lo, hi + 1):
                assert M.speedup(a, c, g) >= (1 - case["flat_tol"]) * s_best, g
            # and the range is maximal: its neighbours fall outside
            assert M.speedup(a, c, lo - 1) < (1 - case["flat_tol"]) * s_best
            assert M.speedup(a, c, hi + 1) < (1 - case["flat_tol"]) * s_best
        if "bound" in case:
            assert M.speedup_bound(a, c) == pytest.approx(case["bound"])


@pytest.mark.parametrize("alpha", [0.0, 0.3, 0.8, 0.95, 0.999])
@pytest.mark.parametrize("gamma", [0, 1, 5, 30])
def test_expected_tau_closed_form(alpha, gamma):
    closed = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert M.expected_tau(alpha, gamma) == pytest.approx(closed, rel=1e-12)


def test_expected_tau_by_simulation():
    """i.i.d. Bernoulli(alpha) acceptance with gamma drafts: tau = accepted
    prefix + 1."""
    rng = np.random.default_rng(0)
    for alpha, gamma in ((0.7, 5), (0.9, 12)):
        acc = rng.random((200000, gamma)) < alpha
        n = np.where(acc.all(1), gamma, np.argmin(acc, axis=1))
        tau = n + 1
        se = tau.std() / math.sqrt(len(tau))
        assert abs(tau.mean() - M.expected_tau(alpha, gamma)) < 4 * se


@pytest.mark.parametrize("alpha,c", [(0.5, 0.1), (0.8, 0.05), (0.3, 0.4), (0.95, 0.2)])
def test_gamma_one_and_break_even(alpha, c):
    assert M.speedup(alpha, c, 1) == pytest.approx((1 + alpha) / (c + 1), rel=1e-14)
    assert (M.speedup(alpha, c, 1) > 1) == (alpha > c)


def test_bound_holds_on_a_grid():
    for alpha in np.linspace(0.05, 0.99, 12):
        for c in np.linspace(0.01, 1.0, 12):
            b = M.speedup_bound(alpha, c)
            for g in (1, 2, 4, 8, 16, 64):
                assert M.speedup(alpha, c, g) <= b * (1 + 1e-12)


@pytest.mark.parametrize("alpha,c", [(0.8, 0.05), (0.95, 0.05), (0.6, 0.02), (0.9, 0.3)])
def test_unimodal_and_continuous_optimum_brackets_the_integer_one(alpha, c):
    s = [M.speedup(alpha, c, g) for g in range(1, 300)]
    k = int(np.argmax(s))
    assert all(np.diff(s[:k + 1]) > 0) and all(np.diff(s[k:]) < 0)
    gc = M.continuous_optimum(alpha, c)
    assert abs(M.stationarity(alpha, c, gc)) < 1e-9
    assert k + 1 - 1 <= gc <= k + 1 + 1           # the integer optimum is a neighbour
    # the stationarity condition's left side strictly decreases
    # (strictly, while alpha^{gamma+1} is still resolved next to c)
    xs = [x for x in np.linspace(0, 80, 400) if alpha ** (x + 1) > 1e-9]
    lhs = [M.stationarity(alpha, c, x) for x in xs]
    assert all(np.diff(lhs) < 0)


def test_compute_ratio_exceeds_one():
    for alpha in (0.2, 0.6, 0.9, 0.99):
        for c_hat in (0.0, 0.01, 0.1):
            for g in (1, 3, 8):
                r = M.compute_ratio(alpha, c_hat, g)
                assert r > 1
                assert r == pytest.approx((1 - alpha) * (g * c_hat + g + 1) / (1 - alpha ** (g + 1)))


def test_measured_statistics():
    alpha = np.array([[0.5, 0.7, np.nan], [0.9, np.nan, np.nan]])
    L = np.array([2, 1])
    assert M.measured_alpha(alpha, L) == pytest.approx((0.5 + 0.7 + 0.9) / 3)
    assert M.measured_tau(np.array([2, 0, -1])) == pytest.approx(2.0)
