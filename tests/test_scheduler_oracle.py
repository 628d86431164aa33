"""Pins of the confidence-head / prefix-scheduler oracle (oracle/scheduler.py)
against hand-worked cases (tests/golden/schedule_worked.json), closed forms of
the sigmoid, exhaustive search over every allocation on tiny batches, and the
causality property of the early stop (DSpark review, sections 2.1 and 2.2)."""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import scheduler as S

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = json.load(open(os.path.join(HERE, "golden", "schedule_worked.json")))["cases"]
UNIT = 2.0 ** -S.TAU_UNIT_BITS


@pytest.mark.parametrize("case", GOLD, ids=[c["what"][:40] for c in GOLD])
def test_golden_schedules(case):
    conf = np.asarray(case["conf"], dtype=np.float32)
    a = S.survival(conf)
    ell, B, tau, theta = S.schedule(a, np.asarray(case["sps"]))
    assert list(ell) == case["ell"]
    assert B == case["B"]
    assert tau * UNIT == pytest.approx(case["tau"], abs=1e-6)
    assert theta == pytest.approx(case["theta"], rel=1e-6)


def test_golden_trace_is_theta_along_the_sorted_pool():
    case = GOLD[0]
    conf = np.asarray(case["conf"], dtype=np.float64)
    # sorted pool by hand: a = 0.9, 0.8, 0.45, 0.24
    pool = sorted([conf[0, 0], conf[1, 0], conf[0, 0] * conf[0, 1], conf[1, 0] * conf[1, 1]],
                  reverse=True)
    tau, trace = 2.0, [2.0 * case["sps"][2]]
    for m, av in enumerate(pool[:3]):
        tau += av
        trace.append(tau * case["sps"][3 + m])
    assert trace == pytest.approx(case["trace"], rel=1e-7)


# ------------------------------------------------------------- confidence head

@pytest.mark.parametrize("c", [0.5, 0.75, 0.1, 0.999, 1e-4])
def test_confidence_inverts_the_logit(c):
    z = math.log(c / (1 - c))
    # the logit split between the hidden part and the embedding part
    h = np.array([z * 0.25, 1.0])
    e = np.array([2.0, 0.0, -1.0])
    w = np.array([1.0, 0.0, z * 0.75, 5.0, z * 0.75])   # z/4 + 2(0.75z) - 0.75z = z
    assert S.confidence(h, e, w) == pytest.approx(c, rel=1e-13)


def test_confidence_zero_weights_is_one_half():
    rng = np.random.default_rng(0)
    assert S.confidence(rng.normal(size=7), rng.normal(size=3), np.zeros(10)) == 0.5


def test_confidence_uses_the_previous_token_row():
    """c for draft row j reads W1[x_j], x_0 = the anchor: with the hidden part
    zero, c reveals which embedding row was read."""
    R, g, d, V, r = 2, 3, 4, 6, 2
    hidden = np.zeros((R, g, d))
    W1 = np.zeros((V, r))
    W1[:, 0] = np.arange(V) - 2.5          # row v has logit v - 2.5 under w_e = (1, 0)
    w = np.zeros(d + r)
    w[d] = 1.0
    anchor = np.array([4, 0])
    tokens = np.array([[1, 5, 2], [3, 3, 0]])
    c = S.confidences(hidden, W1, w, anchor, tokens)
    prev = np.array([[4, 1, 5], [0, 3, 3]])
    assert np.allclose(c, 1 / (1 + np.exp(-(prev - 2.5))), rtol=1e-14, atol=0)


def test_confidence_symmetry():
    rng = np.random.default_rng(1)
    h, e, w = rng.normal(size=5), rng.normal(size=3), rng.normal(size=8)
    assert S.confidence(h, e, w) + S.confidence(h, e, -w) == pytest.approx(1.0, abs=1e-15)


# ------------------------------------------------------------------ survival

def test_survival_halves():
    a = S.survival(np.full((2, 6), 0.5, np.float32))
    assert np.array_equal(a[0], 2.0 ** -np.arange(1, 7))


def test_survival_is_nonincreasing_and_one_stays():
    rng = np.random.default_rng(2)
    c = rng.random((50, 16)).astype(np.float32)
    c[:, 3] = 1.0
    a = S.survival(c)
    assert np.all(np.diff(a.astype(np.float64), axis=1) <= 0)
    assert np.array_equal(a[:, 3], a[:, 2])


# ------------------------------------------------------------------ scheduler

def _cost_table(R, gamma, t0=42.0, knee=None):
    """SPS = 1000 / t(B), t(B) = sqrt(t0^2 + (B t1)^2): convex increasing."""
    knee = knee or R * (1 + gamma / 2)
    t1 = t0 / knee
    B = np.arange(R * (1 + gamma) + 1, dtype=np.float64)
    return 1000.0 / np.sqrt(t0 * t0 + (B * t1) ** 2)


def _theta_of(ell, a, sps):
    B, tau = S.batch_and_tau(ell, a)
    return (tau * UNIT) * sps[B]


def test_batch_and_tau_identities():
    rng = np.random.default_rng(3)
    for _ in range(20):
        R, g = rng.integers(1, 9), rng.integers(1, 9)
        a = S.survival(rng.random((R, g)).astype(np.float32))
        ell, B, tau, theta = S.schedule(a, _cost_table(R, g))
        B2, tau2 = S.batch_and_tau(ell, a)
        assert (B, tau) == (B2, tau2)
        assert B == R + ell.sum() and np.all((ell >= 0) & (ell <= g))
        assert theta == (tau * UNIT) * _cost_table(R, g)[B]


def test_greedy_is_optimal_for_each_batch_size():
    """For a fixed B the top-m survival probabilities maximise tau (exhaustive
    search over every l vector)."""
    rng = np.random.default_rng(4)
    for _ in range(12):
        R, g = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        a = S.survival(rng.random((R, g)).astype(np.float32))
        best = {}
        for ell in itertools.product(range(g + 1), repeat=R):
            B, tau = S.batch_and_tau(np.array(ell), a)
            best[B] = max(best.get(B, -1), tau)
        for m in range(R * g + 1):
            flat = sorted(((-float(a[r, j]), r, j) for r in range(R) for j in range(g)))[:m]
            tau_greedy = (R << S.TAU_UNIT_BITS) + sum(S.tau_units(-k) for k, _, _ in flat)
            assert tau_greedy == best[R + m]


def test_early_stop_finds_the_global_optimum_on_a_convex_cost_curve():
    """With t(B) = 1/SPS(B) convex and increasing, Theta along the greedy order
    rises then falls, so the first decrease is the best allocation overall."""
    rng = np.random.default_rng(5)
    for trial in range(25):
        R, g = int(rng.integers(1, 4)), int(rng.integers(1, 5))
        a = S.survival(rng.random((R, g)).astype(np.float32))
        sps = _cost_table(R, g, knee=float(rng.uniform(0.5, 3.0)) * R)
        ell, B, tau, theta = S.schedule(a, sps)
        brute = max(_theta_of(np.array(e), a, sps)
                    for e in itertools.product(range(g + 1), repeat=R))
        assert theta == pytest.approx(brute, rel=1e-13), trial


def test_stop_depends_only_on_the_processed_prefix():
    """Changing candidates ranked after the stop (keeping them below the first
    rejected one) cannot change the allocation."""
    rng = np.random.default_rng(6)
    n_checked = 0
    for _ in range(40):
        R, g = 6, 5
        c = rng.random((R, g)).astype(np.float32) * 0.5 + 0.5
        a = S.survival(c)
        sps = _cost_table(R, g)
        ell, B, tau, theta = S.schedule(a, sps)
        m = int(ell.sum())
        if m == R * g:
            continue
        order = sorted(((-float(a[r, j]), r, j) for r in range(R) for j in range(g)))
        _, r0, j0 = order[m]                       # the first rejected candidate
        a2 = a.copy()
        for r in range(R):
            for j in range(g):
                if j > ell[r] or (j == ell[r] and (r, j) != (r0, j0)):
                    a2[r, j] = np.float32(a[r0, j0] * rng.random() ** (1 + j - ell[r]))
        a2 = np.minimum.accumulate(a2, axis=1)
        ell2, B2, tau2, theta2 = S.schedule(a2, sps)
        assert np.array_equal(ell, ell2) and (B, tau, theta) == (B2, tau2, theta2)
        n_checked += 1
    assert n_checked > 10


def test_ties_go_to_the_lower_request():
    a = S.survival(np.full((3, 2), 0.5, np.float32))
    sps = np.ones(6)                     # the table ends at B = 5: two admissions fit
    ell, B, tau, _ = S.schedule(a, sps)
    assert list(ell) == [1, 1, 0] and B == 5


def test_certain_tokens_are_always_worth_a_flat_table():
    a = S.survival(np.ones((4, 3), np.float32))
    ell, B, tau, theta = S.schedule(a, np.ones(17))
    assert list(ell) == [3, 3, 3, 3] and tau * UNIT == 16.0 and theta == 16.0


def test_tau_units_are_exact_floors():
    for a in (0.0, 1.0, 0.5, 2.0 ** -40, np.float32(0.3), np.float32(1 - 2 ** -24)):
        assert S.tau_units(a) == math.floor(float(np.float32(a)) * 2.0 ** 36)
    assert S.tau_units(1.0) == 1 << 36
