"""Pins of the float64 oracle against facts the pages and the mathematics fix.

None of these compare the oracle with itself: each check uses an independent
route (numpy/scipy library routines, enumeration, closed forms printed on the
pages, hand-derived worked examples, Monte Carlo against a theorem), chosen so
that a plausible slip in the oracle (a dropped bias term, the wrong previous
token, a swapped p/q, an off-by-one row, an inclusive/exclusive CDF bound)
fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy import special, stats

from oracle import spec_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _zero_w(V, r=1):
    return np.zeros((V, r)), np.zeros((r, V))


# ----------------------------------------------------------------------------- building blocks

def test_inverse_cdf_matches_searchsorted():
    """Inverse CDF = numpy's searchsorted(side='right') on the cumulative sum,
    i.e. the smallest v with F(v) > u; the reported interval contains u."""
    rng = np.random.default_rng(11)
    for V in (1, 2, 5, 37, 1000):
        for _ in range(200):
            p = rng.dirichlet(np.full(V, 0.3))
            u = float(rng.random())
            d = O.inverse_cdf(p, u)
            ref = int(np.searchsorted(np.cumsum(p), u, side="right"))
            if ref < V:
                assert d.token == ref
                assert d.F_lo <= u < d.F_hi
                assert d.dist == pytest.approx(min(u - d.F_lo, d.F_hi - u))
    # u exactly on a breakpoint goes to the next token (strict F(v) > u)
    p = np.array([0.25, 0.25, 0.5])
    assert O.inverse_cdf(p, 0.25).token == 1
    assert O.inverse_cdf(p, 0.5).token == 2
    # zero-probability tokens are never drawn
    p = np.array([0.0, 0.5, 0.0, 0.5, 0.0])
    for u in np.linspace(0.001, 0.999, 101):
        assert O.inverse_cdf(p, u).token in (1, 3)
    # rounding fallback: F never exceeds u -> last token with positive mass
    p = np.array([0.3, 0.3, 0.3999999, 0.0])
    d = O.inverse_cdf(p, 0.99999995)
    assert d.token == 2 and d.fallback


def test_softmax_and_lse_match_scipy():
    rng = np.random.default_rng(12)
    for V in (3, 100, 4096):
        t = rng.normal(0, 3, V)
        for T in (0.6, 1.0, 1.7):
            p, lse = O.target_distribution(t, T)
            np.testing.assert_allclose(p, special.softmax(t / T), rtol=1e-12, atol=1e-300)
            assert lse == pytest.approx(special.logsumexp(t / T), rel=1e-13)
            # W = 0: the Markov draft reduces to a plain tempered softmax
            W1, W2 = _zero_w(V, 4)
            q, lq = O.draft_distribution(t, W1, W2, 0, T)
            np.testing.assert_allclose(q, special.softmax(t / T), rtol=1e-12, atol=1e-300)


def test_temperature_scaling():
    """softmax(z / 0.5) equals softmax(2 z); the bias is scaled together with U."""
    rng = np.random.default_rng(13)
    V, r = 50, 8
    U = rng.normal(0, 2, V)
    W1, W2 = rng.normal(0, 0.5, (V, r)), rng.normal(0, 0.5, (r, V))
    q_half, _ = O.draft_distribution(U, W1, W2, 7, 0.5)
    z = U + np.array([math.fsum(W1[7, i] * W2[i, v] for i in range(r)) for v in range(V)])
    np.testing.assert_allclose(q_half, special.softmax(2.0 * z), rtol=1e-12)


def test_markov_bias_is_row_lookup_times_w2():
    """B(x, .) = W1[x] W2 against an exactly-rounded per-column sum."""
    rng = np.random.default_rng(14)
    V, r = 40, 16
    W1, W2 = rng.normal(0, 1, (V, r)), rng.normal(0, 1, (r, V))
    for x in (0, 5, V - 1):
        ref = np.array([math.fsum(W1[x, i] * W2[i, v] for i in range(r)) for v in range(V)])
        np.testing.assert_allclose(O.markov_bias(W1, W2, x), ref, rtol=0, atol=1e-13)


# ----------------------------------------------------------------------------- golden

def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_golden_verify_worked_examples():
    g = _load("verify_worked.json")
    V, T = g["V"], g["T"]
    W1, W2 = _zero_w(V)
    for case in g["cases"]:
        q_rows = np.log(np.array(case["q_rows"]))
        p_rows = np.log(np.array(case["p_rows"]))
        gamma = q_rows.shape[0]
        d = O.draft_request(q_rows, W1, W2, 0, T, case["u_draft"])
        assert d.tokens.tolist() == case["draft_tokens"], case["name"]
        v = O.verify_request(p_rows, q_rows, W1, W2, 0, T, d.tokens, case["L"],
                             case["u_accept"], case["u_final"])
        assert v.accept_len == case["accept_len"], case["name"]
        assert v.out_tokens.tolist() == case["out_tokens"], case["name"]
        for j in range(gamma):
            exp_a = case["alpha"][j]
            if exp_a is None:
                assert np.isnan(v.alpha[j])
                assert np.isnan(v.ratio[j])
            else:
                assert v.alpha[j] == pytest.approx(exp_a, abs=1e-12)
                assert v.ratio[j] == pytest.approx(case["ratio"][j], abs=1e-12)


def test_golden_markov_worked_examples():
    g = _load("markov_worked.json")
    W1 = np.array(g["W1"])
    W2 = np.array(g["W2_over_ln2"]) * math.log(2.0)
    U = np.log(np.array(g["U_probs"]))
    for case in g["cases"]:
        d = O.draft_request(U, W1, W2, case["anchor"], g["T"], case["u_draft"])
        assert d.tokens.tolist() == case["tokens"]
        np.testing.assert_allclose(d.q_tok, case["q_tok"], rtol=1e-12)


# ----------------------------------------------------------------------------- Markov sampler (P5)

def _joint_by_enumeration(U, W1, W2, x0, T):
    """Probability of every draft sequence, from the factorisation written out
    with scipy's softmax (independent of the oracle's code)."""
    g, V = U.shape
    probs = {}
    for seq in itertools.product(range(V), repeat=g):
        pr, prev = 1.0, x0
        conds = []
        for k, x in enumerate(seq):
            cond = special.softmax((U[k] + W1[prev] @ W2) / T)
            conds.append(cond)
            pr *= cond[x]
            prev = x
        probs[seq] = (pr, conds)
    return probs


def test_markov_draft_deterministic_midpoints():
    """For a chosen token sequence, a uniform at the midpoint of each
    conditional CDF interval must reproduce the sequence exactly."""
    rng = np.random.default_rng(21)
    V, g, r, T = 5, 3, 4, 0.8
    U = rng.normal(0, 1.5, (g, V))
    W1, W2 = rng.normal(0, 0.8, (V, r)), rng.normal(0, 0.8, (r, V))
    joint = _joint_by_enumeration(U, W1, W2, 2, T)
    for seq, (pr, conds) in joint.items():
        us = []
        for k, x in enumerate(seq):
            F = np.cumsum(conds[k])
            lo = F[x - 1] if x > 0 else 0.0
            us.append(0.5 * (lo + F[x]))
        d = O.draft_request(U, W1, W2, 2, T, us)
        assert tuple(d.tokens.tolist()) == seq
        np.testing.assert_allclose(d.q_tok, [conds[k][x] for k, x in enumerate(seq)], rtol=1e-12)


def test_markov_draft_joint_chi_square():
    """Sampled sequences follow prod_k q_k(x_k | x_{k-1}) (chi-square over all 125)."""
    rng = np.random.default_rng(22)
    V, g, r, T = 5, 3, 4, 1.0
    U = rng.normal(0, 0.7, (g, V))
    W1, W2 = rng.normal(0, 0.7, (V, r)), rng.normal(0, 0.7, (r, V))
    joint = _joint_by_enumeration(U, W1, W2, 1, T)
    seqs = list(joint)
    expected_p = np.array([joint[s][0] for s in seqs])
    assert expected_p.sum() == pytest.approx(1.0, abs=1e-12)
    N = 30000
    counts = dict.fromkeys(seqs, 0)
    for _ in range(N):
        d = O.draft_request(U, W1, W2, 1, T, rng.random(g))
        counts[tuple(d.tokens.tolist())] += 1
    obs = np.array([counts[s] for s in seqs], float)
    exp = expected_p * N
    keep = exp >= 5
    obs_k = np.append(obs[keep], obs[~keep].sum())
    exp_k = np.append(exp[keep], exp[~keep].sum())
    pval = stats.chisquare(obs_k, exp_k).pvalue
    assert pval > 1e-3, pval


# ----------------------------------------------------------------------------- losslessness (P1)

@pytest.mark.parametrize("gamma,with_bias", [(1, False), (3, True)])
def test_losslessness_chi_square(gamma, with_bias):
    """The pages' theorem: every emitted token follows the target p.  With
    target rows that do not depend on the prefix, the token emitted at
    position j of a cycle, given the cycle reached j, follows p_j."""
    rng = np.random.default_rng(31 + gamma)
    V, r, T = 6, 3, 1.0
    t = rng.normal(0, 1.0, (gamma + 1, V))
    U = t[:gamma] + rng.normal(0, 1.2, (gamma, V))
    if with_bias:
        W1, W2 = rng.normal(0, 0.8, (V, r)), rng.normal(0, 0.8, (r, V))
    else:
        W1, W2 = _zero_w(V, r)
    N = 25000
    emitted = [[] for _ in range(gamma + 1)]
    for _ in range(N):
        d, v = O.cycle_request(t, U, W1, W2, 0, T, rng.random(gamma), gamma,
                               rng.random(gamma), float(rng.random()))
        for j in range(v.accept_len + 1):
            emitted[j].append(int(v.out_tokens[j]))
    for j in range(gamma + 1):
        obs = np.bincount(emitted[j], minlength=V).astype(float)
        if obs.sum() < 2000:
            continue
        p = special.softmax(t[j] / T)
        pval = stats.chisquare(obs, p * obs.sum()).pvalue
        assert pval > 1e-3, (j, pval)


# ----------------------------------------------------------------------------- alpha (P2)

def test_alpha_closed_forms_and_monte_carlo():
    """alpha = E_{x~q}[min(1, p/q)] = sum min(p, q) = 1 - TV(p, q)."""
    rng = np.random.default_rng(41)
    V, T = 50, 1.0
    W1, W2 = _zero_w(V)
    for _ in range(20):
        t = rng.normal(0, 2, (2, V))
        U = t[:1] + rng.normal(0, 1.5, (1, V))
        p = special.softmax(t[0] / T)
        q = special.softmax(U[0] / T)
        v = O.verify_request(t, U, W1, W2, 0, T, [0], 1, [0.5], 0.5)
        by_expectation = sum(q[x] * min(1.0, p[x] / q[x]) for x in range(V))
        by_tv = 1.0 - 0.5 * np.abs(p - q).sum()
        assert v.alpha[0] == pytest.approx(by_expectation, abs=1e-12)
        assert v.alpha[0] == pytest.approx(by_tv, abs=1e-12)
    # Monte Carlo: the acceptance rate of position 0 is alpha_0
    t = rng.normal(0, 2, (2, 20))
    U = t[:1] + rng.normal(0, 1.0, (1, 20))
    W1, W2 = _zero_w(20)
    N = 20000
    acc = 0
    alpha = None
    for _ in range(N):
        d, v = O.cycle_request(t, U, W1, W2, 0, 1.0, rng.random(1), 1, rng.random(1),
                               float(rng.random()))
        acc += v.accept_len
        alpha = v.alpha[0]
    sigma = math.sqrt(alpha * (1 - alpha) / N)
    assert abs(acc / N - alpha) < 4 * sigma


# ----------------------------------------------------------------------------- E[tau] (P3)

@pytest.mark.parametrize("gamma", [1, 4, 7, 15])
def test_expected_accept_length_iid(gamma):
    """W = 0 and identical rows make acceptances i.i.d. Bernoulli(alpha):
    E[tau] = (1 - alpha^(L+1)) / (1 - alpha) and P(tau >= k+1) = alpha^k."""
    rng = np.random.default_rng(51 + gamma)
    V, T = 8, 1.0
    t_row = rng.normal(0, 1.5, V)
    U_row = t_row + rng.normal(0, 1.0, V)
    t = np.tile(t_row, (gamma + 1, 1))
    U = np.tile(U_row, (gamma, 1))
    W1, W2 = _zero_w(V)
    N = 6000 if gamma < 15 else 3000
    taus = np.empty(N)
    alpha = None
    for i in range(N):
        d, v = O.cycle_request(t, U, W1, W2, 3, T, rng.random(gamma), gamma,
                               rng.random(gamma), float(rng.random()))
        taus[i] = v.accept_len + 1
        alpha = v.alpha[0]
    assert np.allclose(v.alpha[:gamma], alpha)
    e_tau = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert e_tau == pytest.approx(sum(alpha ** k for k in range(gamma + 1)), rel=1e-12)
    assert abs(taus.mean() - e_tau) < 4 * taus.std() / math.sqrt(N)
    for k in range(1, min(gamma, 4) + 1):
        frac = float((taus >= k + 1).mean())
        s = math.sqrt(alpha ** k * (1 - alpha ** k) / N)
        assert abs(frac - alpha ** k) < 4 * s + 1e-9


def test_expected_accept_length_ragged():
    """A verify length L < gamma truncates the geometric sum at L."""
    rng = np.random.default_rng(59)
    V, T, gamma = 8, 1.0, 7
    t_row = rng.normal(0, 1.5, V)
    U_row = t_row + rng.normal(0, 1.0, V)
    t = np.tile(t_row, (gamma + 1, 1))
    U = np.tile(U_row, (gamma, 1))
    W1, W2 = _zero_w(V)
    N = 5000
    for L in (0, 2, 5):
        taus = np.empty(N)
        for i in range(N):
            d, v = O.cycle_request(t, U, W1, W2, 3, T, rng.random(gamma), L,
                                   rng.random(gamma), float(rng.random()))
            taus[i] = v.accept_len + 1
            assert v.accept_len <= L
        a = float(np.sum(np.minimum(special.softmax(t_row / T), special.softmax(U_row / T))))
        e_tau = (1 - a ** (L + 1)) / (1 - a)
        assert abs(taus.mean() - e_tau) < 4 * max(taus.std(), 1e-9) / math.sqrt(N) + 1e-12


# ----------------------------------------------------------------------------- special cases (P6)

def test_identical_distributions_accept_everything():
    """p = q on every verified row: every ratio is 1, alpha = 1, tau = L + 1,
    and the bonus token is the inverse CDF of p_L."""
    rng = np.random.default_rng(61)
    V, gamma, T = 30, 5, 0.7
    U = rng.normal(0, 2, (gamma, V))
    t = np.vstack([U, rng.normal(0, 2, (1, V))])
    W1, W2 = _zero_w(V)
    for L in range(gamma + 1):
        uf = float(rng.random())
        d, v = O.cycle_request(t, U, W1, W2, 0, T, rng.random(gamma), L,
                               rng.random(gamma), uf)
        assert v.accept_len == L
        np.testing.assert_allclose(v.alpha[:L], 1.0, atol=1e-12)
        pL = special.softmax(t[L] / T)
        assert v.out_tokens[L] == int(np.searchsorted(np.cumsum(pL), uf, side="right"))
        assert v.out_tokens[:L].tolist() == d.tokens[:L].tolist()


def test_disjoint_supports_reject_first_and_resample_from_p():
    """Disjoint supports: alpha = 0, the first test rejects, and the residual
    is p itself, so the correction token is the inverse CDF of p_0."""
    rng = np.random.default_rng(62)
    V, gamma, T = 40, 3, 1.0
    A, Bs = np.arange(V) < V // 2, np.arange(V) >= V // 2
    U = np.where(A, rng.normal(0, 1, (gamma, V)), -1e4)
    t = np.where(Bs, rng.normal(0, 1, (gamma + 1, V)), -1e4)
    W1, W2 = _zero_w(V)
    for _ in range(50):
        uf = float(rng.random())
        d, v = O.cycle_request(t, U, W1, W2, 0, T, rng.random(gamma), gamma,
                               rng.random(gamma), uf)
        assert v.accept_len == 0
        assert v.alpha[0] == 0.0
        p0 = special.softmax(t[0] / T)
        assert v.out_tokens[0] == int(np.searchsorted(np.cumsum(p0), uf, side="right"))
        assert v.out_tokens[1:].tolist() == [-1] * gamma


def test_verify_length_zero_is_plain_sampling():
    rng = np.random.default_rng(63)
    V, gamma, T = 100, 4, 1.3
    t = rng.normal(0, 2, (gamma + 1, V))
    U = rng.normal(0, 2, (gamma, V))
    W1, W2 = rng.normal(0, 0.3, (V, 8)), rng.normal(0, 0.3, (8, V))
    for _ in range(30):
        uf = float(rng.random())
        d, v = O.cycle_request(t, U, W1, W2, 5, T, rng.random(gamma), 0, rng.random(gamma), uf)
        p0 = special.softmax(t[0] / T)
        assert v.accept_len == 0
        assert v.out_tokens[0] == int(np.searchsorted(np.cumsum(p0), uf, side="right"))
        assert np.all(np.isnan(v.alpha))


# ----------------------------------------------------------------------------- invariants (P4)

def test_invariants_on_small_workloads():
    from speculative_decoding_draft_04_gb300 import workloads as W
    specs = [W.config("C0"),
             dict(W.config("C2"), V=2056, B=24, name="C2-small"),
             dict(W.config("C4"), V=1032, B=24, gamma=5, name="C4-small")]
    for spec in specs:
        w = W.make_workload(spec, trial=0)
        res = O.cycle(w.f64("target"), w.f64("U"), w.f64("W1"), w.f64("W2"), w.anchor,
                      w.temperature.astype(np.float64), w.u_draft.astype(np.float64),
                      w.verify_len, w.u_accept.astype(np.float64),
                      w.u_final.astype(np.float64))
        for b in range(w.B):
            v, d = res.verify[b], res.draft[b]
            L = int(w.verify_len[b])
            tau = v.accept_len + 1
            assert 1 <= tau <= L + 1
            assert v.out_tokens[:v.accept_len].tolist() == d.tokens[:v.accept_len].tolist()
            assert np.all(v.out_tokens[tau:] == -1)
            assert 0 <= v.out_tokens[v.accept_len] < w.V
            assert np.all((v.alpha[:L] >= 0) & (v.alpha[:L] <= 1 + 1e-12))
            assert np.all(np.isnan(v.alpha[L:]))
            assert np.all((d.q_tok > 0) & (d.q_tok <= 1))
            assert np.all((d.tokens >= 0) & (d.tokens < w.V))
