"""Pins of the oracle's boundary bookkeeping: the distance of every consumed
uniform to its decision boundary (``Draw.dist``, ``VerifyResult.ratio_dist``)
and the per-request minimum ``CycleResult.row_dmin``.  These decide which
GPU/oracle mismatches the parity gate excuses (a request counts as "near a
boundary" when a consumed uniform lies within 1e-6 of a boundary), so they
are checked here against an independent route:

* distributions from ``scipy.special.softmax`` (not the oracle's softmax);
* the draws' tokens from ``numpy.searchsorted`` over the CDF breakpoints;
* the distance of an inverse-CDF draw as the brute-force minimum of |u - F(v)|
  over EVERY breakpoint F(-1) = 0, F(0), ..., F(V-1) (the oracle only looks at
  the two ends of the chosen interval);
* the ratio test's distance |u - p(x)/q(x)| for each test up to and including
  the first reject (the SpecDec blog, "수락 규칙": the tests stop there), and no
  distance for tests that are never run.

Planted uniforms make the minimum come from a draft draw, from a ratio test
and from the final (correction or bonus) draw in turn, so that a dropped
term, a wrong index or a test counted past the first reject fails one case.
"""
from __future__ import annotations

import numpy as np
import pytest
from scipy.special import softmax

from oracle import spec_oracle as O


def _problem(seed, V=12, r=4, g=4, w_sd=0.6):
    rng = np.random.default_rng([77, seed])
    t = rng.normal(0, 1.5, size=(g + 1, V))
    U = t[:g] + rng.normal(0, 1.0, size=(g, V))
    W1 = rng.normal(0, w_sd, size=(V, r))
    W2 = rng.normal(0, w_sd, size=(r, V))
    anchor = int(rng.integers(0, V))
    T = float(rng.choice([0.7, 1.0]))
    u_draft = rng.uniform(0.02, 0.98, size=g)
    u_acc = rng.uniform(0.02, 0.98, size=g)
    u_fin = float(rng.uniform(0.02, 0.98))
    return t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin


def _brute_dist(probs, u):
    """Token by searchsorted and distance to the nearest CDF breakpoint."""
    F = np.concatenate([[0.0], np.cumsum(probs)])
    tok = int(np.searchsorted(F[1:], u, side="right"))
    return tok, float(np.min(np.abs(u - F)))


def _independent(t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin, L):
    """Every consumed uniform's boundary distance, recomputed with scipy."""
    g = U.shape[0]
    prev = anchor
    toks, qrows, ddist = [], [], []
    for k in range(g):
        q = softmax((U[k] + W1[prev] @ W2) / T)
        tok, d = _brute_dist(q, u_draft[k])
        toks.append(tok)
        qrows.append(q)
        ddist.append(d)
        prev = tok
    prows = [softmax(t[j] / T) for j in range(L + 1)]
    rdist = np.full(g, np.inf)
    n = L
    for j in range(L):
        ratio = prows[j][toks[j]] / qrows[j][toks[j]]
        rdist[j] = abs(u_acc[j] - ratio)
        if not (u_acc[j] < ratio):
            n = j
            break
    if n < L:
        res = np.maximum(0.0, prows[n] - qrows[n])
        fin = res / res.sum()
    else:
        fin = prows[L]
    ftok, fdist = _brute_dist(fin, u_fin)
    return dict(tokens=np.array(toks), ddist=np.array(ddist), rdist=rdist, n=n,
                ftok=ftok, fdist=fdist, qrows=qrows, prows=prows, fin=fin)


def _oracle(t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin, L):
    res = O.cycle(t[None], U[None], W1, W2, [anchor], [T], u_draft[None], [L], u_acc[None], [u_fin])
    return res


def _check_against(res, ind):
    d, v = res.draft[0], res.verify[0]
    np.testing.assert_array_equal(d.tokens, ind["tokens"])
    np.testing.assert_allclose(d.dist, ind["ddist"], rtol=1e-9, atol=1e-15)
    fin_r = np.isfinite(ind["rdist"])
    np.testing.assert_array_equal(np.isfinite(v.ratio_dist), fin_r)
    np.testing.assert_allclose(v.ratio_dist[fin_r], ind["rdist"][fin_r], rtol=1e-9, atol=1e-15)
    assert v.accept_len == ind["n"]
    assert v.final.token == ind["ftok"]
    assert v.final.dist == pytest.approx(ind["fdist"], rel=1e-9, abs=1e-15)
    want = min(float(np.min(ind["ddist"])), float(np.min(ind["rdist"])), ind["fdist"])
    assert res.row_dmin(0) == pytest.approx(want, rel=1e-9, abs=1e-15)
    return want


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("L", [0, 2, 4])
def test_distances_match_brute_force(seed, L):
    args = _problem(seed)
    res = _oracle(*args, L)
    _check_against(res, _independent(*args, L))


def test_minimum_from_a_planted_draft_draw():
    t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin = _problem(3)
    L = 4
    ind = _independent(t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin, L)
    # put draw k = 2 just above the CDF breakpoint below its token
    k = 2
    F = np.concatenate([[0.0], np.cumsum(ind["qrows"][k])])
    tok = ind["tokens"][k]
    u_draft = u_draft.copy()
    u_draft[k] = F[tok] + 3e-9 if tok > 0 else F[1] - 3e-9
    ind = _independent(t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin, L)
    res = _oracle(t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin, L)
    want = _check_against(res, ind)
    assert want == pytest.approx(3e-9, rel=1e-5)
    assert int(np.argmin(res.draft[0].dist)) == k


def _ratios(ind, L):
    toks = ind["tokens"]
    return np.array([ind["prows"][j][toks[j]] / ind["qrows"][j][toks[j]] for j in range(L)])


def _seed_with(cond, L):
    for seed in range(100):
        args = _problem(seed)
        ind = _independent(*args, L)
        r = _ratios(ind, L)
        if cond(r):
            return args, ind, r
    raise AssertionError("no seed satisfies the condition")


def test_minimum_from_a_planted_ratio_test():
    L = 4
    args, ind, ratios = _seed_with(lambda r: r[1] < 0.9, L)
    t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin = args
    u_acc = np.minimum(ratios, 1.0) * 0.5            # accept every test by a wide margin
    u_acc[1] = ratios[1] - 2e-9                      # test 1 accepted, 2e-9 below its ratio
    ind = _independent(t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin, L)
    res = _oracle(t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin, L)
    want = _check_against(res, ind)
    assert res.verify[0].accept_len == L
    assert want == pytest.approx(2e-9, rel=1e-5)
    assert int(np.argmin(res.verify[0].ratio_dist)) == 1


def test_tests_after_the_first_reject_are_not_counted():
    L = 4
    args, ind, ratios = _seed_with(lambda r: r[1] < 0.9 and r[3] < 1.0, L)
    t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin = args
    u_acc = np.minimum(ratios, 1.0) * 0.5
    u_acc[1] = min(0.999, ratios[1] + 0.05)          # reject at position 1
    u_acc[3] = ratios[3]                             # never run: exactly on its ratio
    ind = _independent(t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin, L)
    res = _oracle(t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin, L)
    _check_against(res, ind)
    v = res.verify[0]
    assert v.accept_len == 1
    assert np.isfinite(v.ratio_dist[:2]).all() and not np.isfinite(v.ratio_dist[2:]).any()
    assert res.row_dmin(0) > 1e-6


@pytest.mark.parametrize("kind", ["residual", "bonus"])
def test_minimum_from_a_planted_final_draw(kind):
    t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin = _problem(11)
    L = 3
    ind = _independent(t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin, L)
    toks = ind["tokens"]
    ratios = np.array([ind["prows"][j][toks[j]] / ind["qrows"][j][toks[j]] for j in range(L)])
    u_acc = np.minimum(ratios, 1.0) * 0.5             # accept everything ...
    if kind == "residual":
        j = int(np.argmin(ratios))
        assert ratios[j] < 0.9
        u_acc[j] = min(0.99, ratios[j] + 0.05)        # ... except test j (reject)
    ind = _independent(t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin, L)
    F = np.concatenate([[0.0], np.cumsum(ind["fin"])])
    v0 = len(F) // 2
    u_fin = F[v0] - 4e-9
    ind = _independent(t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin, L)
    res = _oracle(t, U, W1, W2, anchor, T, u_draft, u_acc, u_fin, L)
    want = _check_against(res, ind)
    assert res.verify[0].final_kind == kind
    assert want == pytest.approx(4e-9, rel=1e-5)
    assert res.verify[0].final.dist == pytest.approx(4e-9, rel=1e-5)
