"""Pins of the tree oracle (oracle/tree.py; VESSL AI blog, section "gamma
재배분: 체인 대신 트리"): the selection's prefix closure and optimality
(exhaustive search), its tie rule, the reduction of a chain-shaped tree to the
chain draft and verification (oracle/spec_oracle.py), and the losslessness of
the tree verification (chi-square of the emitted tokens against the target)."""
import itertools

import numpy as np
import pytest
from scipy.stats import chisquare

from oracle import spec_oracle as O
from oracle import tree as TR


def random_tree(rng, N, max_depth=6):
    parent = []
    for s in range(N):
        cands = [-1] + [p for p in range(s) if TR.depths(parent + [p])[s] <= max_depth]
        parent.append(int(rng.choice(cands)))
    return parent


def test_survival_halves_by_depth():
    parent = [-1, 0, 1, 0, -1, 4]
    a = TR.survival(parent, np.full(6, 0.5, np.float32))
    assert np.array_equal(a, 2.0 ** -TR.depths(parent).astype(np.float64))


@pytest.mark.parametrize("seed", range(6))
def test_selection_is_prefix_closed_and_optimal(seed):
    rng = np.random.default_rng(seed)
    N = 9
    parent = random_tree(rng, N)
    c = rng.random(N).astype(np.float32)
    a = TR.survival(parent, c).astype(np.float64)
    for n in range(N + 1):
        mask = TR.select(parent, c, n)
        assert mask.sum() == n
        assert all(parent[s] < 0 or mask[parent[s]] for s in range(N) if mask[s])
        best = -1.0
        for sub in itertools.combinations(range(N), n):
            if all(parent[s] < 0 or parent[s] in sub for s in sub):
                best = max(best, sum(a[list(sub)]))
        assert a[mask].sum() == pytest.approx(best, rel=1e-12)


def test_ties_take_the_shallower_node():
    parent = [-1, 0, -1]
    c = np.array([0.5, 1.0, 0.5], np.float32)        # a = 0.5, 0.5, 0.5
    assert list(TR.select(parent, c, 1)) == [True, False, False]
    assert list(TR.select(parent, c, 2)) == [True, False, True]   # depth 1 before depth 2


def _chain_case(rng, V, g, r):
    W1 = rng.normal(0, 0.5, (V, r))
    W2 = rng.normal(0, 0.5, (r, V))
    t = rng.normal(0, 2, (g + 1, V))
    U = t[:g] + rng.normal(0, 1, (g, V))
    return W1, W2, t, U


@pytest.mark.parametrize("seed", range(5))
def test_chain_tree_is_the_chain(seed):
    rng = np.random.default_rng(10 + seed)
    V, g, r = 60, 5, 4
    W1, W2, t, U = _chain_case(rng, V, g, r)
    parent = [-1] + list(range(g - 1))
    mask = np.ones(g, bool)
    ud, ua, uf = rng.random(g), rng.random(g), float(rng.random())
    d = TR.draft_request(U, W1, W2, 3, 0.9, parent, mask, ud)
    c = O.draft_request(U, W1, W2, 3, 0.9, ud)
    assert np.array_equal(d.tokens, c.tokens) and np.allclose(d.q_tok, c.q_tok, rtol=1e-14)
    v = TR.verify_request(t, U, W1, W2, 3, 0.9, parent, mask, d.tokens, ua, uf, g)
    cv = O.verify_request(t, U, W1, W2, 3, 0.9, c.tokens, g, ua, uf)
    assert len(v.path) == cv.accept_len
    assert np.array_equal(v.out_tokens, cv.out_tokens)


@pytest.mark.parametrize("m", [1, 2, 3])
def test_root_candidates_are_lossless(m):
    """Root with m independent candidates: the first emitted token follows the
    target's p (chi-square over 20000 cycles)."""
    rng = np.random.default_rng(20 + m)
    V, r, trials = 5, 2, 20000
    W1 = np.zeros((V, r))
    W2 = np.zeros((r, V))
    t = np.array([[1.2, -0.3, 0.4, 2.0, -1.0], [0, 0, 0, 0, 0]] + [[0] * V] * m, float)
    U = np.array([[0.1, 1.5, -0.5, 0.2, 0.9]])     # q differs from p
    parent = [-1] * m
    mask = np.ones(m, bool)
    counts = np.zeros(V)
    for _ in range(trials):
        ud, ua, uf = rng.random(m), rng.random(m), float(rng.random())
        d = TR.draft_request(U, W1, W2, 0, 1.0, parent, mask, ud)
        v = TR.verify_request(t, U, W1, W2, 0, 1.0, parent, mask, d.tokens, ua, uf, 1)
        counts[v.out_tokens[0]] += 1
    p, _ = O.target_distribution(t[0], 1.0)
    assert chisquare(counts, p * trials).pvalue > 1e-3


def test_two_level_tree_is_lossless():
    """Root with 2 candidates, each with 2 candidates of its own; target rows
    that depend only on the path: the first two emitted tokens follow
    p_root(a) p_a(b)."""
    rng = np.random.default_rng(30)
    V, r, trials = 4, 2, 30000
    W1 = rng.normal(0, 1.0, (V, r))
    W2 = rng.normal(0, 1.0, (r, V))
    U = rng.normal(0, 1, (2, V))
    root_t = rng.normal(0, 1, V)
    child_t = rng.normal(0, 1.5, (V, V))              # target after token a
    parent = [-1, -1, 0, 0, 1, 1]
    mask = np.ones(6, bool)
    counts = np.zeros((V, V))
    for _ in range(trials):
        ud, ua, uf = rng.random(6), rng.random(6), float(rng.random())
        d = TR.draft_request(U, W1, W2, 1, 1.0, parent, mask, ud)
        t = np.zeros((7, V))
        t[0] = root_t
        for s in range(6):
            t[1 + s] = child_t[d.tokens[s]]
        v = TR.verify_request(t, U, W1, W2, 1, 1.0, parent, mask, d.tokens, ua, uf, 2)
        if len(v.path) >= 1:
            counts[v.out_tokens[0], v.out_tokens[1]] += 1
        else:
            # the first token came from the root's residual; draw the second from the target
            a = v.out_tokens[0]
            pa, _ = O.target_distribution(child_t[a], 1.0)
            counts[a, int(np.searchsorted(np.cumsum(pa), rng.random(), side="right"))] += 1
    pr, _ = O.target_distribution(root_t, 1.0)
    expect = np.array([pr[a] * O.target_distribution(child_t[a], 1.0)[0] for a in range(V)])
    assert chisquare(counts.ravel(), expect.ravel() * trials).pvalue > 1e-3


def test_path_invariants():
    rng = np.random.default_rng(40)
    V, g, r = 50, 4, 4
    W1, W2, _, U = _chain_case(rng, V, g, r)
    for _ in range(20):
        parent = random_tree(rng, 10, max_depth=g)
        mask = TR.select(parent, rng.random(10).astype(np.float32), 7)
        t = rng.normal(0, 2, (11, V))
        d = TR.draft_request(U, W1, W2, 0, 1.0, parent, mask, rng.random(10))
        assert np.all((d.tokens >= 0) == mask)
        v = TR.verify_request(t, U, W1, W2, 0, 1.0, parent, mask, d.tokens, rng.random(10),
                              float(rng.random()), g)
        prev = -1
        for s in v.path:
            assert mask[s] and parent[s] == prev
            prev = s
        assert 0 <= v.out_tokens[len(v.path)] < V and np.all(v.out_tokens[len(v.path) + 1:] == -1)
