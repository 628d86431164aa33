"""Pins of the RNN head oracle (oracle/rnn_head.py, DSpark review section 1.2
"RNN head"): bf16 rounding against float32 bit patterns, closed forms of the
gated update, the reduction to the Markov head (oracle/spec_oracle.py) when
the factor ignores the state, saturated gates, and the verification's
explicit factor rows."""
import math

import numpy as np
import pytest
from scipy.special import softmax

from oracle import rnn_head as H
from oracle import spec_oracle as O


def test_round_bf16_nearest_and_ties_to_even():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 1, 5000), rng.normal(0, 1e-3, 1000), [0.0, 1.0, -2.5]])
    r = H.round_bf16(x)
    bits = r.astype(np.float32).view(np.uint32)
    assert np.all(bits & 0xFFFF == 0)                               # representable in bf16
    # nearest: no other bf16 neighbour is closer
    up = (bits + 0x10000).view(np.float32).astype(np.float64)
    dn = (bits - 0x10000).view(np.float32).astype(np.float64)
    nz = r != 0
    assert np.all(np.abs(x - r)[nz] <= np.abs(x - up)[nz]) and np.all(np.abs(x - r)[nz] <= np.abs(x - dn)[nz])
    # exact midpoints go to the even neighbour
    a = np.float32(1.0).view(np.uint32)
    lo = np.array([a, a + 0x10000], np.uint32).view(np.float32).astype(np.float64)
    mid = (lo[0] + lo[1]) / 2                                       # 1 + 2^-8: tie, 1.0 is even
    assert H.round_bf16(mid) == 1.0
    mid2 = (lo[1] + (a + 0x20000).view(np.float32).astype(np.float64)) / 2
    assert H.round_bf16(mid2) == np.array(a + 0x20000, np.uint32).view(np.float32)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_first_step_closed_form(dtype):
    """Wr = 0: a_1 = tanh(h_o) and s_1 = (1 - sigmoid(h_g)) tanh(h_c) (s_0 = 0)."""
    rng = np.random.default_rng(1)
    r = 8
    hp = rng.normal(0, 1, (3, r))
    a, s = H.rnn_step(np.zeros((3 * r, 2 * r)), np.zeros(r), rng.normal(size=r), hp, dtype)
    sg = 1 / (1 + np.exp(-hp[0]))
    assert np.array_equal(a, H.round_store(np.tanh(hp[2]), dtype))
    assert np.array_equal(s, H.round_store((1 - sg) * np.tanh(hp[1]), dtype))


def test_gates_are_row_dot_products():
    rng = np.random.default_rng(2)
    r = 4
    Wr = rng.normal(size=(3 * r, 2 * r))
    s, e, hp = rng.normal(size=r), rng.normal(size=r), rng.normal(size=(3, r))
    pre = H.gates(Wr, s, e, hp)
    ref = (Wr[:, :r] @ s + Wr[:, r:] @ e).reshape(3, r) + hp
    assert np.allclose(pre, ref, rtol=1e-13, atol=1e-14)


def test_reduces_to_the_markov_head_when_the_factor_ignores_the_state():
    """W_o = [0 | kappa I], h_o = 0: a_k = round(tanh(kappa W1[x_{k-1}])) whatever
    the state, i.e. the Markov head with W1' = round(tanh(kappa W1))."""
    rng = np.random.default_rng(3)
    V, r, g, kappa = 50, 8, 5, 3.0
    W1 = H.round_bf16(rng.normal(0, 0.3, (V, r)))
    W2 = H.round_bf16(rng.normal(0, 0.5, (r, V)))
    Wr = rng.normal(0, 0.5, (3 * r, 2 * r))
    Wr[2 * r:, :r] = 0.0
    Wr[2 * r:, r:] = kappa * np.eye(r)
    hp = rng.normal(0, 1, (g, 3, r))
    hp[:, 2] = 0.0
    U = rng.normal(0, 2, (g, V))
    u = rng.random(g)
    d, a_rows = H.rnn_draft_request(U, W1, W2, Wr, hp, 7, 0.8, u, "bf16")
    W1m = H.round_bf16(np.tanh(kappa * W1))
    m = O.draft_request(U, W1m, W2, 7, 0.8, u)
    assert np.array_equal(d.tokens, m.tokens)
    assert np.array_equal(d.q_tok, m.q_tok) and np.array_equal(d.lse_q, m.lse_q)
    prevs = [7] + list(m.tokens[:-1])
    assert np.array_equal(a_rows, W1m[prevs])


def test_saturated_update_gate_keeps_the_state_at_zero():
    """sigmoid(h_g) = 1 exactly: s_k = s_{k-1} = 0, so with W_o reading only the
    state the bias is zero and q = softmax(U / T)."""
    rng = np.random.default_rng(4)
    V, r, g = 30, 4, 4
    W1 = rng.normal(size=(V, r))
    W2 = rng.normal(size=(r, V))
    Wr = np.zeros((3 * r, 2 * r))
    Wr[:r] = rng.normal(size=(r, 2 * r)) * 1e-3
    Wr[r:2 * r] = rng.normal(size=(r, 2 * r))
    Wr[2 * r:, :r] = np.eye(r)
    hp = np.zeros((g, 3, r))
    hp[:, 0] = 60.0                                   # 1 - sigmoid(60) < 2^-53
    hp[:, 1] = rng.normal(size=(g, r))
    U = rng.normal(0, 2, (g, V))
    u = rng.random(g)
    d, a_rows = H.rnn_draft_request(U, W1, W2, Wr, hp, 3, 1.3, u, "f32")
    assert np.all(a_rows == 0.0)
    for k in range(g):
        q = softmax(U[k] / 1.3)
        assert d.q_tok[k] == pytest.approx(q[d.tokens[k]], rel=1e-12)
        assert d.tokens[k] == int(np.searchsorted(np.cumsum(q), u[k], side="right"))


def test_state_recursion_closed_form():
    """Constant gates (Wr = 0 except W_o = [I | 0]): s_k = tanh(c)(1 - sigma(g)^k)
    and a_k = tanh(s_{k-1}), up to fp32 rounding of each step."""
    rng = np.random.default_rng(5)
    V, r, g = 20, 3, 6
    Wr = np.zeros((3 * r, 2 * r))
    Wr[2 * r:, :r] = np.eye(r)
    gc = np.array([0.3, -1.0, 2.0])
    cc = np.array([0.5, 1.5, -0.7])
    hp = np.zeros((g, 3, r))
    hp[:, 0], hp[:, 1] = gc, cc
    d, a_rows = H.rnn_draft_request(rng.normal(size=(g, V)), rng.normal(size=(V, r)),
                                    rng.normal(size=(r, V)), Wr, hp, 0, 1.0, rng.random(g), "f32")
    sig = 1 / (1 + np.exp(-gc))
    for k in range(g):
        s_prev = np.tanh(cc) * (1 - sig ** k)
        assert np.allclose(a_rows[k], np.tanh(s_prev), atol=1e-6)


def test_verify_with_factor_rows_matches_the_markov_verify():
    rng = np.random.default_rng(6)
    V, r, g = 40, 4, 4
    W1, W2 = rng.normal(0, 0.5, (V, r)), rng.normal(0, 0.5, (r, V))
    t, U = rng.normal(0, 2, (g + 1, V)), rng.normal(0, 2, (g, V))
    toks = rng.integers(0, V, g)
    prevs = [5] + list(toks[:-1])
    for L in range(g + 1):
        args = (t, U, W1, W2, 5, 1.0, toks, L, rng.random(g), rng.random())
        a = O.verify_request(*args)
        b = O.verify_request(*args, a_rows=W1[prevs])
        assert a.accept_len == b.accept_len and np.array_equal(a.out_tokens, b.out_tokens)
        assert np.allclose(a.alpha, b.alpha, equal_nan=True, rtol=1e-13)


def test_sigmoid_tails():
    assert H.sigmoid(0.0) == 0.5
    assert H.sigmoid(800.0) == 1.0 and H.sigmoid(-800.0) == 0.0
    assert H.sigmoid(-30.0) == pytest.approx(math.exp(-30.0), rel=1e-12)
