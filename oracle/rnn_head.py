"""Plain float64 oracle of DSpark's RNN head draft.

TEST INFRASTRUCTURE, like spec_oracle.py: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import or run this module.

Source: "[논문리뷰] DSpark: Confidence-Scheduled Speculative Decoding with
Semi-Autoregressive Generation" (review page), section 1.2, "RNN head": the
recurrent state s_k (s_0 = 0) carries the block's prefix; at each step
z_k = [s_{k-1}; W1[x_{k-1}]; h_k] and

    s_k = sigma(W_g z_k) * s_{k-1} + (1 - sigma(W_g z_k)) * tanh(W_c z_k)
    B_k(x_<k, .) = W2^T tanh(W_o z_k)

with p_k = softmax(U_k + B_k) as for the Markov head (tempered by T_b here,
as everywhere on this path).

Readings (shared with the kernel):
* the h_k block of z_k enters the three gates linearly and does not depend on
  the drafted tokens, so its projections hproj[b, k] = (W_g^h h_k, W_c^h h_k,
  W_o^h h_k) are formed by the parallel stage with U_k and arrive as inputs;
  the recurrent part Wr = [W^s | W^e] ([3r, 2r]: rows g, c, o; columns s, then
  W1[x]) is applied on the path;
* the state s_k and the factor a_k = tanh(W_o z_k) are held in the model's
  storage type (bf16, or fp32 for fp32 models): each is the float64 value
  rounded to nearest-even once per step, and the rounded values feed the next
  step and the bias B_k = a_k W2;
* draft row j (0-based) draws x_{j+1} from z built with s_j and W1[x_j]
  (x_0 = the anchor).
"""
from __future__ import annotations

import math

import numpy as np

from oracle import spec_oracle as O


def round_bf16(x) -> np.ndarray:
    """Nearest bfloat16 value (ties to even) of float64 values, as float64."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def round_store(x, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_bf16(x)
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def sigmoid(x: float) -> float:
    return 1.0 / (1.0 + math.exp(-x)) if x >= 0 else math.exp(x) / (1.0 + math.exp(x))


def gates(Wr: np.ndarray, s: np.ndarray, e: np.ndarray, hp: np.ndarray) -> np.ndarray:
    """Pre-activations [3, r]: row i of Wr dotted with [s; e] plus hp, each sum
    correctly rounded (math.fsum of exact float64 products)."""
    z = np.concatenate([s, e])
    r = s.shape[0]
    out = np.empty(3 * r)
    for i in range(3 * r):
        out[i] = math.fsum(list(Wr[i] * z) + [float(hp.reshape(-1)[i])])
    return out.reshape(3, r)


def rnn_step(Wr, s, e, hp, dtype):
    """One step: (a_k, s_k), both rounded to the storage type."""
    pre = gates(Wr, s, e, hp)
    g = np.array([sigmoid(v) for v in pre[0]])
    c = np.tanh(pre[1])
    a = np.tanh(pre[2])
    s_new = g * s + (1.0 - g) * c
    return round_store(a, dtype), round_store(s_new, dtype)


def rnn_draft_request(U_b, W1, W2, Wr, hproj_b, anchor, T, u_draft_b, dtype):
    """Draft x_1..x_gamma with the RNN head.  Returns (DraftResult, a_rows
    [gamma, r]) -- a_rows are the rounded factors the verification needs."""
    g, V = U_b.shape
    r = W1.shape[1]
    s = np.zeros(r)
    prev = int(anchor)
    W2f = np.asarray(W2, dtype=np.float64)
    tokens = np.zeros(g, np.int32)
    q_tok, lse_q, dist, F_lo, F_hi = (np.zeros(g) for _ in range(5))
    a_rows = np.zeros((g, r))
    for k in range(g):
        a, s = rnn_step(Wr, s, np.asarray(W1[prev], dtype=np.float64), hproj_b[k], dtype)
        a_rows[k] = a
        q, lse = O.softmax_with_lse((np.asarray(U_b[k], dtype=np.float64) + a @ W2f) / float(T))
        d = O.inverse_cdf(q, float(u_draft_b[k]))
        tokens[k] = d.token
        q_tok[k], lse_q[k], dist[k], F_lo[k], F_hi[k] = q[d.token], lse, d.dist, d.F_lo, d.F_hi
        prev = d.token
    return O.DraftResult(tokens, q_tok, lse_q, dist, F_lo, F_hi), a_rows


def rnn_cycle_request(t_b, U_b, W1, W2, Wr, hproj_b, anchor, T, u_draft_b, L, u_accept_b,
                      u_final, dtype):
    """Draft with the RNN head, then verify that draft (q rebuilt from a_rows)."""
    d, a_rows = rnn_draft_request(U_b, W1, W2, Wr, hproj_b, anchor, T, u_draft_b, dtype)
    v = O.verify_request(t_b, U_b, W1, W2, anchor, T, d.tokens, L, u_accept_b, u_final,
                         a_rows=a_rows)
    return d, v, a_rows
