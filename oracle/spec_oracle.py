"""Plain float64 CPU oracle of the speculative-decoding sampling hot path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import or run this module.
The product path (the CUDA library and its Python binding) never calls it and
shares no code with it.

Everything is float64, one request at a time, numpy over the vocabulary only.
Inputs are the exact stored values (bf16 or fp32) widened to float64; the
uniforms are the exact float32 values widened.

Sources (the three web pages the method is defined on):

* [DSpark] "[논문리뷰] DSpark: Confidence-Scheduled Speculative Decoding with
  Semi-Autoregressive Generation" (review page), section 1.2 "Sequential
  stage": block factorisation P(X|x_0) = prod_k p_k(x_k | x_0, x_<k) with
  p_k = softmax(U_k + B_k), sampled left to right; "Markov head":
  B(x_{k-1}, .) = W1[x_{k-1}] W2.
* [SpecDec] "Speculative Decoding Part 1: 도입 전에 확인해야 할 것들" (VESSL AI
  blog), section "알고리즘" (the speculative cycle), section "수락 규칙"
  (acceptance rule min(1, p/q), residual max(0, p-q) normalised), the
  closed form alpha = sum_v min(p, q).
* Readings where the pages are silent (all stated once here):
  - q is the draft distribution, p the target distribution.
  - temperature T_b divides both the draft logits (U + B) and the target
    logits; the same T_b for both.
  - draft row j (U_{j+1} in the pages' 1-based notation) produces token
    x_{j+1} from the bias of x_j (x_0 = anchor); target row j tests x_{j+1};
    the bonus token uses target row L_b.
  - sampling is inverse-CDF in vocabulary-index order: the smallest v with
    F(v) > u; if rounding leaves no such v, the largest v with positive
    probability.
  - the ratio test accepts iff u < p(x)/q(x) (equality rejects).
  - verification stops at the per-request verify length L_b (0 <= L_b <=
    gamma); L_b = 0 emits only the bonus token sampled from target row 0.
  - if the residual has zero mass, the correction token is sampled from p.
"""
from __future__ import annotations

import dataclasses

import numpy as np


# --------------------------------------------------------------------------- building blocks

def softmax_with_lse(logits: np.ndarray) -> tuple[np.ndarray, float]:
    """softmax(l) and logsumexp(l) of a float64 vector (max-shifted)."""
    l = np.asarray(logits, dtype=np.float64)
    m = float(np.max(l))
    e = np.exp(l - m)
    s = float(np.sum(e))
    return e / s, m + float(np.log(s))


def markov_bias(W1: np.ndarray, W2: np.ndarray, prev_token: int) -> np.ndarray:
    """[DSpark] §1.2 Markov head: transition bias B(x_{k-1}, .) = W1[x_{k-1}] W2."""
    return np.asarray(W1[int(prev_token)], dtype=np.float64) @ np.asarray(W2, dtype=np.float64)


def draft_distribution(U_row, W1, W2, prev_token, T) -> tuple[np.ndarray, float]:
    """[DSpark] §1.2 eq. for p_k with the Markov head, tempered:
    q = softmax((U_k + W1[x_{k-1}] W2) / T).  Returns (q, logsumexp of the
    tempered logits)."""
    l = (np.asarray(U_row, dtype=np.float64) + markov_bias(W1, W2, prev_token)) / float(T)
    return softmax_with_lse(l)


def target_distribution(t_row, T) -> tuple[np.ndarray, float]:
    """Target p = softmax(t / T) (same temperature as the draft)."""
    return softmax_with_lse(np.asarray(t_row, dtype=np.float64) / float(T))


@dataclasses.dataclass
class Draw:
    token: int
    dist: float      # distance of u to the nearer end of the chosen CDF interval
    F_lo: float      # F(token - 1)
    F_hi: float      # F(token)
    fallback: bool   # rounding left no v with F(v) > u


def inverse_cdf(probs: np.ndarray, u: float) -> Draw:
    """[SpecDec] "알고리즘": sample(dist) read as inverse-CDF in index order:
    the smallest v with F(v) > u, F the running sum of probs."""
    p = np.asarray(probs, dtype=np.float64)
    F = np.cumsum(p)
    above = np.nonzero(F > u)[0]
    if above.size:
        v = int(above[0])
        lo = float(F[v - 1]) if v > 0 else 0.0
        hi = float(F[v])
        return Draw(v, min(u - lo, hi - u), lo, hi, False)
    pos = np.nonzero(p > 0)[0]
    v = int(pos[-1]) if pos.size else len(p) - 1
    lo = float(F[v - 1]) if v > 0 else 0.0
    return Draw(v, 0.0, lo, float(F[v]), True)


# --------------------------------------------------------------------------- draft

@dataclasses.dataclass
class DraftResult:
    tokens: np.ndarray    # int32 [gamma]   x_1..x_gamma
    q_tok: np.ndarray     # float64 [gamma] q_k(x_k)
    lse_q: np.ndarray     # float64 [gamma] logsumexp((U_k + B)/T)
    dist: np.ndarray      # float64 [gamma] boundary distance of each draw
    F_lo: np.ndarray
    F_hi: np.ndarray
    q_rows: np.ndarray | None = None   # [gamma, V] when requested


def draft_request(U_b, W1, W2, anchor, T, u_draft_b, return_rows: bool = False) -> DraftResult:
    """[DSpark] §1.2: sample x_1..x_gamma left to right; x_k ~ q_k(. | x_{k-1}),
    x_0 the anchor.  U_b is the request's [gamma, V] base logits."""
    g = U_b.shape[0]
    tokens = np.zeros(g, np.int32)
    q_tok = np.zeros(g)
    lse_q = np.zeros(g)
    dist = np.zeros(g)
    F_lo = np.zeros(g)
    F_hi = np.zeros(g)
    rows = np.zeros((g, U_b.shape[1])) if return_rows else None
    prev = int(anchor)
    for k in range(g):
        q, lse = draft_distribution(U_b[k], W1, W2, prev, T)
        d = inverse_cdf(q, float(u_draft_b[k]))
        tokens[k] = d.token
        q_tok[k] = q[d.token]
        lse_q[k] = lse
        dist[k] = d.dist
        F_lo[k], F_hi[k] = d.F_lo, d.F_hi
        if rows is not None:
            rows[k] = q
        prev = d.token
    return DraftResult(tokens, q_tok, lse_q, dist, F_lo, F_hi, rows)


# --------------------------------------------------------------------------- verify

@dataclasses.dataclass
class VerifyResult:
    accept_len: int            # n_b (tau = n_b + 1)
    out_tokens: np.ndarray     # int32 [gamma+1]: x_1..x_n, correction/bonus, -1 padding
    alpha: np.ndarray          # float64 [gamma]: sum_v min(p_j, q_j) for j < L, NaN beyond
    p_tok: np.ndarray          # float64 [gamma]: p_j(x_{j+1}) for j < L, NaN beyond
    ratio: np.ndarray          # float64 [gamma]: p_j(x_{j+1}) / q_j(x_{j+1}) for j < L
    ratio_dist: np.ndarray     # float64 [gamma]: |u_accept - ratio| for consumed tests, inf else
    final: Draw                # the correction / bonus draw
    final_kind: str            # "residual", "residual-empty" or "bonus"
    lse_p: np.ndarray          # float64 [gamma+1] for j <= L, NaN beyond
    p_rows: np.ndarray | None = None


def verify_request(t_b, U_b, W1, W2, anchor, T, draft_tokens_b, L, u_accept_b, u_final,
                   return_rows: bool = False, a_rows=None) -> VerifyResult:
    """[SpecDec] "알고리즘" + "수락 규칙" for one request with verify length L.

    Ratio tests j = 0..L-1 accept iff u_accept[j] < p_j(x_{j+1}) / q_j(x_{j+1});
    n = the first rejected j, else L.  Emit x_1..x_n, then the correction
    token ~ normalize(max(0, p_n - q_n)) if n < L, else the bonus token ~ p_L.
    alpha_j = sum_v min(p_j(v), q_j(v)) ("수락 규칙", closed form).

    ``a_rows`` [gamma, r], when given, replaces the Markov head's factor
    W1[x_j] of draft row j (the RNN head's tanh(W_o z) rows, [DSpark] §1.2)."""
    g = U_b.shape[0]
    V = U_b.shape[1]
    L = int(L)
    if not (0 <= L <= g):
        raise ValueError("verify length out of range")
    prevs = [int(anchor)] + [int(x) for x in draft_tokens_b[: g - 1]]
    p_rows = [target_distribution(t_b[j], T) for j in range(L + 1)]
    if a_rows is None:
        q_rows = [draft_distribution(U_b[j], W1, W2, prevs[j], T) for j in range(L)]
    else:
        W2f = np.asarray(W2, dtype=np.float64)
        q_rows = [softmax_with_lse((np.asarray(U_b[j], dtype=np.float64)
                                    + np.asarray(a_rows[j], dtype=np.float64) @ W2f) / float(T))
                  for j in range(L)]

    alpha = np.full(g, np.nan)
    p_tok = np.full(g, np.nan)
    ratio = np.full(g, np.nan)
    ratio_dist = np.full(g, np.inf)
    for j in range(L):
        p, _ = p_rows[j]
        q, _ = q_rows[j]
        alpha[j] = float(np.sum(np.minimum(p, q)))
        x = int(draft_tokens_b[j])
        p_tok[j] = p[x]
        ratio[j] = p[x] / q[x]

    n = L
    for j in range(L):
        u = float(u_accept_b[j])
        ratio_dist[j] = abs(u - ratio[j])
        if not (u < ratio[j]):
            n = j
            break

    if n < L:
        p, _ = p_rows[n]
        q, _ = q_rows[n]
        res = np.maximum(0.0, p - q)
        mass = float(np.sum(res))
        if mass > 0.0:
            final = inverse_cdf(res / mass, float(u_final))
            kind = "residual"
        else:
            final = inverse_cdf(p, float(u_final))
            kind = "residual-empty"
    else:
        final = inverse_cdf(p_rows[L][0], float(u_final))
        kind = "bonus"

    out = np.full(g + 1, -1, np.int32)
    out[:n] = np.asarray(draft_tokens_b[:n], dtype=np.int32)
    out[n] = final.token
    lse_p = np.full(g + 1, np.nan)
    for j in range(L + 1):
        lse_p[j] = p_rows[j][1]
    rows = None
    if return_rows:
        rows = np.full((g + 1, V), np.nan)
        for j in range(L + 1):
            rows[j] = p_rows[j][0]
    return VerifyResult(n, out, alpha, p_tok, ratio, ratio_dist, final, kind, lse_p, rows)


# --------------------------------------------------------------------------- batch helpers

@dataclasses.dataclass
class CycleResult:
    draft: list            # DraftResult per request
    verify: list           # VerifyResult per request

    def tokens(self) -> np.ndarray:
        return np.stack([d.tokens for d in self.draft])

    def accept_len(self) -> np.ndarray:
        return np.array([v.accept_len for v in self.verify], np.int32)

    def out_tokens(self) -> np.ndarray:
        return np.stack([v.out_tokens for v in self.verify])

    def alpha(self) -> np.ndarray:
        return np.stack([v.alpha for v in self.verify])

    def row_dmin(self, b: int) -> float:
        """Smallest boundary distance over every uniform request b consumed:
        all gamma draft draws, the ratio tests up to the first reject, and the
        final draw."""
        d = self.draft[b]
        v = self.verify[b]
        cand = [float(np.min(d.dist))] if d.dist.size else []
        finite = v.ratio_dist[np.isfinite(v.ratio_dist)]
        if finite.size:
            cand.append(float(np.min(finite)))
        cand.append(v.final.dist)
        return min(cand)


def cycle_request(t_b, U_b, W1, W2, anchor, T, u_draft_b, L, u_accept_b, u_final):
    """One speculative cycle for one request: draft, then verify the draft."""
    d = draft_request(U_b, W1, W2, anchor, T, u_draft_b)
    v = verify_request(t_b, U_b, W1, W2, anchor, T, d.tokens, L, u_accept_b, u_final)
    return d, v


def cycle(target, U, W1, W2, anchor, T, u_draft, L, u_accept, u_final, rows=None) -> CycleResult:
    """Draft + verify for the requests in ``rows`` (default: all).  ``target``
    and ``U`` may be any per-request indexable returning float64 [., V] rows
    (e.g. a callable wrapper); plain float64 arrays work."""
    B = len(anchor)
    rows = range(B) if rows is None else rows
    ds, vs = [], []
    for b in rows:
        d, v = cycle_request(target[b], U[b], W1, W2, anchor[b], T[b], u_draft[b], L[b],
                             u_accept[b], u_final[b])
        ds.append(d)
        vs.append(v)
    return CycleResult(ds, vs)
