"""Plain float64 oracle of the analytic operating-point report.

TEST INFRASTRUCTURE, like spec_oracle.py: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import or run this module.

Source: "Speculative Decoding Part 1: 도입 전에 확인해야 할 것들" (VESSL AI blog),
section "속도 향상을 결정하는 방정식" (the speed-up equation) and the section on
why speculation spends more compute.  With i.i.d. Bernoulli(alpha) acceptance
and the draft cost ratio c = T_draft / (gamma T_target):

* E[tau] = sum_{k=0}^{gamma} alpha^k (tokens per cycle);
* S(gamma) = E[tau] / (c gamma + 1) (wall-clock speed-up);
* S <= min(1/c, 1/(1 - alpha));
* gamma = 1: S = (1 + alpha)/(c + 1), a gain only when alpha > c;
* dS/dgamma = 0 gives alpha^{gamma+1} (c - (c gamma + 1) ln alpha) = c, whose
  left side strictly decreases in gamma (S is unimodal);
* expected compute ratio (1 - alpha)(gamma c_hat + gamma + 1)/(1 - alpha^{gamma+1}),
  c_hat the draft's compute ratio.

Every quantity is taken from its definition (sums, enumeration over integer
gamma, bisection on the stationarity condition) rather than a rearranged form.
"""
from __future__ import annotations

import math

import numpy as np


def expected_tau(alpha: float, gamma: int) -> float:
    """E[tau] = sum_{k=0}^{gamma} alpha^k."""
    return math.fsum(alpha ** k for k in range(gamma + 1))


def speedup(alpha: float, c: float, gamma: int) -> float:
    """S(gamma) = E[tau] / (c gamma + 1)."""
    return expected_tau(alpha, gamma) / (c * gamma + 1.0)


def speedup_bound(alpha: float, c: float) -> float:
    """min(1/c, 1/(1 - alpha)); infinite terms for c = 0 or alpha = 1."""
    a = math.inf if c == 0 else 1.0 / c
    b = math.inf if alpha >= 1.0 else 1.0 / (1.0 - alpha)
    return min(a, b)


def optimal_gamma(alpha: float, c: float, gamma_max: int) -> tuple[int, float]:
    """Integer gamma in 1..gamma_max with the largest S (the smallest on ties)."""
    best_g, best_s = 1, speedup(alpha, c, 1)
    for g in range(2, gamma_max + 1):
        s = speedup(alpha, c, g)
        if s > best_s:
            best_g, best_s = g, s
    return best_g, best_s


def stationarity(alpha: float, c: float, gamma: float) -> float:
    """alpha^{gamma+1} (c - (c gamma + 1) ln alpha) - c for real gamma."""
    return alpha ** (gamma + 1.0) * (c - (c * gamma + 1.0) * math.log(alpha)) - c


def continuous_optimum(alpha: float, c: float, hi: float = 1e6) -> float:
    """Real gamma >= 0 where the stationarity condition holds (bisection; the
    left side strictly decreases).  0 if S already decreases at gamma = 0."""
    if stationarity(alpha, c, 0.0) <= 0.0:
        return 0.0
    lo, up = 0.0, 1.0
    while stationarity(alpha, c, up) > 0.0 and up < hi:
        up *= 2.0
    for _ in range(200):
        mid = 0.5 * (lo + up)
        if stationarity(alpha, c, mid) > 0.0:
            lo = mid
        else:
            up = mid
    return 0.5 * (lo + up)


def compute_ratio(alpha: float, c_hat: float, gamma: int) -> float:
    """(gamma c_hat + gamma + 1) / E[tau]: expected total compute relative to
    plain decoding."""
    return (gamma * c_hat + gamma + 1.0) / expected_tau(alpha, gamma)


def measured_alpha(alpha: np.ndarray, verify_len: np.ndarray) -> float:
    """Mean of the per-position acceptance rates alpha[b, j] over j < L_b."""
    vals = [float(alpha[b, j]) for b in range(alpha.shape[0]) for j in range(int(verify_len[b]))]
    return math.fsum(vals) / len(vals) if vals else float("nan")


def measured_tau(accept_len: np.ndarray) -> float:
    """Mean tokens emitted per request per cycle: n_b + 1."""
    vals = [float(n) + 1.0 for n in accept_len if n >= 0]
    return math.fsum(vals) / len(vals) if vals else float("nan")
