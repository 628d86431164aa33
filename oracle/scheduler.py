"""Plain float64 oracle of the confidence head and the hardware-aware prefix
scheduler.

TEST INFRASTRUCTURE, like spec_oracle.py: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import or run this module.

Source: "[논문리뷰] DSpark: Confidence-Scheduled Speculative Decoding with
Semi-Autoregressive Generation" (review page), section 2.1 "Confidence Head"
(c_k = sigmoid(w^T [h_k; W1[x_{k-1}]])) and section 2.2 "Hardware-Aware Prefix
Scheduler": survival a_{r,j} = prod_{i<=j} c_{r,i}; batch size
B = sum_r (1 + l_r); expected accepted tokens tau = sum_r (1 + sum_{j<=l_r} a_{r,j});
throughput Theta = tau * SPS(B) from a cost table; all prefix extensions sorted
by a in descending order and admitted greedily, Theta updated from the table,
the search stopped at the first decrease of Theta (so the decision depends only
on the prefix processed so far).

Readings (where the page leaves the arithmetic open), shared with the kernel
so that both take the integer decisions in the same precision:
* a is the float32 cumulative product, left to right, of the float32 c values;
* tau is accumulated in integer units of 2^-36 (each a rounded down), so any
  summation order gives the same total; Theta = (tau units * 2^-36) * SPS[B] in
  float64;
* candidates with equal a are taken in (request, position) order;
* the search stops when Theta strictly decreases (equal Theta keeps going), and
  when B would exceed the cost table;
* the confidence head's input index: c for draft row j (the row that draws
  x_{j+1}) uses h row j and W1[x_j] (x_0 = the anchor), the same alignment as
  the draft logits U row j.
"""
from __future__ import annotations

import math

import numpy as np

TAU_UNIT_BITS = 36


def confidence(h_row: np.ndarray, w1_row: np.ndarray, w: np.ndarray) -> float:
    """c = sigmoid(w^T [h; W1 row]) in float64."""
    z = math.fsum(np.concatenate([h_row, w1_row]).astype(np.float64) * w.astype(np.float64))
    return 1.0 / (1.0 + math.exp(-z))


def confidences(hidden, W1, w, anchor, tokens) -> np.ndarray:
    """c[b, j] for every draft row, given the draft tokens (x_1..x_gamma)."""
    B, gamma, _ = hidden.shape
    out = np.empty((B, gamma))
    for b in range(B):
        for j in range(gamma):
            prev = int(anchor[b]) if j == 0 else int(tokens[b, j - 1])
            out[b, j] = confidence(hidden[b, j], W1[prev], w)
    return out


def survival(conf32: np.ndarray) -> np.ndarray:
    """a[r, j] = prod_{i<=j} c[r, i], float32, left to right."""
    c = np.asarray(conf32, dtype=np.float32)
    a = np.empty_like(c)
    a[:, 0] = c[:, 0]
    for j in range(1, c.shape[1]):
        a[:, j] = (a[:, j - 1] * c[:, j]).astype(np.float32)
    return a


def tau_units(a32: float) -> int:
    """floor(a * 2^36) for a float32 a in [0, 1]."""
    return int(math.floor(float(np.float32(a32)) * (1 << TAU_UNIT_BITS)))


def schedule(a32: np.ndarray, sps: np.ndarray):
    """Greedy admission with early stop.  sps[B] is the cost table for batch
    sizes B = 0..len(sps)-1.  Returns (l [R], B, tau units, Theta)."""
    R, gamma = a32.shape
    scale = 2.0 ** -TAU_UNIT_BITS
    order = sorted(((-float(a32[r, j]), r, j) for r in range(R) for j in range(gamma)))
    ell = np.zeros(R, dtype=np.int64)
    bsz = R
    tau = R << TAU_UNIT_BITS
    theta = (tau * scale) * float(sps[bsz]) if bsz < len(sps) else -math.inf
    for _, r, j in order:
        assert j == ell[r], "sorted order must extend each request's prefix"
        nb = bsz + 1
        if nb >= len(sps):
            break
        ntau = tau + tau_units(a32[r, j])
        ntheta = (ntau * scale) * float(sps[nb])
        if ntheta < theta:
            break
        ell[r] = j + 1
        bsz, tau, theta = nb, ntau, ntheta
    return ell, bsz, tau, theta


def batch_and_tau(ell: np.ndarray, a32: np.ndarray):
    """B = sum(1 + l_r) and tau = sum(1 + sum_{j<=l_r} a_{r,j}) (exact units)."""
    bsz = int(sum(1 + int(l) for l in ell))
    tau = sum((1 << TAU_UNIT_BITS) + sum(tau_units(a32[r, j]) for j in range(int(ell[r])))
              for r in range(len(ell)))
    return bsz, tau
