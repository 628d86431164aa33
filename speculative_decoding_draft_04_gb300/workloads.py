"""Seeded synthetic workloads for the speculative-decoding sampling path.

This module only draws random numbers and rounds them to the storage type.
It holds none of the method's arithmetic (no softmax, no bias, no sampling):
the CPU oracle and the CUDA path both take their inputs from here, and from
nowhere else.

Recipe (one request = one row of the batch b):

* ``target[b, j, :]`` for j = 0..gamma are the target model's logits at the
  gamma+1 verified positions ("Speculative Decoding Part 1", section
  "알고리즘": one target pass scores gamma+1 positions).  Either i.i.d.
  N(0, sd^2), or Zipf-shaped: N(0, sd^2) - slope * ln(1 + pi_b(v)) where pi_b
  is a per-request random permutation of the vocabulary (the rank of v).
* ``U[b, j, :] = target[b, j, :] + N(0, s_b^2)`` for j = 0..gamma-1: the
  drafter's base logits U_1..U_gamma (DSpark review, section 1.1 "Parallel
  stage") are a noisy copy of the target, so the draft/target agreement
  alpha is controlled by the per-request noise scale s_b.  The noise is
  added in float64 and the SUM is rounded once to the storage type.
* ``W1 [V, r]`` and ``W2 [r, V]``: the Markov head's low-rank factors (DSpark
  review, section 1.2, "Markov head"), i.i.d. N(0, w_sd^2).
* ``anchor[b]`` uniform in [0, V): the token x_0 left by the previous cycle.
* ``temperature[b]``: one value or a per-request draw from a small set.
* ``verify_len[b] = L_b``: gamma (fixed-length verification, H-Spec review,
  Appx. B.2) or a per-request uniform integer draw (DSpark review, section
  2.2: the scheduler picks l_r in {0..gamma}).
* uniforms: every random decision of the method takes a caller-supplied
  uniform u = (m + 0.5) * 2^-23 with m uniform in [0, 2^23): exact in float32
  (float32 spacing in [0.5, 1) is 2^-24) and strictly inside (0, 1), the
  largest being 1 - 2^-24.  u_draft[b, k] samples draft token x_{k+1},
  u_accept[b, j] is the ratio-test uniform of position j, u_final[b] samples
  the correction or bonus token.

Seeds: inputs come from ``numpy.random.default_rng([seed_index, trial, 1])``
and uniforms from ``numpy.random.default_rng(trial)``.  Draw order: noise
scales, temperatures, verify lengths, W1, W2, anchors, then per request
(target base, permutation if Zipf, noise); uniforms: u_draft, u_accept,
u_final.

Confidence-head and scheduler inputs (``make_schedule_inputs``, DSpark
review, sections 2.1 and 2.2), from ``default_rng([seed_index, trial, 2])``:

* ``hidden[b, k, :]`` (the drafter backbone's h_{k+1}, width d): N(0, 1)
  except coordinate 0, which holds a per-request offset mu_b ~ U[-1, 3] (a
  stand-in for the domain: low for chat-like, high for code-like requests);
* ``w [d + r]`` float32: w[0] = 1 (so mu_b shifts the logit), w[1:d] ~
  N(0, 1/d) (hidden noise of unit variance), w[d:] ~ N(0, (0.5 / (sqrt(r) *
  w_sd))^2) (the embedding part adds variance 0.25);
* ``sps[B']`` for B' = 0..B (1 + gamma): the engine's steps per second at
  batch B', 1000 / t(B') with t(B') = sqrt(t0^2 + (B' t1)^2) ms, t0 = 42 ms
  (the memory-bound decode step of the VESSL blog's 70B example) and t1 =
  t0 / (B (1 + gamma / 2)), so the curve bends half-way through the
  candidates.

Draw order: mu, w, then hidden per request.

Tree inputs (``make_tree_inputs``, VESSL AI blog, section "gamma 재배분"),
from ``default_rng([seed_index, trial, 4])`` for a candidate tree of N slots:

* ``parent[b, s]``: slot s hangs under the root or an earlier slot, drawn
  uniformly among those that keep depth <= gamma (a random bushy tree);
* ``conf[b, s]`` U[0.3, 0.95]: the slot's conditional survival factor;
* ``target[b, 0]`` = the workload's target row 0 and ``target[b, 1 + s]`` =
  its target row depth(s) plus N(0, 0.5^2): every node has its own target
  row, close to the chain's at that depth, so the shared U row of a depth
  still agrees with it;
* uniforms (``uniforms``): u_draft [B, N], u_accept [B, N], u_final [B].

Draw order: per request parent, conf, target noise; then the uniforms from
``default_rng([trial, 4])``.

RNN head inputs (``make_rnn_inputs``, DSpark review, section 1.2 "RNN head"),
from ``default_rng([seed_index, trial, 3])``:

* ``Wr [3r, 2r]`` (storage dtype): rows g, c, o of the gates' recurrent part;
  columns [0, r) act on the state, N(0, 1/r); columns [r, 2r) on W1[x],
  N(0, 1/(r w_sd^2)) (so that part of each pre-activation has unit variance);
* ``hproj [B, gamma, 3, r]`` float32: the parallel stage's projections of
  h_k into the three gates, N(0, 1).

Draw order: Wr, then hproj per request.

bf16 storage is round-to-nearest-even from float64, done directly (no
intermediate float32 rounding).
"""
from __future__ import annotations

import dataclasses
from typing import Any

import numpy as np

U23 = float(2.0 ** -23)

# Named workloads.  C0 is small enough for exhaustive oracle comparison; C1-C4
# carry the shapes of the pages' drafter (rank 256, vocabulary 32000, k=7 from
# the H-Spec review, Appx. B.1/B.2) and of larger vocabularies.
CONFIGS: dict[str, dict[str, Any]] = {
    "C0": dict(seed_index=0, d=64, B=4, gamma=4, V=1000, r=16, dtype="f32",
               target=("normal", 3.0), noise=("fixed", 1.0), temps=(1.0,),
               L="full", w_sd=0.1),
    "C1": dict(seed_index=1, d=4096, B=32, gamma=7, V=32000, r=256, dtype="bf16",
               target=("normal", 3.0), noise=("uniform", 0.5, 3.0), temps=(1.0,),
               L="full", w_sd=0.02),
    "C2": dict(seed_index=2, d=4096, B=128, gamma=7, V=32000, r=256, dtype="bf16",
               target=("normal", 3.0), noise=("uniform", 0.5, 3.0), temps=(1.0,),
               L=("uniform", 1, 7), w_sd=0.02),
    "C3": dict(seed_index=3, d=4096, B=64, gamma=15, V=151936, r=256, dtype="bf16",
               target=("zipf", 2.0, 1.1), noise=("uniform", 0.5, 3.0), temps=(0.6, 1.0),
               L="full", w_sd=0.02),
    "C4": dict(seed_index=4, d=4096, B=256, gamma=7, V=128256, r=256, dtype="bf16",
               target=("normal", 3.0), noise=("uniform", 0.3, 4.0), temps=(0.7, 1.0),
               L=("uniform", 0, 7), w_sd=0.02),
}

CONFIG_DESCRIPTIONS = {
    "C0": "B4 g4 V1000 r16 fp32, N(0,9) target, U=t+N(0,1), W~N(0,0.01), T=1, L=gamma",
    "C1": "B32 g7 V32000 r256 bf16, N(0,9) target, s~U[0.5,3], W~N(0,4e-4), T=1, L=gamma",
    "C2": "B128 g7 V32000 r256 bf16, as C1, ragged L~U{1..7}",
    "C3": "B64 g15 V151936 r256 bf16, Zipf target, s~U[0.5,3], T in {0.6,1.0}, L=gamma",
    "C4": "B256 g7 V128256 r256 bf16, N(0,9) target, s~U[0.3,4], T in {0.7,1.0}, L~U{0..7}",
}


def config(cfg: str, **overrides: Any) -> dict[str, Any]:
    """A copy of a named workload spec with fields overridden (including its
    display ``name``)."""
    spec = dict(CONFIGS[cfg])
    spec["name"] = cfg
    spec.update(overrides)
    return spec


def stress(spec: dict[str, Any], w_sd: float = 0.3) -> dict[str, Any]:
    """Parity-only variant: large Markov factors so the transition bias moves
    the draft distribution by O(1) (a dropped or mis-indexed bias would then
    change almost every sample)."""
    out = dict(spec)
    out["w_sd"] = w_sd
    out["name"] = spec.get("name", "custom") + "-stress"
    return out


# --------------------------------------------------------------------------- rounding

def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even); returns the
    16-bit patterns as uint16."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
    q = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)   # keep 8 significant bits, RNE
    bits = q.astype(np.float32).view(np.uint32)    # exact: q has <= 8 significant bits
    return (bits >> 16).astype(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def to_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Widen a stored array (bf16 bit patterns or float32) to float64, exactly."""
    if dtype == "bf16":
        return bf16_to_f64(arr)
    return np.asarray(arr, dtype=np.float32).astype(np.float64)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_round(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


# --------------------------------------------------------------------------- uniforms

def uniforms(rng: np.random.Generator, shape) -> np.ndarray:
    """u = (m + 0.5) * 2^-23, m uniform in [0, 2^23): float32, exactly representable."""
    m = rng.integers(0, 1 << 23, size=shape, dtype=np.int64)
    return ((m.astype(np.float64) + 0.5) * U23).astype(np.float32)


# --------------------------------------------------------------------------- workload

@dataclasses.dataclass
class Workload:
    spec: dict
    trial: int
    dtype: str
    B: int
    gamma: int
    V: int
    r: int
    target: np.ndarray      # [B, gamma+1, V]  storage dtype (uint16 bf16 bits or float32)
    U: np.ndarray           # [B, gamma, V]
    W1: np.ndarray          # [V, r]
    W2: np.ndarray          # [r, V]
    anchor: np.ndarray      # int32 [B]
    temperature: np.ndarray  # float32 [B]
    verify_len: np.ndarray  # int32 [B]
    u_draft: np.ndarray     # float32 [B, gamma]
    u_accept: np.ndarray    # float32 [B, gamma]
    u_final: np.ndarray     # float32 [B]

    @property
    def name(self) -> str:
        return self.spec.get("name", "custom")

    def f64(self, field: str) -> np.ndarray:
        """Float64 widening of a stored floating-point field."""
        return to_f64(getattr(self, field), self.dtype)

    def row_f64(self, field: str, b: int, j: int) -> np.ndarray:
        return to_f64(getattr(self, field)[b, j], self.dtype)

    def nbytes_inputs(self) -> int:
        return sum(getattr(self, f).nbytes for f in
                   ("target", "U", "W1", "W2", "anchor", "temperature", "verify_len",
                    "u_draft", "u_accept", "u_final"))

    def subset(self, rows) -> "Workload":
        """The same workload restricted to a list of requests (weights shared)."""
        rows = np.asarray(rows, dtype=np.int64)
        return dataclasses.replace(
            self, B=len(rows), target=self.target[rows], U=self.U[rows],
            anchor=self.anchor[rows], temperature=self.temperature[rows],
            verify_len=self.verify_len[rows], u_draft=self.u_draft[rows],
            u_accept=self.u_accept[rows], u_final=self.u_final[rows])


def make_workload(spec: dict[str, Any], trial: int = 0, *, B: int | None = None) -> Workload:
    """Draw one seeded workload from a spec (see module docstring for the recipe).

    ``B`` overrides the batch size (the per-request draws of the first B
    requests are identical to the full-size draw's)."""
    Bn = int(spec["B"] if B is None else B)
    g, V, r = int(spec["gamma"]), int(spec["V"]), int(spec["r"])
    dtype = spec["dtype"]
    rng = np.random.default_rng([int(spec["seed_index"]), int(trial), 1])
    Bfull = int(spec["B"]) if B is None else max(Bn, int(spec["B"]))

    noise = spec["noise"]
    if noise[0] == "fixed":
        s = np.full(Bfull, float(noise[1]))
    elif noise[0] == "uniform":
        s = rng.uniform(float(noise[1]), float(noise[2]), size=Bfull)
    else:
        raise ValueError(noise)
    temps = tuple(spec["temps"])
    if len(temps) == 1:
        T = np.full(Bfull, temps[0], dtype=np.float32)
    else:
        T = np.asarray(rng.choice(np.asarray(temps, dtype=np.float64), size=Bfull),
                       dtype=np.float32)
    Ls = spec["L"]
    if Ls == "full":
        L = np.full(Bfull, g, dtype=np.int32)
    elif Ls[0] == "uniform":
        L = rng.integers(int(Ls[1]), min(int(Ls[2]), g) + 1, size=Bfull).astype(np.int32)
    elif Ls[0] == "fixed":
        L = np.full(Bfull, int(Ls[1]), dtype=np.int32)
    else:
        raise ValueError(Ls)
    w_sd = float(spec["w_sd"])
    W1 = _store(rng.normal(0.0, w_sd, size=(V, r)), dtype)
    W2 = _store(rng.normal(0.0, w_sd, size=(r, V)), dtype)
    anchor = rng.integers(0, V, size=Bfull).astype(np.int32)

    sdt = np.uint16 if dtype == "bf16" else np.float32
    target = np.empty((Bn, g + 1, V), dtype=sdt)
    U = np.empty((Bn, g, V), dtype=sdt)
    tgt = spec["target"]
    for b in range(Bn):
        if tgt[0] == "normal":
            t = rng.normal(0.0, float(tgt[1]), size=(g + 1, V))
        elif tgt[0] == "zipf":
            t = rng.normal(0.0, float(tgt[1]), size=(g + 1, V))
            rank = rng.permutation(V)
            t = t - float(tgt[2]) * np.log1p(rank.astype(np.float64))[None, :]
        else:
            raise ValueError(tgt)
        u = t[:g] + rng.normal(0.0, 1.0, size=(g, V)) * s[b]
        target[b] = _store(t, dtype)
        U[b] = _store(u, dtype)

    urng = np.random.default_rng(int(trial))
    u_draft = uniforms(urng, (Bfull, g))[:Bn]
    u_acc = uniforms(urng, (Bfull, g))[:Bn]
    u_fin = uniforms(urng, (Bfull,))[:Bn]
    return Workload(spec=dict(spec), trial=int(trial), dtype=dtype, B=Bn, gamma=g, V=V, r=r,
                    target=target, U=U, W1=W1, W2=W2, anchor=anchor[:Bn].copy(),
                    temperature=T[:Bn].copy(), verify_len=L[:Bn].copy(),
                    u_draft=np.ascontiguousarray(u_draft),
                    u_accept=np.ascontiguousarray(u_acc),
                    u_final=np.ascontiguousarray(u_fin))


@dataclasses.dataclass
class ScheduleInputs:
    d: int
    hidden: np.ndarray      # [B, gamma, d] storage dtype
    w: np.ndarray           # float32 [d + r]
    sps: np.ndarray         # float64 [B (1 + gamma) + 1]


SPS_T0_MS = 42.0


def cost_table(B: int, gamma: int, t0: float = SPS_T0_MS) -> np.ndarray:
    """Synthetic steps-per-second table for batch sizes 0..B (1 + gamma)."""
    t1 = t0 / (B * (1.0 + gamma / 2.0))
    Bs = np.arange(B * (1 + gamma) + 1, dtype=np.float64)
    return 1000.0 / np.sqrt(t0 * t0 + (Bs * t1) ** 2)


def make_schedule_inputs(spec: dict[str, Any], trial: int = 0, *,
                         B: int | None = None) -> ScheduleInputs:
    """Confidence-head inputs and the cost table of one workload (see the
    module docstring); ``B`` as in make_workload."""
    Bn = int(spec["B"] if B is None else B)
    g, r, d = int(spec["gamma"]), int(spec["r"]), int(spec["d"])
    dtype = spec["dtype"]
    rng = np.random.default_rng([int(spec["seed_index"]), int(trial), 2])
    Bfull = int(spec["B"]) if B is None else max(Bn, int(spec["B"]))
    mu = rng.uniform(-1.0, 3.0, size=Bfull)
    w = np.empty(d + r, dtype=np.float64)
    w[0] = 1.0
    w[1:d] = rng.normal(0.0, 1.0 / np.sqrt(d), size=d - 1)
    w[d:] = rng.normal(0.0, 0.5 / (np.sqrt(r) * float(spec["w_sd"])), size=r)
    sdt = np.uint16 if dtype == "bf16" else np.float32
    hidden = np.empty((Bn, g, d), dtype=sdt)
    for b in range(Bn):
        h = rng.normal(0.0, 1.0, size=(g, d))
        h[:, 0] = mu[b]
        hidden[b] = _store(h, dtype)
    return ScheduleInputs(d=d, hidden=hidden, w=w.astype(np.float32), sps=cost_table(Bn, g))


@dataclasses.dataclass
class TreeInputs:
    N: int
    parent: np.ndarray      # int32 [B, N]
    conf: np.ndarray        # float32 [B, N]
    target: np.ndarray      # [B, N + 1, V] storage dtype
    u_draft: np.ndarray     # float32 [B, N]
    u_accept: np.ndarray    # float32 [B, N]
    u_final: np.ndarray     # float32 [B]


def make_tree_inputs(spec: dict[str, Any], w: "Workload", N: int, trial: int = 0) -> TreeInputs:
    """Candidate trees and per-node target rows for the requests of ``w``."""
    B, g, V = w.B, w.gamma, w.V
    rng = np.random.default_rng([int(spec["seed_index"]), int(trial), 4])
    parent = np.empty((B, N), np.int32)
    conf = np.empty((B, N), np.float32)
    sdt = np.uint16 if w.dtype == "bf16" else np.float32
    target = np.empty((B, N + 1, V), dtype=sdt)
    for b in range(B):
        depth = []
        for s in range(N):
            cands = [-1] + [p for p in range(s) if depth[p] < g]
            p = int(rng.choice(cands))
            parent[b, s] = p
            depth.append(1 if p < 0 else depth[p] + 1)
        conf[b] = rng.uniform(0.3, 0.95, size=N).astype(np.float32)
        base = to_f64(w.target[b], w.dtype)
        rows = np.empty((N + 1, V))
        rows[0] = base[0]
        for s in range(N):
            rows[1 + s] = base[depth[s]] + rng.normal(0.0, 0.5, size=V)
        target[b] = _store(rows, w.dtype)
    urng = np.random.default_rng([int(trial), 4])
    return TreeInputs(N=N, parent=parent, conf=conf, target=target,
                      u_draft=uniforms(urng, (B, N)), u_accept=uniforms(urng, (B, N)),
                      u_final=uniforms(urng, (B,)))


@dataclasses.dataclass
class RnnInputs:
    Wr: np.ndarray          # [3r, 2r] storage dtype
    hproj: np.ndarray       # float32 [B, gamma, 3, r]


def make_rnn_inputs(spec: dict[str, Any], trial: int = 0, *, B: int | None = None) -> RnnInputs:
    """RNN head inputs of one workload (see the module docstring)."""
    Bn = int(spec["B"] if B is None else B)
    g, r = int(spec["gamma"]), int(spec["r"])
    rng = np.random.default_rng([int(spec["seed_index"]), int(trial), 3])
    Wr = np.empty((3 * r, 2 * r))
    Wr[:, :r] = rng.normal(0.0, 1.0 / np.sqrt(r), size=(3 * r, r))
    Wr[:, r:] = rng.normal(0.0, 1.0 / (np.sqrt(r) * float(spec["w_sd"])), size=(3 * r, r))
    hproj = np.empty((Bn, g, 3, r), dtype=np.float32)
    for b in range(Bn):
        hproj[b] = rng.normal(0.0, 1.0, size=(g, 3, r)).astype(np.float32)
    return RnnInputs(Wr=_store(Wr, spec["dtype"]), hproj=hproj)


def shard_rows(B: int, rank: int, world: int) -> np.ndarray:
    """Requests owned by ``rank`` when a batch of B independent requests is
    split over ``world`` replicas: contiguous, sizes differ by at most one."""
    if not (0 <= rank < world):
        raise ValueError("rank out of range")
    base, extra = divmod(B, world)
    start = rank * base + min(rank, extra)
    n = base + (1 if rank < extra else 0)
    return np.arange(start, start + n, dtype=np.int64)
