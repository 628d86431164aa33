"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI and the float64 oracle on the same seeded inputs, then compare."""
from __future__ import annotations

import dataclasses

import numpy as np

from oracle import spec_oracle as O
from speculative_decoding_draft_04_gb300 import engine
from speculative_decoding_draft_04_gb300 import workloads as W

BOUNDARY = 1e-6      # a row is "near a boundary" when a consumed uniform is this close
FLOAT_TOL = 1e-5     # probabilities and alpha (absolute)


class LazyRows:
    """Per-request float64 rows of a stored [B, rows, V] array (keeps memory low)."""

    def __init__(self, arr, dtype):
        self.arr, self.dtype = arr, dtype

    def __getitem__(self, b):
        return W.to_f64(self.arr[b], self.dtype)


def oracle_cycle(w: W.Workload, rows=None) -> O.CycleResult:
    return O.cycle(LazyRows(w.target, w.dtype), LazyRows(w.U, w.dtype), w.f64("W1"), w.f64("W2"),
                   w.anchor, w.temperature.astype(np.float64), w.u_draft.astype(np.float64),
                   w.verify_len, w.u_accept.astype(np.float64), w.u_final.astype(np.float64),
                   rows=rows)


@dataclasses.dataclass
class GpuResult:
    draft_tokens: np.ndarray
    q_tok: np.ndarray
    lse_q: np.ndarray
    accept_len: np.ndarray
    out_tokens: np.ndarray
    alpha: np.ndarray
    p_tok: np.ndarray
    dstatus: list
    vstatus: list
    ddiag: np.ndarray | None = None
    vdiag: np.ndarray | None = None


def gpu_cycle(w: W.Workload, diag=False, device="cuda") -> GpuResult:
    import torch
    d = engine.DeviceWorkload.from_workload(w, device)
    b = engine.Buffers.for_workload(d, device, diag=diag)
    engine.cycle(d, b)
    torch.cuda.synchronize()
    return GpuResult(b.draft_tokens.cpu().numpy(), b.q_tok.cpu().numpy(), b.lse_q.cpu().numpy(),
                     b.accept_len.cpu().numpy(), b.out_tokens.cpu().numpy(),
                     b.alpha.cpu().numpy(), b.p_tok.cpu().numpy(),
                     engine.status_words(b.dstatus), engine.status_words(b.vstatus),
                     b.ddiag.cpu().numpy() if diag else None,
                     b.vdiag.cpu().numpy() if diag else None)


@dataclasses.dataclass
class Report:
    rows: int
    mismatched: list          # request ids whose tokens / accept length differ
    far_mismatched: list      # ... of which no consumed uniform was near a boundary
    near_rows: int            # rows with a consumed uniform within BOUNDARY of a boundary
    max_q_err: float
    max_lse_err: float
    max_alpha_err: float
    max_ptok_err: float

    def summary(self) -> str:
        return (f"rows={self.rows} mismatched={len(self.mismatched)} far={len(self.far_mismatched)} "
                f"near={self.near_rows} q_err={self.max_q_err:.2e} lse_err={self.max_lse_err:.2e} "
                f"alpha_err={self.max_alpha_err:.2e} ptok_err={self.max_ptok_err:.2e}")


def compare(w: W.Workload, g: GpuResult, res: O.CycleResult, rows=None) -> Report:
    rows = list(range(w.B)) if rows is None else list(rows)
    mism, far = [], []
    near = 0
    qe = le = ae = pe = 0.0
    for i, b in enumerate(rows):
        dr, vr = res.draft[i], res.verify[i]
        dmin = res.row_dmin(i)
        if dmin < BOUNDARY:
            near += 1
        same_draft = np.array_equal(g.draft_tokens[b], dr.tokens)
        same = (same_draft and g.accept_len[b] == vr.accept_len
                and np.array_equal(g.out_tokens[b], vr.out_tokens))
        if not same:
            mism.append(b)
            if dmin >= BOUNDARY:
                far.append(b)
        if same_draft:
            qe = max(qe, float(np.max(np.abs(g.q_tok[b] - dr.q_tok))))
            le = max(le, float(np.max(np.abs(g.lse_q[b] - dr.lse_q))))
            L = int(w.verify_len[b])
            if L:
                ae = max(ae, float(np.max(np.abs(g.alpha[b, :L] - vr.alpha[:L]))))
                pe = max(pe, float(np.max(np.abs(g.p_tok[b, :L] - vr.p_tok[:L]))))
            assert np.all(np.isnan(g.alpha[b, L:])), b
    return Report(len(rows), mism, far, near, qe, le, ae, pe)


def assert_parity(rep: Report, max_mismatch_rate: float = 1e-4) -> None:
    assert not rep.far_mismatched, f"mismatch away from any boundary: {rep.far_mismatched}; {rep.summary()}"
    assert len(rep.mismatched) <= max_mismatch_rate * rep.rows, rep.summary()
    assert rep.max_q_err <= FLOAT_TOL, rep.summary()
    assert rep.max_lse_err <= FLOAT_TOL, rep.summary()
    assert rep.max_alpha_err <= FLOAT_TOL, rep.summary()
    assert rep.max_ptok_err <= FLOAT_TOL, rep.summary()
