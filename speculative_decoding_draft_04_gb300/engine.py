"""Device-side plumbing around the C ABI: moves a seeded workload to the GPU
(torch allocations), owns the output buffers and the workspace, and
enqueues one speculative cycle (spec_markov_draft then spec_verify) on a
stream, or the confidence-scheduled cycle (draft, spec_confidence,
spec_prefix_schedule, then spec_verify with the scheduled lengths).
Nothing here computes any part of the method."""
from __future__ import annotations

import dataclasses

import numpy as np

from . import _lib
from .workloads import RnnInputs, ScheduleInputs, TreeInputs, Workload


def _dev_logits(arr: np.ndarray, dtype: str, device):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(device)


@dataclasses.dataclass
class DeviceWorkload:
    B: int
    gamma: int
    V: int
    r: int
    dtype: str
    target: object
    U: object
    W1: object
    W2: object
    anchor: object
    temperature: object
    verify_len: object
    u_draft: object
    u_accept: object
    u_final: object

    @classmethod
    def from_workload(cls, w: Workload, device="cuda") -> "DeviceWorkload":
        import torch

        def i32(a):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)

        def f32(a):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)

        return cls(w.B, w.gamma, w.V, w.r, w.dtype, _dev_logits(w.target, w.dtype, device),
                   _dev_logits(w.U, w.dtype, device), _dev_logits(w.W1, w.dtype, device),
                   _dev_logits(w.W2, w.dtype, device), i32(w.anchor), f32(w.temperature),
                   i32(w.verify_len), f32(w.u_draft), f32(w.u_accept), f32(w.u_final))

    @property
    def dtype_code(self) -> int:
        return _lib.SPEC_BF16 if self.dtype == "bf16" else _lib.SPEC_F32


@dataclasses.dataclass
class Buffers:
    draft_tokens: object
    q_tok: object
    lse_q: object
    dstatus: object
    accept_len: object
    out_tokens: object
    alpha: object
    p_tok: object
    vstatus: object
    workspace: object
    ddiag: object = None
    vdiag: object = None

    @classmethod
    def allocate(cls, B, gamma, V, r, dtype_code, device="cuda", diag=False) -> "Buffers":
        import torch
        nbytes = _lib.spec_workspace_bytes(B, gamma, V, r, dtype_code)
        if nbytes == 0:
            raise _lib.SpecError("unsupported shape for libspec")
        o = dict(device=device)
        return cls(
            draft_tokens=torch.empty((B, gamma), dtype=torch.int32, **o),
            q_tok=torch.empty((B, gamma), dtype=torch.float32, **o),
            lse_q=torch.empty((B, gamma), dtype=torch.float64, **o),
            dstatus=torch.zeros(4, dtype=torch.int32, **o),
            accept_len=torch.empty(B, dtype=torch.int32, **o),
            out_tokens=torch.empty((B, gamma + 1), dtype=torch.int32, **o),
            alpha=torch.empty((B, gamma), dtype=torch.float32, **o),
            p_tok=torch.empty((B, gamma), dtype=torch.float32, **o),
            vstatus=torch.zeros(4, dtype=torch.int32, **o),
            workspace=torch.empty(nbytes, dtype=torch.uint8, **o),
            ddiag=torch.empty((B, gamma, 4), dtype=torch.float32, **o) if diag else None,
            vdiag=torch.empty((B, 4), dtype=torch.float32, **o) if diag else None,
        )

    @classmethod
    def for_workload(cls, d: DeviceWorkload, device="cuda", diag=False) -> "Buffers":
        return cls.allocate(d.B, d.gamma, d.V, d.r, d.dtype_code, device, diag)


def draft(d: DeviceWorkload, b: Buffers, stream=None) -> None:
    _lib.spec_markov_draft(d.U, d.W1, d.W2, d.anchor, d.temperature, d.u_draft, b.draft_tokens,
                           b.q_tok, b.lse_q, b.dstatus, b.workspace, diag=b.ddiag, stream=stream)


def verify(d: DeviceWorkload, b: Buffers, stream=None, draft_tokens=None, q_tok=None,
           lse_q=None, verify_len=None) -> None:
    _lib.spec_verify(d.target, d.U, d.W1, d.W2, d.anchor, d.temperature,
                     b.draft_tokens if draft_tokens is None else draft_tokens,
                     b.q_tok if q_tok is None else q_tok,
                     b.lse_q if lse_q is None else lse_q,
                     d.verify_len if verify_len is None else verify_len, d.u_accept, d.u_final,
                     b.accept_len, b.out_tokens, b.alpha, b.vstatus, b.workspace, p_tok=b.p_tok,
                     diag=b.vdiag, stream=stream)


def cycle(d: DeviceWorkload, b: Buffers, stream=None) -> None:
    """One speculative cycle: draft gamma tokens per request, then verify them."""
    draft(d, b, stream)
    verify(d, b, stream)


@dataclasses.dataclass
class HostStep:
    """One cycle's inputs and results in page-locked host memory."""
    U: object
    target: object
    anchor: object
    temperature: object
    u_draft: object
    verify_len: object
    u_accept: object
    u_final: object
    accept_len: object
    out_tokens: object
    draft_tokens: object
    alpha: object

    @classmethod
    def like(cls, d: DeviceWorkload) -> "HostStep":
        """Pinned copies of d's per-cycle inputs, and pinned result buffers."""
        import torch

        def pin(t):
            return t.cpu().pin_memory()

        def out(shape, dtype):
            return torch.empty(shape, dtype=dtype).pin_memory()
        B, g = d.B, d.gamma
        return cls(pin(d.U), pin(d.target), pin(d.anchor), pin(d.temperature), pin(d.u_draft),
                   pin(d.verify_len), pin(d.u_accept), pin(d.u_final),
                   out((B,), torch.int32), out((B, g + 1), torch.int32),
                   out((B, g), torch.int32), out((B, g), torch.float32))

    def h2d_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in
                   (self.U, self.target, self.anchor, self.temperature, self.u_draft,
                    self.verify_len, self.u_accept, self.u_final))

    def d2h_bytes(self, with_extras: bool = False) -> int:
        ts = [self.accept_len, self.out_tokens] + ([self.draft_tokens, self.alpha]
                                                   if with_extras else [])
        return sum(t.numel() * t.element_size() for t in ts)


def cycle_host(d: DeviceWorkload, b: Buffers, h: HostStep, stream=None, copy_stream=None,
               extras: bool = False) -> None:
    """One cycle through spec_cycle_host: h's inputs are copied into d's device
    buffers, the cycle runs, and accept_len / out_tokens (with ``extras`` also
    draft_tokens / alpha) are copied back into h."""
    da = _lib.draft_args(d.U, d.W1, d.W2, d.anchor, d.temperature, d.u_draft, b.draft_tokens,
                         b.q_tok, b.lse_q, b.dstatus, b.workspace, diag=b.ddiag)
    va = _lib.verify_args(d.target, d.U, d.W1, d.W2, d.anchor, d.temperature, b.draft_tokens,
                          b.q_tok, b.lse_q, d.verify_len, d.u_accept, d.u_final, b.accept_len,
                          b.out_tokens, b.alpha, b.vstatus, b.workspace, p_tok=b.p_tok,
                          diag=b.vdiag)
    _lib.spec_cycle_host(da, va, h.U, h.target, h.anchor, h.temperature, h.u_draft,
                         h.verify_len, h.u_accept, h.u_final, h.accept_len, h.out_tokens,
                         h.draft_tokens if extras else None, h.alpha if extras else None,
                         stream=stream, copy_stream=copy_stream)


@dataclasses.dataclass
class DeviceSchedule:
    """Confidence-head inputs, the cost table and the scheduler's outputs."""
    hidden: object
    w: object
    sps: object
    conf: object
    survival: object
    verify_len: object
    totals: object
    theta: object
    status: object
    workspace: object

    @classmethod
    def from_inputs(cls, s: ScheduleInputs, B: int, gamma: int, dtype: str,
                    device="cuda") -> "DeviceSchedule":
        import torch
        o = dict(device=device)
        nbytes = _lib.spec_schedule_workspace_bytes(B, gamma)
        if nbytes == 0:
            raise _lib.SpecError("unsupported shape for the scheduler")
        return cls(hidden=_dev_logits(s.hidden, dtype, device),
                   w=torch.from_numpy(np.ascontiguousarray(s.w, dtype=np.float32)).to(device),
                   sps=torch.from_numpy(np.ascontiguousarray(s.sps, dtype=np.float64)).to(device),
                   conf=torch.empty((B, gamma), dtype=torch.float32, **o),
                   survival=torch.empty((B, gamma), dtype=torch.float32, **o),
                   verify_len=torch.empty(B, dtype=torch.int32, **o),
                   totals=torch.empty(4, dtype=torch.int64, **o),
                   theta=torch.empty(1, dtype=torch.float64, **o),
                   status=torch.zeros(4, dtype=torch.int32, **o),
                   workspace=torch.empty(nbytes, dtype=torch.uint8, **o))


def schedule(d: DeviceWorkload, b: Buffers, s: DeviceSchedule, stream=None) -> None:
    """Confidence of every drafted row, then the verify lengths."""
    _lib.spec_confidence(s.hidden, d.W1, s.w, d.anchor, b.draft_tokens, s.conf, s.status, stream)
    _lib.spec_prefix_schedule(s.conf, s.sps, s.survival, s.verify_len, s.totals, s.theta, s.status,
                              s.workspace, stream)


def scheduled_cycle(d: DeviceWorkload, b: Buffers, s: DeviceSchedule, stream=None) -> None:
    """Draft, schedule, and verify each request up to its scheduled length."""
    draft(d, b, stream)
    schedule(d, b, s, stream)
    verify(d, b, stream, verify_len=s.verify_len)


@dataclasses.dataclass
class DeviceRnn:
    """RNN head inputs on the device and its factor rows (draft output)."""
    Wr: object
    hproj: object
    a_rows: object

    @classmethod
    def from_inputs(cls, s: RnnInputs, d: DeviceWorkload, device="cuda") -> "DeviceRnn":
        import torch
        a = torch.empty((d.gamma, d.B, d.r), dtype=d.W1.dtype, device=device)
        return cls(Wr=_dev_logits(s.Wr, d.dtype, device),
                   hproj=torch.from_numpy(np.ascontiguousarray(s.hproj)).to(device), a_rows=a)


def rnn_draft(d: DeviceWorkload, b: Buffers, h: DeviceRnn, stream=None) -> None:
    _lib.spec_rnn_draft(d.U, d.W1, d.W2, h.Wr, h.hproj, d.anchor, d.temperature, d.u_draft,
                        b.draft_tokens, b.q_tok, b.lse_q, h.a_rows, b.dstatus, b.workspace,
                        diag=b.ddiag, stream=stream)


def rnn_cycle(d: DeviceWorkload, b: Buffers, h: DeviceRnn, stream=None) -> None:
    """One speculative cycle with the RNN head: draft, then verify with its
    factor rows."""
    rnn_draft(d, b, h, stream)
    _lib.spec_verify(d.target, d.U, d.W1, d.W2, d.anchor, d.temperature, b.draft_tokens, b.q_tok,
                     b.lse_q, d.verify_len, d.u_accept, d.u_final, b.accept_len, b.out_tokens,
                     b.alpha, b.vstatus, b.workspace, p_tok=b.p_tok, diag=b.vdiag, stream=stream,
                     a_rows=h.a_rows)


@dataclasses.dataclass
class DeviceTree:
    """A batch of candidate trees on the device and the tree path's outputs."""
    N: int
    n: int
    parent: object
    conf: object
    target: object
    u_draft: object
    u_accept: object
    u_final: object
    survival: object
    mask: object
    tokens: object
    q_tok: object
    accept_len: object
    out_tokens: object
    path: object
    status: object
    workspace: object

    @classmethod
    def from_inputs(cls, t: TreeInputs, d: DeviceWorkload, n: int, device="cuda") -> "DeviceTree":
        import torch
        o = dict(device=device)
        B, N = t.parent.shape

        def dev(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(device)
        nbytes = _lib.spec_tree_workspace_bytes(B, N, d.V)
        return cls(N=N, n=n, parent=dev(t.parent), conf=dev(t.conf),
                   target=_dev_logits(t.target, d.dtype, device), u_draft=dev(t.u_draft),
                   u_accept=dev(t.u_accept), u_final=dev(t.u_final),
                   survival=torch.empty((B, N), dtype=torch.float32, **o),
                   mask=torch.empty((B, N), dtype=torch.uint8, **o),
                   tokens=torch.full((B, N), -1, dtype=torch.int32, **o),
                   q_tok=torch.full((B, N), float("nan"), dtype=torch.float32, **o),
                   accept_len=torch.empty(B, dtype=torch.int32, **o),
                   out_tokens=torch.empty((B, d.gamma + 1), dtype=torch.int32, **o),
                   path=torch.empty((B, d.gamma), dtype=torch.int32, **o),
                   status=torch.zeros(4, dtype=torch.int32, **o),
                   workspace=torch.empty(nbytes, dtype=torch.uint8, **o))


def tree_cycle(d: DeviceWorkload, t: DeviceTree, stream=None) -> None:
    """Select each request's tree, draft it, verify it."""
    _lib.spec_tree_select(t.parent, t.conf, t.n, t.survival, t.mask, t.status, d.gamma,
                          stream=stream)
    _lib.spec_tree_draft(d.U, d.W1, d.W2, d.anchor, d.temperature, t.parent, t.mask, t.u_draft,
                         t.tokens, t.q_tok, t.status, t.workspace, stream)
    _lib.spec_tree_verify(t.target, d.U, d.W1, d.W2, d.anchor, d.temperature, t.parent, t.mask,
                          t.tokens, t.u_accept, t.u_final, t.accept_len, t.out_tokens, t.path,
                          t.status, t.workspace, stream)


def status_words(t) -> list[int]:
    return [int(x) & 0xFFFFFFFF for x in t.cpu().tolist()]
