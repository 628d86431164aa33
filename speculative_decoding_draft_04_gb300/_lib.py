"""ctypes binding of libspec.so: the C ABI of include/spec.h, same names.

Argument marshalling only -- every step of the path runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (torch is used for device
memory and streams); pointers, sizes and the stream handle are passed as
plain integers.  There is no CPU fallback: if the library is missing or a
call fails, a SpecError is raised.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libspec.so")

SPEC_F32, SPEC_BF16 = 0, 1
SPEC_OPT_EPS_SCALE, SPEC_OPT_FORCE_SIMT, SPEC_OPT_BIAS_PATH, SPEC_OPT_TRACE = 1, 2, 3, 5
SPEC_OPT_PERTURB = 6
SPEC_OPT_TEST_STALL = 7
SPEC_OPT_DRAFT_KERNEL = 8
SPEC_OPT_VERIFY_KERNEL = 9
DEV_BITS = {1: "BAD_TOKEN", 2: "BAD_LEN", 4: "BAD_TEMP", 8: "TIMEOUT", 16: "REFINED",
            32: "OVERFLOW", 64: "BAD_CONF", 128: "BAD_TREE"}

EXPORTED = ("spec_workspace_bytes", "spec_markov_draft", "spec_markov_draft_static",
            "spec_verify", "spec_status_string",
            "spec_set_option", "spec_profile_enable", "spec_profile_read", "spec_stage_name",
            "spec_num_stages", "spec_operating_point", "spec_acceptance_stats",
            "spec_confidence", "spec_schedule_workspace_bytes", "spec_prefix_schedule",
            "spec_rnn_draft", "spec_tree_select", "spec_tree_draft", "spec_tree_verify",
            "spec_tree_workspace_bytes", "spec_cycle_host")


class SpecError(RuntimeError):
    pass


_i32, _vp, _sz = ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t


class DraftArgs(ctypes.Structure):
    _fields_ = [("B", _i32), ("gamma", _i32), ("V", _i32), ("r", _i32), ("dtype", _i32),
                ("U", _vp), ("W1", _vp), ("W2", _vp), ("anchor", _vp), ("temperature", _vp),
                ("u_draft", _vp), ("draft_tokens", _vp), ("q_tok", _vp), ("lse_q", _vp),
                ("dev_status", _vp), ("diag", _vp), ("workspace", _vp), ("workspace_bytes", _sz)]


class VerifyArgs(ctypes.Structure):
    _fields_ = [("B", _i32), ("gamma", _i32), ("V", _i32), ("r", _i32), ("dtype", _i32),
                ("target", _vp), ("U", _vp), ("W1", _vp), ("W2", _vp), ("anchor", _vp),
                ("temperature", _vp), ("draft_tokens", _vp), ("q_tok", _vp), ("lse_q", _vp),
                ("verify_len", _vp), ("u_accept", _vp), ("u_final", _vp), ("accept_len", _vp),
                ("out_tokens", _vp), ("alpha", _vp), ("p_tok", _vp), ("dev_status", _vp),
                ("a_rows", _vp), ("diag", _vp), ("workspace", _vp), ("workspace_bytes", _sz)]


class CycleHostArgs(ctypes.Structure):
    _fields_ = [("draft", DraftArgs), ("verify", VerifyArgs), ("h_U", _vp), ("h_target", _vp),
                ("h_anchor", _vp), ("h_temperature", _vp), ("h_u_draft", _vp),
                ("h_verify_len", _vp), ("h_u_accept", _vp), ("h_u_final", _vp),
                ("h_accept_len", _vp), ("h_out_tokens", _vp), ("h_draft_tokens", _vp),
                ("h_alpha", _vp), ("copy_stream", _vp)]


class RnnDraftArgs(ctypes.Structure):
    _fields_ = [("draft", DraftArgs), ("Wr", _vp), ("hproj", _vp), ("a_rows", _vp)]


_LIB = None


class OpArgs(ctypes.Structure):
    _fields_ = [("alpha", ctypes.c_double), ("c", ctypes.c_double), ("c_hat", ctypes.c_double),
                ("gamma", ctypes.c_int32), ("gamma_max", ctypes.c_int32)]


class OpResult(ctypes.Structure):
    _fields_ = [("expected_tau", ctypes.c_double), ("speedup", ctypes.c_double),
                ("speedup_gamma1", ctypes.c_double), ("bound", ctypes.c_double),
                ("gamma_continuous", ctypes.c_double), ("speedup_star", ctypes.c_double),
                ("compute_ratio", ctypes.c_double), ("gamma_star", ctypes.c_int32),
                ("gains", ctypes.c_int32)]


class ConfidenceArgs(ctypes.Structure):
    _fields_ = [("R", _i32), ("gamma", _i32), ("d", _i32), ("V", _i32), ("r", _i32),
                ("dtype", _i32), ("hidden", _vp), ("W1", _vp), ("w", _vp), ("anchor", _vp),
                ("draft_tokens", _vp), ("conf", _vp), ("dev_status", _vp)]


class ScheduleArgs(ctypes.Structure):
    _fields_ = [("R", _i32), ("gamma", _i32), ("conf", _vp), ("sps", _vp), ("sps_len", _i32),
                ("survival", _vp), ("verify_len", _vp), ("totals", _vp), ("theta", _vp),
                ("dev_status", _vp), ("workspace", _vp), ("workspace_bytes", _sz)]


class TreeDraftArgs(ctypes.Structure):
    _fields_ = [("B", _i32), ("N", _i32), ("gamma", _i32), ("V", _i32), ("r", _i32),
                ("dtype", _i32), ("U", _vp), ("W1", _vp), ("W2", _vp), ("anchor", _vp),
                ("temperature", _vp), ("parent", _vp), ("mask", _vp), ("u_draft", _vp),
                ("tokens", _vp), ("q_tok", _vp), ("dev_status", _vp), ("workspace", _vp),
                ("workspace_bytes", _sz)]


class TreeVerifyArgs(ctypes.Structure):
    _fields_ = [("B", _i32), ("N", _i32), ("gamma", _i32), ("V", _i32), ("r", _i32),
                ("dtype", _i32), ("target", _vp), ("U", _vp), ("W1", _vp), ("W2", _vp),
                ("anchor", _vp), ("temperature", _vp), ("parent", _vp), ("mask", _vp),
                ("tokens", _vp), ("u_accept", _vp), ("u_final", _vp), ("accept_len", _vp),
                ("out_tokens", _vp), ("path", _vp), ("dev_status", _vp), ("workspace", _vp),
                ("workspace_bytes", _sz)]


def lib(path: str | None = None) -> ctypes.CDLL:
    """Load libspec.so (built in-tree by build.build())."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise SpecError(f"{p} is missing: build it with speculative_decoding_draft_04_gb300."
                        "build.build() (there is no CPU fallback)")
    L = ctypes.CDLL(p)
    L.spec_workspace_bytes.restype = _sz
    L.spec_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32, _i32]
    L.spec_markov_draft.restype = _i32
    L.spec_markov_draft.argtypes = [ctypes.POINTER(DraftArgs), _vp]
    L.spec_markov_draft_static.restype = _i32
    L.spec_markov_draft_static.argtypes = [ctypes.POINTER(DraftArgs), _vp]
    L.spec_cycle_host.restype = _i32
    L.spec_cycle_host.argtypes = [ctypes.POINTER(CycleHostArgs), _vp]
    L.spec_verify.restype = _i32
    L.spec_verify.argtypes = [ctypes.POINTER(VerifyArgs), _vp]
    L.spec_status_string.restype = ctypes.c_char_p
    L.spec_status_string.argtypes = [_i32]
    L.spec_set_option.restype = _i32
    L.spec_set_option.argtypes = [_i32, ctypes.c_double]
    L.spec_profile_enable.restype = _i32
    L.spec_profile_enable.argtypes = [_i32]
    L.spec_profile_read.restype = _i32
    L.spec_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_i32), _i32]
    L.spec_stage_name.restype = ctypes.c_char_p
    L.spec_stage_name.argtypes = [_i32]
    L.spec_num_stages.restype = _i32
    L.spec_num_stages.argtypes = []
    L.spec_operating_point.restype = _i32
    L.spec_operating_point.argtypes = [ctypes.POINTER(OpArgs), ctypes.POINTER(OpResult)]
    L.spec_acceptance_stats.restype = _i32
    L.spec_acceptance_stats.argtypes = [_i32, _i32, _vp, _vp, _vp, _vp, _vp]
    L.spec_tree_select.restype = _i32
    L.spec_tree_select.argtypes = [_i32, _i32, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp]
    L.spec_tree_draft.restype = _i32
    L.spec_tree_draft.argtypes = [ctypes.POINTER(TreeDraftArgs), _vp]
    L.spec_tree_verify.restype = _i32
    L.spec_tree_verify.argtypes = [ctypes.POINTER(TreeVerifyArgs), _vp]
    L.spec_tree_workspace_bytes.restype = _sz
    L.spec_tree_workspace_bytes.argtypes = [_i32, _i32, _i32]
    L.spec_rnn_draft.restype = _i32
    L.spec_rnn_draft.argtypes = [ctypes.POINTER(RnnDraftArgs), _vp]
    L.spec_confidence.restype = _i32
    L.spec_confidence.argtypes = [ctypes.POINTER(ConfidenceArgs), _vp]
    L.spec_schedule_workspace_bytes.restype = _sz
    L.spec_schedule_workspace_bytes.argtypes = [_i32, _i32]
    L.spec_prefix_schedule.restype = _i32
    L.spec_prefix_schedule.argtypes = [ctypes.POINTER(ScheduleArgs), _vp]
    if path is None:
        _LIB = L
    return L


def _check(rc: int, what: str) -> None:
    if rc != 0:
        msg = lib().spec_status_string(rc).decode()
        raise SpecError(f"{what} failed: {rc} ({msg})")


def _hptr(t) -> int | None:
    """Address of a contiguous host (CPU) tensor."""
    if t is None:
        return None
    if t.is_cuda:
        raise SpecError("host buffers must be CPU tensors")
    if not t.is_contiguous():
        raise SpecError("tensors must be contiguous")
    return t.data_ptr()


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise SpecError("tensors must be CUDA tensors")
    if not t.is_contiguous():
        raise SpecError("tensors must be contiguous")
    return t.data_ptr()


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise SpecError(f"unsupported logits dtype {t.dtype}")


def _stream(stream) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def spec_workspace_bytes(B: int, gamma: int, V: int, r: int, dtype: int) -> int:
    return int(lib().spec_workspace_bytes(B, gamma, V, r, dtype))


def spec_status_string(status: int) -> str:
    return lib().spec_status_string(status).decode()


def spec_set_option(key: int, value: float) -> None:
    _check(lib().spec_set_option(key, float(value)), "spec_set_option")


def spec_markov_draft(U, W1, W2, anchor, temperature, u_draft, draft_tokens, q_tok, lse_q,
                      dev_status, workspace, diag=None, stream=None) -> None:
    """Enqueue the Markov-head draft (shapes as in include/spec.h)."""
    B, gamma, V = U.shape
    a = DraftArgs(B, gamma, V, W1.shape[1], _dtype_code(U), _ptr(U), _ptr(W1), _ptr(W2),
                  _ptr(anchor), _ptr(temperature), _ptr(u_draft), _ptr(draft_tokens),
                  _ptr(q_tok), _ptr(lse_q), _ptr(dev_status), _ptr(diag), _ptr(workspace),
                  workspace.numel() * workspace.element_size())
    _check(lib().spec_markov_draft(ctypes.byref(a), _stream(stream)), "spec_markov_draft")


def spec_markov_draft_static(U, W1, W2, anchor, temperature, u_draft, draft_tokens, q_tok,
                             lse_q, dev_status, diag=None, stream=None) -> None:
    """The draft with the library's built-in scratch area instead of a caller
    workspace, for callers that cannot allocate device memory (see spec.h)."""
    B, gamma, V = U.shape
    a = DraftArgs(B, gamma, V, W1.shape[1], _dtype_code(U), _ptr(U), _ptr(W1), _ptr(W2),
                  _ptr(anchor), _ptr(temperature), _ptr(u_draft), _ptr(draft_tokens),
                  _ptr(q_tok), _ptr(lse_q), _ptr(dev_status), _ptr(diag), None, 0)
    _check(lib().spec_markov_draft_static(ctypes.byref(a), _stream(stream)),
           "spec_markov_draft_static")


def spec_verify(target, U, W1, W2, anchor, temperature, draft_tokens, q_tok, lse_q, verify_len,
                u_accept, u_final, accept_len, out_tokens, alpha, dev_status, workspace,
                p_tok=None, diag=None, stream=None, a_rows=None) -> None:
    """Enqueue the verification (shapes as in include/spec.h); ``a_rows`` are
    the RNN head's factor rows (None: the Markov head)."""
    B, gamma, V = U.shape
    a = VerifyArgs(B, gamma, V, W1.shape[1], _dtype_code(U), _ptr(target), _ptr(U), _ptr(W1),
                   _ptr(W2), _ptr(anchor), _ptr(temperature), _ptr(draft_tokens), _ptr(q_tok),
                   _ptr(lse_q), _ptr(verify_len), _ptr(u_accept), _ptr(u_final),
                   _ptr(accept_len), _ptr(out_tokens), _ptr(alpha), _ptr(p_tok),
                   _ptr(dev_status), _ptr(a_rows), _ptr(diag), _ptr(workspace),
                   workspace.numel() * workspace.element_size())
    _check(lib().spec_verify(ctypes.byref(a), _stream(stream)), "spec_verify")


def spec_cycle_host(draft: DraftArgs, verify: VerifyArgs, h_U, h_target, h_anchor,
                    h_temperature, h_u_draft, h_verify_len, h_u_accept, h_u_final, h_accept_len,
                    h_out_tokens, h_draft_tokens=None, h_alpha=None, stream=None,
                    copy_stream=None) -> None:
    """Enqueue one cycle whose inputs and results live in host memory (CPU
    tensors, page-locked for asynchronous copies); ``draft`` / ``verify``
    name the device buffers (see include/spec.h)."""
    a = CycleHostArgs(draft, verify, _hptr(h_U), _hptr(h_target), _hptr(h_anchor),
                      _hptr(h_temperature), _hptr(h_u_draft), _hptr(h_verify_len),
                      _hptr(h_u_accept), _hptr(h_u_final), _hptr(h_accept_len),
                      _hptr(h_out_tokens), _hptr(h_draft_tokens), _hptr(h_alpha),
                      None if copy_stream is None else int(copy_stream.cuda_stream))
    _check(lib().spec_cycle_host(ctypes.byref(a), _stream(stream)), "spec_cycle_host")


def draft_args(U, W1, W2, anchor, temperature, u_draft, draft_tokens, q_tok, lse_q, dev_status,
               workspace, diag=None) -> DraftArgs:
    """The spec_draft_args of these device tensors."""
    B, gamma, V = U.shape
    return DraftArgs(B, gamma, V, W1.shape[1], _dtype_code(U), _ptr(U), _ptr(W1), _ptr(W2),
                     _ptr(anchor), _ptr(temperature), _ptr(u_draft), _ptr(draft_tokens),
                     _ptr(q_tok), _ptr(lse_q), _ptr(dev_status), _ptr(diag), _ptr(workspace),
                     workspace.numel() * workspace.element_size())


def verify_args(target, U, W1, W2, anchor, temperature, draft_tokens, q_tok, lse_q, verify_len,
                u_accept, u_final, accept_len, out_tokens, alpha, dev_status, workspace,
                p_tok=None, diag=None, a_rows=None) -> VerifyArgs:
    """The spec_verify_args of these device tensors."""
    B, gamma, V = U.shape
    return VerifyArgs(B, gamma, V, W1.shape[1], _dtype_code(U), _ptr(target), _ptr(U), _ptr(W1),
                      _ptr(W2), _ptr(anchor), _ptr(temperature), _ptr(draft_tokens),
                      _ptr(q_tok), _ptr(lse_q), _ptr(verify_len), _ptr(u_accept),
                      _ptr(u_final), _ptr(accept_len), _ptr(out_tokens), _ptr(alpha),
                      _ptr(p_tok), _ptr(dev_status), _ptr(a_rows), _ptr(diag), _ptr(workspace),
                      workspace.numel() * workspace.element_size())


def spec_profile_enable(on: bool) -> None:
    _check(lib().spec_profile_enable(1 if on else 0), "spec_profile_enable")


def spec_profile_read() -> dict[str, tuple[float, int]]:
    """{stage name: (total ms, launches)} since the previous read."""
    L = lib()
    n = L.spec_num_stages()
    ms = (ctypes.c_double * n)()
    cnt = (_i32 * n)()
    _check(L.spec_profile_read(ms, cnt, n), "spec_profile_read")
    return {L.spec_stage_name(i).decode(): (ms[i], cnt[i]) for i in range(n)}


def spec_operating_point(alpha: float, c: float, gamma: int, gamma_max: int = 256,
                         c_hat: float = 0.0) -> dict:
    """The analytic operating point (host computation, no GPU work)."""
    out = OpResult()
    _check(lib().spec_operating_point(ctypes.byref(OpArgs(alpha, c, c_hat, gamma, gamma_max)),
                                      ctypes.byref(out)), "spec_operating_point")
    return {f: getattr(out, f) for f, _ in OpResult._fields_}


def spec_acceptance_stats(alpha, verify_len, accept_len, out, stream=None) -> None:
    """Device sums (alpha over j < L_b, positions, tau, requests) into out (float64[4])."""
    B, gamma = alpha.shape
    _check(lib().spec_acceptance_stats(B, gamma, _ptr(alpha), _ptr(verify_len), _ptr(accept_len),
                                       _ptr(out), _stream(stream)), "spec_acceptance_stats")


def spec_confidence(hidden, W1, w, anchor, draft_tokens, conf, dev_status, stream=None) -> None:
    """Enqueue the confidence head: conf[r, k] = sigmoid(w . [h; W1[x_k]])."""
    R, gamma, d = hidden.shape
    V, r = W1.shape
    a = ConfidenceArgs(R, gamma, d, V, r, _dtype_code(hidden), _ptr(hidden), _ptr(W1), _ptr(w),
                       _ptr(anchor), _ptr(draft_tokens), _ptr(conf), _ptr(dev_status))
    _check(lib().spec_confidence(ctypes.byref(a), _stream(stream)), "spec_confidence")


def spec_schedule_workspace_bytes(R: int, gamma: int) -> int:
    return int(lib().spec_schedule_workspace_bytes(R, gamma))


def spec_prefix_schedule(conf, sps, survival, verify_len, totals, theta, dev_status, workspace,
                         stream=None) -> None:
    """Enqueue the hardware-aware prefix scheduler (verify lengths from conf)."""
    R, gamma = conf.shape
    a = ScheduleArgs(R, gamma, _ptr(conf), _ptr(sps), sps.numel(), _ptr(survival),
                     _ptr(verify_len), _ptr(totals), _ptr(theta), _ptr(dev_status),
                     _ptr(workspace), workspace.numel() * workspace.element_size())
    _check(lib().spec_prefix_schedule(ctypes.byref(a), _stream(stream)), "spec_prefix_schedule")


def spec_rnn_draft(U, W1, W2, Wr, hproj, anchor, temperature, u_draft, draft_tokens, q_tok,
                   lse_q, a_rows, dev_status, workspace, diag=None, stream=None) -> None:
    """Enqueue the RNN head draft (shapes as in include/spec.h)."""
    B, gamma, V = U.shape
    d = DraftArgs(B, gamma, V, W1.shape[1], _dtype_code(U), _ptr(U), _ptr(W1), _ptr(W2),
                  _ptr(anchor), _ptr(temperature), _ptr(u_draft), _ptr(draft_tokens),
                  _ptr(q_tok), _ptr(lse_q), _ptr(dev_status), _ptr(diag), _ptr(workspace),
                  workspace.numel() * workspace.element_size())
    a = RnnDraftArgs(d, _ptr(Wr), _ptr(hproj), _ptr(a_rows))
    _check(lib().spec_rnn_draft(ctypes.byref(a), _stream(stream)), "spec_rnn_draft")


def spec_tree_workspace_bytes(B: int, N: int, V: int) -> int:
    return int(lib().spec_tree_workspace_bytes(B, N, V))


def spec_tree_select(parent, conf, n, survival, mask, dev_status, gamma, expected=None,
                     stream=None) -> None:
    """Top-n slots of each request's candidate tree by survival."""
    B, N = parent.shape
    _check(lib().spec_tree_select(B, N, gamma, _ptr(parent), _ptr(conf), n, _ptr(survival),
                                  _ptr(mask), _ptr(expected), _ptr(dev_status), _stream(stream)),
           "spec_tree_select")


def spec_tree_draft(U, W1, W2, anchor, temperature, parent, mask, u_draft, tokens, q_tok,
                    dev_status, workspace, stream=None) -> None:
    B, gamma, V = U.shape
    a = TreeDraftArgs(B, parent.shape[1], gamma, V, W1.shape[1], _dtype_code(U), _ptr(U),
                      _ptr(W1), _ptr(W2), _ptr(anchor), _ptr(temperature), _ptr(parent),
                      _ptr(mask), _ptr(u_draft), _ptr(tokens), _ptr(q_tok), _ptr(dev_status),
                      _ptr(workspace), workspace.numel() * workspace.element_size())
    _check(lib().spec_tree_draft(ctypes.byref(a), _stream(stream)), "spec_tree_draft")


def spec_tree_verify(target, U, W1, W2, anchor, temperature, parent, mask, tokens, u_accept,
                     u_final, accept_len, out_tokens, path, dev_status, workspace,
                     stream=None) -> None:
    B, gamma, V = U.shape
    a = TreeVerifyArgs(B, parent.shape[1], gamma, V, W1.shape[1], _dtype_code(U), _ptr(target),
                       _ptr(U), _ptr(W1), _ptr(W2), _ptr(anchor), _ptr(temperature), _ptr(parent),
                       _ptr(mask), _ptr(tokens), _ptr(u_accept), _ptr(u_final), _ptr(accept_len),
                       _ptr(out_tokens), _ptr(path), _ptr(dev_status), _ptr(workspace),
                       workspace.numel() * workspace.element_size())
    _check(lib().spec_tree_verify(ctypes.byref(a), _stream(stream)), "spec_tree_verify")
