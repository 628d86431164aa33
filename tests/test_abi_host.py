"""The C-ABI library on the host: it loads, exports every entry point that
include/spec.h declares, and its host-side checks reject bad arguments
before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

from speculative_decoding_draft_04_gb300 import _lib
from speculative_decoding_draft_04_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    B.build()
    return _lib.lib()


def declared_functions():
    with open(os.path.join(ROOT, "include", "spec.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[\w]+\**\s+\**(spec_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert "spec_markov_draft" in names and "spec_verify" in names
    for n in names:
        assert hasattr(L, n), n
    assert set(_lib.EXPORTED) <= set(names)


def test_workspace_and_shape_checks(L):
    assert _lib.spec_workspace_bytes(128, 7, 32000, 256, _lib.SPEC_BF16) > 0
    assert _lib.spec_workspace_bytes(4, 4, 1000, 16, _lib.SPEC_F32) > 0
    # unsupported / invalid shapes report 0
    for args in [(0, 7, 32000, 256, 1), (8, 17, 32000, 256, 1), (8, 7, 32004, 256, 1),
                 (8, 7, 32000, 250, 1), (8, 7, 32000, 512, 1), (8, 7, 32000, 128, 0),
                 (8, 7, 32000, 256, 7), (5000, 7, 32000, 256, 1)]:
        assert _lib.spec_workspace_bytes(*args) == 0, args


def _draft_args(**kw):
    a = _lib.DraftArgs(8, 4, 1024, 64, _lib.SPEC_BF16)
    for f in ("U", "W1", "W2", "anchor", "temperature", "u_draft", "draft_tokens", "q_tok",
              "lse_q", "dev_status"):
        setattr(a, f, 0x100000)
    a.workspace = 0x200000
    a.workspace_bytes = 1 << 40
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_draft_host_validation(L):
    call = lambda a: L.spec_markov_draft(ctypes.byref(a), None)  # noqa: E731
    assert L.spec_markov_draft(None, None) == -1
    assert call(_draft_args(U=None)) == -1                     # NULL tensor
    assert call(_draft_args(dev_status=None)) == -1
    assert call(_draft_args(gamma=0)) == -1                    # size out of range
    assert call(_draft_args(gamma=17)) == -2                   # unsupported
    assert call(_draft_args(r=24)) == -2
    assert call(_draft_args(dtype=3)) == -2
    assert call(_draft_args(U=0x100008)) == -3                 # misaligned
    assert call(_draft_args(lse_q=0x100004)) == -3
    assert call(_draft_args(workspace=None)) == -4             # workspace
    assert call(_draft_args(workspace_bytes=16)) == -4
    assert call(_draft_args(workspace=0x200010)) == -3


def test_verify_host_validation(L):
    a = _lib.VerifyArgs(8, 4, 1024, 64, _lib.SPEC_BF16)
    for f, _ in _lib.VerifyArgs._fields_[5:-2]:
        setattr(a, f, 0x100000)
    a.p_tok = None
    a.diag = None
    a.workspace = 0x200000
    a.workspace_bytes = 1 << 40
    call = lambda: L.spec_verify(ctypes.byref(a), None)  # noqa: E731
    a.target = None
    assert call() == -1
    a.target = 0x100002
    assert call() == -3
    a.target = 0x100000
    a.workspace_bytes = 100
    assert call() == -4


def test_cycle_host_validation(L):
    """spec_cycle_host checks both argument blocks, their agreement and the
    host pointers before it enqueues anything."""
    def cycle(**kw):
        v = _lib.VerifyArgs(8, 4, 1024, 64, _lib.SPEC_BF16)
        for f, _ in _lib.VerifyArgs._fields_[5:-2]:
            setattr(v, f, 0x100000)
        v.p_tok = v.diag = v.a_rows = None
        v.workspace, v.workspace_bytes = 0x200000, 1 << 40
        c = _lib.CycleHostArgs(_draft_args(), v)
        for f, _ in _lib.CycleHostArgs._fields_[2:-3]:
            setattr(c, f, 0x300000)
        for k, val in kw.items():
            obj, _, f = k.partition("__")
            if f:
                setattr(getattr(c, obj), f, val)
            else:
                setattr(c, k, val)
        return L.spec_cycle_host(ctypes.byref(c), None)
    assert L.spec_cycle_host(None, None) == -1
    assert cycle(draft__U=None) == -1                   # the draft's own checks
    assert cycle(verify__target=0x100002) == -3         # the verification's
    assert cycle(verify__V=2048) == -1                  # the two blocks disagree
    assert cycle(verify__draft_tokens=0x100100) == -1
    assert cycle(verify__workspace=0x300000) == -1
    assert cycle(h_target=None) == -1                   # a host input missing
    assert cycle(h_out_tokens=None) == -1


def test_status_strings_and_options(L):
    for code in (0, -1, -2, -3, -4, -5, 99):
        assert isinstance(_lib.spec_status_string(code), str)
    assert _lib.spec_status_string(-4).startswith("workspace")
    assert L.spec_set_option(999, 1.0) == -1
    assert L.spec_set_option(_lib.SPEC_OPT_EPS_SCALE, -1.0) == -1
    assert L.spec_set_option(_lib.SPEC_OPT_EPS_SCALE, 1.0) == 0
    n = L.spec_num_stages()
    names = [L.spec_stage_name(i).decode() for i in range(n)]
    assert "draft_persistent" in names and "verify_tile" in names and len(set(names)) == n
    assert {"confidence", "sched_rank", "sched_select"} <= set(names)
    assert L.spec_set_option(4, 1.0) == -1          # unused key


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(_lib.SpecError):
        _lib.lib(str(tmp_path / "nope.so"))


def test_confidence_host_validation(L):
    def args(**kw):
        a = _lib.ConfidenceArgs(8, 4, 64, 1000, 16, _lib.SPEC_BF16)
        for f in ("hidden", "W1", "w", "anchor", "draft_tokens", "conf", "dev_status"):
            setattr(a, f, 0x100000)
        for k, v in kw.items():
            setattr(a, k, v)
        return a
    call = lambda a: L.spec_confidence(ctypes.byref(a), None)  # noqa: E731
    assert L.spec_confidence(None, None) == -1
    assert call(args(hidden=None)) == -1
    assert call(args(R=0)) == -1 and call(args(R=4097)) == -1
    assert call(args(d=4)) == -1
    assert call(args(gamma=17)) == -2 and call(args(d=12)) == -2 and call(args(r=24)) == -2
    assert call(args(r=512)) == -2 and call(args(dtype=2)) == -2
    assert call(args(hidden=0x100008)) == -3 and call(args(w=0x100004)) == -3


def test_schedule_host_validation(L):
    assert _lib.spec_schedule_workspace_bytes(128, 7) == 128 * 7 * 4 + 128 * 7 * 8
    assert _lib.spec_schedule_workspace_bytes(0, 7) == 0
    assert _lib.spec_schedule_workspace_bytes(8, 17) == 0

    def args(**kw):
        a = _lib.ScheduleArgs(8, 4)
        for f in ("conf", "sps", "survival", "verify_len", "totals", "theta", "dev_status"):
            setattr(a, f, 0x100000)
        a.sps_len = 41
        a.workspace = 0x200000
        a.workspace_bytes = 1 << 20
        for k, v in kw.items():
            setattr(a, k, v)
        return a
    call = lambda a: L.spec_prefix_schedule(ctypes.byref(a), None)  # noqa: E731
    assert L.spec_prefix_schedule(None, None) == -1
    assert call(args(conf=None)) == -1
    assert call(args(sps_len=8)) == -1            # the table must cover B = R
    assert call(args(gamma=17)) == -2
    assert call(args(totals=0x100004)) == -3
    assert call(args(workspace=None)) == -4 and call(args(workspace_bytes=64)) == -4
    assert call(args(workspace=0x200008)) == -3
