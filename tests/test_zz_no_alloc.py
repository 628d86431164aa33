"""spec_markov_draft_static: the draft for callers that cannot allocate device
memory (code running under someone else's stream capture, services with a
fixed device-memory budget, plug-ins that only receive a stream).  It uses
the library's built-in scratch area instead of a caller workspace; here it is
called through the C ABI and must reproduce spec_markov_draft's outputs on
two calls in a row.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from speculative_decoding_draft_04_gb300 import _lib, engine  # noqa: E402
from speculative_decoding_draft_04_gb300 import build as B  # noqa: E402
from speculative_decoding_draft_04_gb300 import workloads as W  # noqa: E402

TOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    _lib.lib()
    _lib.spec_set_option(_lib.SPEC_OPT_FORCE_SIMT, 0)
    _lib.spec_set_option(_lib.SPEC_OPT_EPS_SCALE, 1.0)
    _lib.spec_set_option(_lib.SPEC_OPT_BIAS_PATH, 2)


def _draft_both(w):
    d = engine.DeviceWorkload.from_workload(w)
    ref = engine.Buffers.for_workload(d)
    engine.draft(d, ref)
    out = dict(tok=torch.empty_like(ref.draft_tokens), q=torch.empty_like(ref.q_tok),
               lse=torch.empty_like(ref.lse_q), st=torch.zeros(4, dtype=torch.int32, device="cuda"))
    _lib.spec_markov_draft_static(d.U, d.W1, d.W2, d.anchor, d.temperature, d.u_draft,
                                  out["tok"], out["q"], out["lse"], out["st"])
    torch.cuda.synchronize()
    return ref, out


def _check(ref, out):
    np.testing.assert_array_equal(out["tok"].cpu().numpy(), ref.draft_tokens.cpu().numpy())
    np.testing.assert_allclose(out["q"].cpu().numpy(), ref.q_tok.cpu().numpy(), atol=TOL, rtol=0)
    np.testing.assert_allclose(out["lse"].cpu().numpy(), ref.lse_q.cpu().numpy(), atol=TOL, rtol=0)
    st_ref = engine.status_words(ref.dstatus)
    st = engine.status_words(out["st"])
    assert st[0] & ~16 == 0 and st_ref[0] & ~16 == 0, (st, st_ref)


@pytest.mark.parametrize("name,overrides", [("C2", {}), ("C4", {}), ("C0", {})])
def test_static_draft_matches_workspace_draft_twice(name, overrides):
    """Two consecutive calls on different inputs (no state carried between
    them), each equal to the workspace entry point's result."""
    for trial in (0, 1):
        w = W.make_workload(W.config(name, **overrides), trial=trial)
        ref, out = _draft_both(w)
        _check(ref, out)


MODES = {
    # each kernel family the static entry point can run
    "simt": {_lib.SPEC_OPT_FORCE_SIMT: 1},
    "warp-mma": {_lib.SPEC_OPT_BIAS_PATH: 1},
    "tile-strided": {_lib.SPEC_OPT_DRAFT_KERNEL: 1},
    # most draws queued: the queue, block sums and counters in the shared
    # area carry state from one call's re-decisions to the next call's
    "re-decided": {_lib.SPEC_OPT_EPS_SCALE: 3000.0},
    # every queued draw first writes a wrong token, so re-decisions change
    # tokens and the later steps are redone
    "redo": {_lib.SPEC_OPT_EPS_SCALE: 3000.0, _lib.SPEC_OPT_PERTURB: 1},
}
DEFAULTS = {_lib.SPEC_OPT_FORCE_SIMT: 0, _lib.SPEC_OPT_BIAS_PATH: 2, _lib.SPEC_OPT_DRAFT_KERNEL: 0,
            _lib.SPEC_OPT_EPS_SCALE: 1.0, _lib.SPEC_OPT_PERTURB: 0}


@pytest.mark.parametrize("mode", list(MODES))
def test_static_draft_in_every_mode(mode):
    """Two calls in a row per mode, each equal to the workspace draft run in the
    same mode; in the re-decision modes the re-decisions (and the redo) must
    actually have run through the shared area."""
    spec = W.config("C2", B=48, V=8200, r=256, name="noalloc-mode")
    try:
        for k, v in MODES[mode].items():
            _lib.spec_set_option(k, v)
        for trial in (2, 3):
            w = W.make_workload(spec, trial=trial)
            ref, out = _draft_both(w)
            _check(ref, out)
            st = engine.status_words(out["st"])
            if mode in ("re-decided", "redo"):
                assert st[1] > 0, st              # re-decisions ran
            if mode == "redo":
                assert st[2] > 0, st              # ... changed tokens, and the steps were redone
    finally:
        for k, v in DEFAULTS.items():
            _lib.spec_set_option(k, v)


def test_static_draft_rejects_problems_beyond_its_scratch():
    L = _lib.lib()
    a = _lib.DraftArgs(4096, 16, 8 << 20, 256, _lib.SPEC_BF16)
    for f in ("U", "W1", "W2", "anchor", "temperature", "u_draft", "draft_tokens", "q_tok",
              "lse_q", "dev_status"):
        setattr(a, f, 0x100000)
    assert L.spec_markov_draft_static(ctypes.byref(a), None) == -4   # SPEC_EWORKSPACE
    assert L.spec_markov_draft_static(None, None) == -1
