"""The draft re-decides a step's near-boundary draws during the next step's
tile phase; a re-decision that changes a token sends the later steps of the
draft through a redo.  Changed tokens are rare, so these tests force them:
with the SPEC_OPT_PERTURB hook every queued draw first writes the next token,
the re-decision restores the exact one, and the redo must leave the cycle
identical to the float64 oracle (Markov and RNN heads)."""
import numpy as np
import pytest

from speculative_decoding_draft_04_gb300 import workloads as W

from parity import assert_parity, compare, gpu_cycle, oracle_cycle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_draft_04_gb300 import build as B
    B.build()
    return t


@pytest.fixture()
def perturbed():
    from speculative_decoding_draft_04_gb300 import _lib
    _lib.spec_set_option(_lib.SPEC_OPT_PERTURB, 1)
    _lib.spec_set_option(_lib.SPEC_OPT_EPS_SCALE, 3000.0)   # most draws queued
    yield
    _lib.spec_set_option(_lib.SPEC_OPT_PERTURB, 0)
    _lib.spec_set_option(_lib.SPEC_OPT_EPS_SCALE, 1.0)


SMALL = dict(W.config("C4"), B=40, gamma=5, V=4104, r=64, name="small-ragged")


@pytest.mark.parametrize("spec,B", [(W.config("C0"), None), (SMALL, None), (W.config("C2"), 24)])
def test_redo_after_changed_tokens(torch, perturbed, spec, B):
    w = W.make_workload(spec, trial=1, B=B)
    g = gpu_cycle(w)
    assert g.dstatus[2] > 0, g.dstatus                     # tokens were changed and redone
    assert_parity(compare(w, g, oracle_cycle(w)))


def test_redo_with_the_rnn_head(torch, perturbed):
    from test_rnn_gpu import check_factor_rows, run_gpu, run_oracle
    spec = W.config("C2")
    w = W.make_workload(spec, 0, B=16)
    ri = W.make_rnn_inputs(spec, 0, B=16)
    g, a_gpu = run_gpu(torch, w, ri)
    assert g.dstatus[2] > 0, g.dstatus
    res, a_ref = run_oracle(w, ri)
    check_factor_rows(g, res, a_gpu, a_ref)
    assert_parity(compare(w, g, res))


def test_perturb_hook_is_off_by_default(torch):
    w = W.make_workload(W.config("C0"), trial=2)
    g = gpu_cycle(w)
    assert_parity(compare(w, g, oracle_cycle(w)))
    assert np.all(g.draft_tokens >= 0)
