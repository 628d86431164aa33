"""The two persistent draft kernels behind spec_markov_draft, against the
float64 oracle and against each other, and the bounded-wait error path.

* The slice-resident kernel (each CTA keeps the W2 columns of one vocabulary
  slice in shared memory for every step; B <= 128, V <= 256 x SMs) runs by
  default where it fits; SPEC_OPT_DRAFT_KERNEL = 1 forces the tile-strided
  kernel.  Shapes below span 1 to 8 chunks of 32 columns per CTA (MMAs of
  N = 32 to 256, U chunks in the ring only or also in the A tile's space),
  ragged vocabulary tails, r = 64 / 128 / 256, and rows beyond B.
* Both kernels must reproduce the oracle (tokens and accept lengths
  bit-exact up to the near-boundary rule, probabilities within 1e-5) and,
  request by request, each other's tokens.
* SPEC_OPT_TEST_STALL runs a test build whose first grid barrier waits for a
  CTA that does not exist: the launch must return with SPEC_DEV_TIMEOUT set
  after its one-second limit, and the next normal call on the same context
  must be exact again (the kernel drained its copies and freed its tensor
  memory)."""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from speculative_decoding_draft_04_gb300 import _lib, engine  # noqa: E402
from speculative_decoding_draft_04_gb300 import build as B  # noqa: E402
from speculative_decoding_draft_04_gb300 import workloads as W  # noqa: E402

from parity import assert_parity, compare, gpu_cycle, oracle_cycle  # noqa: E402

TIMEOUT = 8


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    _lib.lib()
    _lib.spec_set_option(_lib.SPEC_OPT_FORCE_SIMT, 0)
    _lib.spec_set_option(_lib.SPEC_OPT_EPS_SCALE, 1.0)
    _lib.spec_set_option(_lib.SPEC_OPT_BIAS_PATH, 2)
    _lib.spec_set_option(_lib.SPEC_OPT_DRAFT_KERNEL, 0)
    yield
    _lib.spec_set_option(_lib.SPEC_OPT_DRAFT_KERNEL, 0)


def _nsm():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _spec(B_, V, r, gamma, stress=False, L=None):
    spec = dict(W.config("C4"), B=B_, V=V, r=r, gamma=gamma, temps=(0.7, 1.0),
                L=L or ("uniform", 0, gamma), name=f"slice-B{B_}-V{V}-r{r}")
    return W.stress(spec) if stress else spec


def _with_kernel(kernel, w):
    _lib.spec_set_option(_lib.SPEC_OPT_DRAFT_KERNEL, kernel)
    try:
        return gpu_cycle(w)
    finally:
        _lib.spec_set_option(_lib.SPEC_OPT_DRAFT_KERNEL, 0)


# chunks of 32 columns per CTA = ceil(ceil(V / 32) / SMs): V up to 256 x SMs
SHAPES = [
    (1, 16, 64, 1),            # one chunk, one request
    (40, 4104, 64, 5),         # 1 chunk per CTA, 8-column tail chunk
    (128, 9000, 128, 4),       # 2 chunks, ragged
    (96, 19456, 256, 3),       # 4 chunks (N = 128), U chunk 3 in the A tile's space
    (128, 32000, 256, 7),      # 7 chunks (C2's shape), N = 224
]


@pytest.mark.parametrize("B_,V,r,gamma", SHAPES)
def test_slice_kernel_matches_oracle_and_the_tile_strided_kernel(B_, V, r, gamma):
    spec = _spec(B_, V, r, gamma)
    w = W.make_workload(spec, trial=3)
    rows = None if B_ * gamma * V <= 40_000_000 else list(range(0, B_, 5))
    g = gpu_cycle(w)
    assert g.dstatus[0] & 8 == 0 and g.vstatus[0] & 8 == 0
    assert_parity(compare(w, g, oracle_cycle(w, rows=rows), rows=rows))
    g1 = _with_kernel(1, w)
    assert g1.dstatus[0] & 8 == 0
    same = [b for b in range(w.B) if np.array_equal(g.draft_tokens[b], g1.draft_tokens[b])]
    assert len(same) == w.B, f"kernels disagree on {w.B - len(same)} requests"
    np.testing.assert_allclose(g.q_tok, g1.q_tok, atol=1e-5, rtol=0)
    np.testing.assert_allclose(g.lse_q, g1.lse_q, atol=1e-5, rtol=0)


def test_slice_kernel_widest_slice():
    """Eight chunks per CTA (N = 256 accumulator columns): the largest
    vocabulary the slice-resident kernel takes on this GPU."""
    V = 256 * _nsm()
    spec = _spec(64, V, 256, 3)
    w = W.make_workload(spec, trial=1)
    rows = list(range(0, 64, 4))
    g = gpu_cycle(w)
    assert g.dstatus[0] & 8 == 0
    assert_parity(compare(w, g, oracle_cycle(w, rows=rows), rows=rows))


@pytest.mark.parametrize("trial", range(2))
def test_slice_kernel_stress_bias(trial):
    w = W.make_workload(_spec(128, 9000, 256, 5, stress=True), trial=trial)
    g = gpu_cycle(w)
    assert_parity(compare(w, g, oracle_cycle(w)))


def test_slice_kernel_adversarial_uniforms_and_redo():
    """Uniforms on the oracle's breakpoints: many draws queued over all steps
    and re-decided after the last one (and a re-decision that changes a token
    triggers the redo of the later steps)."""
    w = W.make_workload(_spec(48, 4104, 128, 6), trial=5)
    res = oracle_cycle(w)
    for b in range(w.B):
        for k in range(w.gamma):
            if (b + k) % 2 == 0:
                F = res.draft[b].F_hi[k] if b % 3 else res.draft[b].F_lo[k]
                w.u_draft[b, k] = np.float32(min(max(F, 1e-7), 1.0 - 6e-8))
    g = gpu_cycle(w)
    assert g.dstatus[1] > 0 and g.dstatus[0] & 8 == 0
    assert_parity(compare(w, g, oracle_cycle(w)))


@pytest.mark.parametrize("spec_fn", [lambda: W.config("C0"), lambda: _spec(128, 32000, 256, 7)],
                         ids=["tile-strided-fp32", "slice-resident"])
def test_stalled_barrier_times_out_and_the_context_survives(spec_fn):
    spec = spec_fn()
    w = W.make_workload(spec, trial=0)
    d = engine.DeviceWorkload.from_workload(w)
    b = engine.Buffers.for_workload(d)
    _lib.spec_set_option(_lib.SPEC_OPT_TEST_STALL, 1)
    try:
        t0 = time.time()
        engine.draft(d, b)
        torch.cuda.synchronize()
        el = time.time() - t0
    finally:
        _lib.spec_set_option(_lib.SPEC_OPT_TEST_STALL, 0)
    st = engine.status_words(b.dstatus)
    assert st[0] & 8, st                     # SPEC_DEV_TIMEOUT
    assert 0.5 < el < TIMEOUT, el
    # the same context runs the next call exactly
    g = gpu_cycle(w)
    assert g.dstatus[0] & 8 == 0 and g.vstatus[0] & 8 == 0
    rows = None if w.B <= 8 else list(range(0, w.B, 8))
    assert_parity(compare(w, g, oracle_cycle(w, rows=rows), rows=rows))


# ----------------------------------------------------------------- verification tiles

def _with_verify_kernel(kernel, w):
    _lib.spec_set_option(_lib.SPEC_OPT_VERIFY_KERNEL, kernel)
    try:
        return gpu_cycle(w)
    finally:
        _lib.spec_set_option(_lib.SPEC_OPT_VERIFY_KERNEL, 0)


@pytest.mark.parametrize("B_,V,r,gamma", SHAPES + [(200, 9000, 256, 7)])
def test_slice_verification_tiles_match_oracle_and_tile_strided(B_, V, r, gamma):
    """The slice-resident verification tiles (W2 columns resident per CTA,
    packed rows in tiles of 128 with two TMEM accumulators; 200 requests give
    up to 1400 packed rows, i.e. 11 row tiles) against the oracle and against
    the tile-strided verification tiles on the same draft."""
    w = W.make_workload(_spec(B_, V, r, gamma), trial=4)
    rows = None if B_ * gamma * V <= 40_000_000 else list(range(0, B_, 5))
    g = _with_verify_kernel(0, w)
    assert g.dstatus[0] & 8 == 0 and g.vstatus[0] & 8 == 0
    assert_parity(compare(w, g, oracle_cycle(w, rows=rows), rows=rows))
    g1 = _with_verify_kernel(1, w)
    np.testing.assert_array_equal(g.draft_tokens, g1.draft_tokens)
    np.testing.assert_array_equal(g.accept_len, g1.accept_len)
    np.testing.assert_array_equal(g.out_tokens, g1.out_tokens)
    np.testing.assert_allclose(g.alpha, g1.alpha, atol=1e-5, rtol=0, equal_nan=True)
    np.testing.assert_allclose(g.p_tok, g1.p_tok, atol=1e-5, rtol=0, equal_nan=True)


@pytest.mark.parametrize("kernel", [0, 1], ids=["cooperative-redecide", "work-unit-passes"])
def test_many_final_draws_redecided(kernel):
    """Every request's final draw (correction or bonus) placed on one of the
    oracle's own CDF breakpoints: 64 queued verification items, beyond the 16
    whose weights are kept, so the re-decision also recomputes weights column
    by column; both re-decision implementations must give the oracle's tokens."""
    w = W.make_workload(_spec(64, 9000, 256, 5), trial=6)
    res = oracle_cycle(w)
    for b in range(w.B):
        v = res.verify[b]
        F = v.final.F_hi if b % 2 else v.final.F_lo
        w.u_final[b] = np.float32(min(max(F, 1e-7), 1.0 - 6e-8))
    g = _with_verify_kernel(kernel, w)
    assert g.vstatus[1] >= 17, g.vstatus                 # more items than the kept ones
    assert g.vstatus[0] & 8 == 0
    assert_parity(compare(w, g, oracle_cycle(w)))
