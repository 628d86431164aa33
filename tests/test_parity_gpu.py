"""CUDA path (through the C ABI) against the float64 oracle, element by
element on the same seeded inputs.

Tokens and accept lengths must be bit-exact on every request, except that a
request with a consumed uniform within 1e-6 of a decision boundary may differ
-- and such requests must stay under 0.01% (with the sizes here that means
none).  q(x), logsumexp, alpha and p(x) agree within 1e-5 absolute."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from speculative_decoding_draft_04_gb300 import _lib, engine  # noqa: E402
from speculative_decoding_draft_04_gb300 import build as B  # noqa: E402
from speculative_decoding_draft_04_gb300 import workloads as W  # noqa: E402

from parity import assert_parity, compare, gpu_cycle, oracle_cycle  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    _lib.lib()
    _lib.spec_set_option(_lib.SPEC_OPT_FORCE_SIMT, 0)
    _lib.spec_set_option(_lib.SPEC_OPT_EPS_SCALE, 1.0)


def run_and_compare(w, rows=None, diag=False):
    g = gpu_cycle(w, diag=diag)
    res = oracle_cycle(w, rows=rows)
    rep = compare(w, g, res, rows=rows)
    return g, res, rep


# ----------------------------------------------------------------------------- small cases

def test_c0_fp32_many_trials():
    worst = None
    for trial in range(40):
        w = W.make_workload(W.config("C0"), trial=trial)
        g, res, rep = run_and_compare(w)
        assert_parity(rep)
        assert g.dstatus[0] & ~16 == 0 and g.vstatus[0] & ~16 == 0
        worst = rep
    print(worst.summary())


SMALL = dict(W.config("C4"), B=40, gamma=5, V=4104, r=64, name="small-ragged")


@pytest.mark.parametrize("trial", range(4))
def test_small_bf16_ragged(trial):
    """Several row tiles (BM=128 over 200 packed rows), 33 slices with an
    8-column tail slice, L in {0..5} including 0, T in {0.7, 1.0}."""
    w = W.make_workload(SMALL, trial=trial)
    g, res, rep = run_and_compare(w)
    assert_parity(rep)
    assert (w.verify_len == 0).any() or trial > 0


@pytest.mark.parametrize("trial", range(3))
def test_small_stress_bias(trial):
    """Markov factors with sd 0.3: the bias moves q by O(1), so a dropped or
    mis-indexed bias term would change most draws."""
    w = W.make_workload(W.stress(SMALL), trial=trial)
    g, res, rep = run_and_compare(w)
    assert_parity(rep)


def test_simt_bias_path_matches_oracle():
    _lib.spec_set_option(_lib.SPEC_OPT_FORCE_SIMT, 1)
    try:
        w = W.make_workload(W.config("C2", B=24, V=2048, r=128, name="simt"), trial=5)
        g, res, rep = run_and_compare(w)
        assert_parity(rep)
    finally:
        _lib.spec_set_option(_lib.SPEC_OPT_FORCE_SIMT, 0)


@pytest.mark.parametrize("B_,gamma,V,r", [(1, 1, 16, 16), (3, 16, 264, 32), (64, 2, 1024, 256),
                                         (33, 7, 8192, 16)])
def test_shape_edges(B_, gamma, V, r):
    spec = dict(W.config("C2"), B=B_, gamma=gamma, V=V, r=r, L=("uniform", 0, gamma),
                name="edge")
    w = W.make_workload(spec, trial=1)
    g, res, rep = run_and_compare(w)
    assert_parity(rep)


def test_verify_length_zero_everywhere():
    spec = dict(SMALL, L=("fixed", 0), name="L0")
    w = W.make_workload(spec, trial=2)
    g, res, rep = run_and_compare(w)
    assert_parity(rep)
    assert np.all(g.accept_len == 0)
    assert np.all(np.isnan(g.alpha))


def test_verify_with_oracle_draft():
    """The verify call alone, fed the oracle's draft tokens, q(x) and lse."""
    w = W.make_workload(SMALL, trial=7)
    res = oracle_cycle(w)
    d = engine.DeviceWorkload.from_workload(w)
    b = engine.Buffers.for_workload(d)
    toks = torch.tensor(np.stack([r.tokens for r in res.draft]), dtype=torch.int32, device="cuda")
    qt = torch.tensor(np.stack([r.q_tok for r in res.draft]), dtype=torch.float32, device="cuda")
    lq = torch.tensor(np.stack([r.lse_q for r in res.draft]), dtype=torch.float64, device="cuda")
    engine.verify(d, b, draft_tokens=toks, q_tok=qt, lse_q=lq)
    torch.cuda.synchronize()
    al = b.accept_len.cpu().numpy()
    ot = b.out_tokens.cpu().numpy()
    for i in range(w.B):
        assert al[i] == res.verify[i].accept_len
        assert np.array_equal(ot[i], res.verify[i].out_tokens)
        L = int(w.verify_len[i])
        np.testing.assert_allclose(b.alpha.cpu().numpy()[i, :L], res.verify[i].alpha[:L], atol=1e-5)


# ----------------------------------------------------------------------------- boundaries

def _near(x):
    """The float32 uniform nearest to a breakpoint (within ~3e-8 of it)."""
    return np.float32(min(max(x, 1e-7), 1.0 - 6e-8))


def test_adversarial_uniforms_force_redecision():
    """Uniforms placed on (the float32 nearest to) the oracle's own breakpoints:
    first draft draw, every ratio test with ratio < 1, and the final draw.
    The first pass cannot decide these; the extended-precision path must, and
    must agree with the oracle."""
    w = W.make_workload(dict(SMALL, B=24, name="adv"), trial=3)
    res = oracle_cycle(w)
    for b in range(w.B):
        d = res.draft[b]
        w.u_draft[b, 0] = _near(d.F_hi[0] if b % 2 else d.F_lo[0])
        v = res.verify[b]
        for j in range(int(w.verify_len[b])):
            if v.ratio[j] < 1.0 and b % 3 == 0:
                w.u_accept[b, j] = _near(v.ratio[j])
        w.u_final[b] = _near(v.final.F_hi if b % 2 else v.final.F_lo)
    g, res2, rep = run_and_compare(w)
    assert_parity(rep)
    assert g.dstatus[1] > 0, g.dstatus          # draft re-decisions happened
    assert g.vstatus[1] > 0, g.vstatus          # verify re-decisions happened


def test_adversarial_c0_fp32():
    w = W.make_workload(W.config("C0"), trial=11)
    res = oracle_cycle(w)
    for b in range(w.B):
        for k in range(w.gamma):
            if (b + k) % 2 == 0:
                w.u_draft[b, k] = _near(res.draft[b].F_hi[k])
    g, res2, rep = run_and_compare(w)
    assert_parity(rep)
    assert g.dstatus[1] > 0


# ----------------------------------------------------------------------------- full sizes

@pytest.mark.parametrize("name,sample", [("C1", None), ("C2", 24), ("C3", 3), ("C4", 5)])
def test_full_size_sampled(name, sample):
    """Full-size configurations in the launch configuration the bench times;
    the oracle checks a sample of requests one by one, and invariants that
    hold at any size are checked on every request."""
    w = W.make_workload(W.config(name), trial=0)
    rows = None
    if sample is not None:
        rng = np.random.default_rng(123)
        rows = sorted(rng.choice(w.B, size=sample, replace=False).tolist())
    g, res, rep = run_and_compare(w, rows=rows)
    print(name, rep.summary(), "draft status", g.dstatus, "verify status", g.vstatus)
    assert_parity(rep)
    # invariants on every request
    L = w.verify_len
    assert np.all((g.accept_len >= 0) & (g.accept_len <= L))
    for b in range(w.B):
        n = int(g.accept_len[b])
        assert np.array_equal(g.out_tokens[b, :n], g.draft_tokens[b, :n])
        assert 0 <= g.out_tokens[b, n] < w.V
        assert np.all(g.out_tokens[b, n + 1:] == -1)
    a = g.alpha[np.arange(w.gamma)[None, :] < L[:, None]]
    assert np.all((a >= 0) & (a <= 1 + 1e-5))
    assert np.all((g.q_tok > 0) & (g.q_tok <= 1))
    assert g.dstatus[0] & ~16 == 0 and g.vstatus[0] & ~16 == 0


# ----------------------------------------------------------------------------- errors

def test_invalid_requests_are_flagged_not_fatal():
    w = W.make_workload(dict(SMALL, B=8, name="bad"), trial=0)
    w.anchor[1] = w.V + 5            # bad anchor token
    w.verify_len[2] = w.gamma + 1    # bad verify length
    w.temperature[3] = 0.0           # bad temperature
    g = gpu_cycle(w)
    assert g.dstatus[0] & 1 and g.dstatus[0] & 4
    assert g.vstatus[0] & 1 and g.vstatus[0] & 2 and g.vstatus[0] & 4
    assert np.all(g.draft_tokens[1] == -1) and np.all(np.isnan(g.q_tok[3]))
    for b in (1, 2, 3):
        assert g.accept_len[b] == -1 and np.all(g.out_tokens[b] == -1)
    good = [0, 4, 5, 6, 7]
    res = oracle_cycle(w, rows=good)
    rep = compare(w, g, res, rows=good)
    assert_parity(rep)


def test_profile_api_counts_launches():
    w = W.make_workload(dict(SMALL, B=8, name="prof"), trial=0)
    d = engine.DeviceWorkload.from_workload(w)
    b = engine.Buffers.for_workload(d)
    _lib.spec_profile_enable(True)
    try:
        engine.cycle(d, b)
        torch.cuda.synchronize()
        prof = _lib.spec_profile_read()
    finally:
        _lib.spec_profile_enable(False)
    # the whole draft is one cooperative launch (of one of the two draft kernels)
    assert prof["draft_persistent"][1] + prof["draft_slice"][1] == 1
    assert prof["verify_tile"][1] + prof["verify_slice"][1] == 1
    assert all(ms >= 0 for ms, _ in prof.values())


# ----------------------------------------------------------------------------- tcgen05 path

@pytest.fixture()
def tc_path():
    _lib.spec_set_option(_lib.SPEC_OPT_BIAS_PATH, 2)
    yield
    _lib.spec_set_option(_lib.SPEC_OPT_BIAS_PATH, 2)


@pytest.fixture()
def warp_mma_path():
    _lib.spec_set_option(_lib.SPEC_OPT_BIAS_PATH, 1)
    yield
    _lib.spec_set_option(_lib.SPEC_OPT_BIAS_PATH, 2)


@pytest.mark.parametrize("trial", range(2))
def test_warp_mma_bias_path_parity(warp_mma_path, trial):
    """The legacy warp-MMA bias path stays selectable and exact."""
    w = W.make_workload(dict(SMALL, r=256, name="wmma"), trial=trial)
    g, res, rep = run_and_compare(w)
    assert_parity(rep)


@pytest.mark.parametrize("B_,V,r,gamma", [(8, 1024, 64, 3), (130, 4104, 128, 4), (40, 4104, 256, 5),
                                         (3, 264, 256, 2)])
def test_tcgen05_bias_path_parity(tc_path, B_, V, r, gamma):
    """Tensor-memory bias tiles (one or two 128-row tiles, ragged tails)."""
    spec = dict(SMALL, B=B_, V=V, r=r, gamma=gamma, L=("uniform", 0, gamma), name="tc")
    w = W.make_workload(spec, trial=4)
    g, res, rep = run_and_compare(w)
    assert g.dstatus[0] & 8 == 0 and g.vstatus[0] & 8 == 0, "bounded wait expired"
    assert_parity(rep)
    w2 = W.make_workload(W.stress(spec), trial=4)
    g2, res2, rep2 = run_and_compare(w2)
    assert_parity(rep2)


@pytest.mark.parametrize("name,sample", [("C2", 24), ("C4", 5)])
def test_tcgen05_full_size(tc_path, name, sample):
    w = W.make_workload(W.config(name), trial=1)
    rng = np.random.default_rng(7)
    rows = sorted(rng.choice(w.B, size=sample, replace=False).tolist())
    g, res, rep = run_and_compare(w, rows=rows)
    print(name, "tcgen05", rep.summary(), g.dstatus, g.vstatus)
    assert g.dstatus[0] & 8 == 0 and g.vstatus[0] & 8 == 0
    assert_parity(rep)


# ----------------------------------------------------------------------------- persistent draft

@pytest.mark.parametrize("spec_name", ["C0", "small"])
def test_draft_near_boundary_at_step_one(spec_name):
    """Every request's second draw sits just past a CDF breakpoint (the draw
    after the first token, so the step reads tokens written by the previous
    step of the same launch)."""
    spec = {"C0": W.config("C0"), "small": dict(SMALL, B=24)}[spec_name]
    w = W.make_workload(spec, trial=6)
    res = oracle_cycle(w)
    for b in range(w.B):
        w.u_draft[b, 1] = _near(res.draft[b].F_hi[1])
    g, res, rep = run_and_compare(w)
    assert g.dstatus[0] & 8 == 0
    assert_parity(rep)


@pytest.mark.parametrize("spec_name", ["C0", "small", "stress", "tc-two-tiles"])
def test_persistent_draft_parity(spec_name):
    """The whole draft as one cooperative launch (grid barriers between the
    tile, sampling and re-decision phases of every step)."""
    spec = {"C0": W.config("C0"), "small": SMALL, "stress": W.stress(SMALL),
            "tc-two-tiles": dict(SMALL, B=130, r=256, gamma=4, L=("uniform", 0, 4))}[spec_name]
    for trial in range(3):
        w = W.make_workload(spec, trial=trial)
        g, res, rep = run_and_compare(w)
        assert g.dstatus[0] & 8 == 0, "grid barrier or MMA wait timed out"
        assert_parity(rep)


def test_persistent_adversarial():
    w = W.make_workload(dict(SMALL, B=24, name="adv-p"), trial=5)
    res = oracle_cycle(w)
    for b in range(w.B):
        for k in range(w.gamma):
            if (b + k) % 3 == 0:
                w.u_draft[b, k] = _near(res.draft[b].F_hi[k] if b % 2 else res.draft[b].F_lo[k])
    g, res2, rep = run_and_compare(w)
    assert_parity(rep)
    assert g.dstatus[1] > 0 and g.dstatus[0] & 8 == 0


@pytest.mark.parametrize("name,sample", [("C1", None), ("C2", 24), ("C3", 3), ("C4", 5)])
def test_persistent_full_size(name, sample):
    w = W.make_workload(W.config(name), trial=2)
    rows = None
    if sample is not None:
        rows = sorted(np.random.default_rng(9).choice(w.B, size=sample, replace=False).tolist())
    g, res, rep = run_and_compare(w, rows=rows)
    print(name, "persistent", rep.summary(), g.dstatus)
    assert g.dstatus[0] & 8 == 0
    assert_parity(rep)
