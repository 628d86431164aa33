"""The library's operating-point report (spec_operating_point, host code) and
its measured acceptance statistics (spec_acceptance_stats, a device
reduction) against the float64 oracle (oracle/speedup_model.py)."""
import ctypes
import math

import numpy as np
import pytest

from oracle import speedup_model as M
from speculative_decoding_draft_04_gb300 import _lib
from speculative_decoding_draft_04_gb300 import build as B


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    B.build()
    _lib.lib()


ALPHAS = [0.0, 0.05, 0.3, 0.5, 0.8, 0.9, 0.95, 0.99, 0.999]
CS = [0.001, 0.02, 0.05, 0.2, 0.7, 1.5]


@pytest.mark.parametrize("alpha", ALPHAS)
@pytest.mark.parametrize("c", CS)
def test_operating_point_matches_oracle(alpha, c):
    for gamma in (1, 3, 7, 21):
        r = _lib.spec_operating_point(alpha, c, gamma, 300, c_hat=0.01)
        assert r["expected_tau"] == pytest.approx(M.expected_tau(alpha, gamma), rel=1e-13)
        assert r["speedup"] == pytest.approx(M.speedup(alpha, c, gamma), rel=1e-13)
        assert r["speedup_gamma1"] == pytest.approx(M.speedup(alpha, c, 1), rel=1e-13)
        assert r["bound"] == pytest.approx(M.speedup_bound(alpha, c), rel=1e-13)
        assert r["compute_ratio"] == pytest.approx(M.compute_ratio(alpha, 0.01, gamma), rel=1e-13)
        assert r["gains"] == int(M.speedup(alpha, c, gamma) > 1)
    g, s = M.optimal_gamma(alpha, c, 300)
    assert r["gamma_star"] == g
    assert r["speedup_star"] == pytest.approx(s, rel=1e-13)
    if 0 < alpha < 1:
        assert r["gamma_continuous"] == pytest.approx(M.continuous_optimum(alpha, c), rel=1e-9, abs=1e-9)


def test_operating_point_alpha_one():
    r = _lib.spec_operating_point(1.0, 0.05, 7, 50)
    assert r["expected_tau"] == 8.0
    assert r["bound"] == pytest.approx(20.0)
    assert math.isinf(r["gamma_continuous"])
    assert r["gamma_star"] == 50                       # S grows in gamma when alpha = 1, c < 1


def test_operating_point_rejects_bad_arguments():
    L = _lib.lib()
    out = _lib.OpResult()
    for args in ((1.5, 0.1, 0.0, 3, 10), (-0.1, 0.1, 0.0, 3, 10), (0.5, 0.0, 0.0, 3, 10),
                 (0.5, 0.1, -1.0, 3, 10), (0.5, 0.1, 0.0, 0, 10), (0.5, 0.1, 0.0, 5, 4),
                 (float("nan"), 0.1, 0.0, 3, 10), (0.5, 0.1, 0.0, 3, 200000)):
        assert L.spec_operating_point(ctypes.byref(_lib.OpArgs(*args)), ctypes.byref(out)) == -1
    assert L.spec_operating_point(None, ctypes.byref(out)) == -1
    assert L.spec_operating_point(ctypes.byref(_lib.OpArgs(0.5, 0.1, 0.0, 3, 10)), None) == -1


@pytest.mark.gpu
def test_acceptance_stats_match_oracle():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rng = np.random.default_rng(5)
    for Bn, gamma in ((1, 1), (37, 7), (600, 16)):
        L = rng.integers(0, gamma + 1, Bn).astype(np.int32)
        acc = np.array([rng.integers(0, l + 1) for l in L], np.int32)
        acc[rng.random(Bn) < 0.1] = -1                   # invalid requests are skipped
        alpha = rng.random((Bn, gamma)).astype(np.float32)
        alpha[np.arange(gamma)[None, :] >= L[:, None]] = np.nan
        valid = acc >= 0
        d = [torch.from_numpy(x).cuda() for x in (alpha, L, acc)]
        out = torch.zeros(4, dtype=torch.float64, device="cuda")
        _lib.spec_acceptance_stats(d[0], d[1], d[2], out)
        o = out.cpu().numpy()
        ref_a = M.measured_alpha(alpha[valid].astype(np.float64), L[valid])
        n_pos = int(L[valid].sum())
        assert o[1] == n_pos and o[3] == int(valid.sum())
        if n_pos:
            assert o[0] / o[1] == pytest.approx(ref_a, rel=1e-12)
        assert o[2] / o[3] == pytest.approx(M.measured_tau(acc), rel=1e-12)
