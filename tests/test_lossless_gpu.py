"""Losslessness of the CUDA path, by chi-square at a tiny vocabulary.

The SpecDec blog ("수락 규칙", the losslessness theorem) states that the
tokens the speculative cycle emits follow the target distribution whatever
the draft distribution is.  With target rows that do not depend on the
prefix (as in these synthetic inputs), the token emitted at position j of a
cycle, given that the cycle reached position j, follows p_j = softmax(t_j/T).
This runs that check on the GPU path itself, through the C ABI: one small
problem (V = 16) replicated over 4096 requests per launch, each request with
fresh uniforms, so every launch is 4096 independent cycles.

For each reached position the emitted tokens are compared with p_j by a
chi-square test (p-value > 1e-3); the first draft token is compared the same
way with q_1 = softmax((U_0 + W1[x_0] W2)/T) (the DSpark review, section 1.2,
Markov head); and the acceptance rate of position 0 is checked against
alpha_0 = sum_v min(p_0, q_1) (the blog's closed form) within 4 sigma.
Reference distributions come from scipy, not from the oracle.
"""
import numpy as np
import pytest
from scipy import special, stats

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from speculative_decoding_draft_04_gb300 import _lib, engine  # noqa: E402
from speculative_decoding_draft_04_gb300 import build as B  # noqa: E402
from speculative_decoding_draft_04_gb300 import workloads as W  # noqa: E402

NREQ = 4096
LAUNCHES = 24


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    _lib.lib()
    _lib.spec_set_option(_lib.SPEC_OPT_FORCE_SIMT, 0)
    _lib.spec_set_option(_lib.SPEC_OPT_EPS_SCALE, 1.0)
    _lib.spec_set_option(_lib.SPEC_OPT_BIAS_PATH, 2)


def _problem(gamma, with_bias, dtype, seed):
    rng = np.random.default_rng([901, gamma, int(with_bias), seed])
    V, r, T = 16, 16, 0.8
    t = rng.normal(0, 1.0, (gamma + 1, V))
    U = t[:gamma] + rng.normal(0, 1.3, (gamma, V))
    sd = 0.5 if with_bias else 0.0
    W1 = rng.normal(0, sd, (V, r))
    W2 = rng.normal(0, sd, (r, V))
    anchor = int(rng.integers(0, V))
    st = W._store
    return dict(V=V, r=r, T=T, anchor=anchor, t=st(t, dtype), U=st(U, dtype), W1=st(W1, dtype),
                W2=st(W2, dtype))


def _workload(pb, gamma, dtype, rng):
    V = pb["V"]
    tile = lambda a: np.ascontiguousarray(np.broadcast_to(a, (NREQ,) + a.shape))  # noqa: E731
    spec = dict(name="lossless", B=NREQ, gamma=gamma, V=V, r=pb["r"], dtype=dtype)
    return W.Workload(
        spec=spec, trial=0, dtype=dtype, B=NREQ, gamma=gamma, V=V, r=pb["r"],
        target=tile(pb["t"]), U=tile(pb["U"]), W1=pb["W1"], W2=pb["W2"],
        anchor=np.full(NREQ, pb["anchor"], np.int32),
        temperature=np.full(NREQ, pb["T"], np.float32),
        verify_len=np.full(NREQ, gamma, np.int32),
        u_draft=W.uniforms(rng, (NREQ, gamma)), u_accept=W.uniforms(rng, (NREQ, gamma)),
        u_final=W.uniforms(rng, (NREQ,)))


@pytest.mark.parametrize("gamma,with_bias,dtype", [(1, False, "f32"), (1, True, "bf16"),
                                                   (3, False, "bf16"), (3, True, "f32")])
def test_emitted_tokens_follow_the_target(gamma, with_bias, dtype):
    pb = _problem(gamma, with_bias, dtype, 0)
    f64 = lambda a: W.to_f64(a, dtype)  # noqa: E731
    t, U, W1, W2 = f64(pb["t"]), f64(pb["U"]), f64(pb["W1"]), f64(pb["W2"])
    T = float(np.float32(pb["T"]))
    p = [special.softmax(t[j] / T) for j in range(gamma + 1)]
    q1 = special.softmax((U[0] + W1[pb["anchor"]] @ W2) / T)
    V = pb["V"]
    rng = np.random.default_rng([902, gamma, int(with_bias)])
    emitted = [np.zeros(V) for _ in range(gamma + 1)]
    first_draft = np.zeros(V)
    accepted0 = tested0 = 0
    bufs = None
    for _ in range(LAUNCHES):
        w = _workload(pb, gamma, dtype, rng)
        d = engine.DeviceWorkload.from_workload(w)
        if bufs is None:
            bufs = engine.Buffers.for_workload(d)
        engine.cycle(d, bufs)
        torch.cuda.synchronize()
        dst, vst = engine.status_words(bufs.dstatus), engine.status_words(bufs.vstatus)
        assert dst[0] & ~16 == 0 and vst[0] & ~16 == 0, (dst, vst)
        acc = bufs.accept_len.cpu().numpy()
        out = bufs.out_tokens.cpu().numpy()
        dt = bufs.draft_tokens.cpu().numpy()
        assert ((acc >= 0) & (acc <= gamma)).all()
        first_draft += np.bincount(dt[:, 0], minlength=V)
        for j in range(gamma + 1):
            sel = acc >= j
            emitted[j] += np.bincount(out[sel, j], minlength=V)
            assert (out[acc < j, j] == -1).all() if j > 0 else True
        tested0 += NREQ
        accepted0 += int((acc >= 1).sum())
    n_cycles = LAUNCHES * NREQ
    pv = stats.chisquare(first_draft, q1 * first_draft.sum()).pvalue
    assert pv > 1e-3, ("first draft token vs q_1", pv)
    for j in range(gamma + 1):
        obs = emitted[j]
        if obs.sum() < 2000:
            continue
        pv = stats.chisquare(obs, p[j] * obs.sum()).pvalue
        assert pv > 1e-3, (j, obs.sum(), pv)
    alpha0 = float(np.minimum(p[0], q1).sum())
    rate = accepted0 / tested0
    sigma = np.sqrt(alpha0 * (1 - alpha0) / n_cycles)
    assert abs(rate - alpha0) < 4 * sigma + 1e-12, (rate, alpha0, sigma)
