"""GPU parity of the RNN head (spec_rnn_draft, then spec_verify with its factor
rows) against the float64 oracle (oracle/rnn_head.py): factor rows a_j bit-exact
(each the correctly rounded float64 value), tokens and accept lengths
bit-exact except near a boundary (the Markov head's bar), probabilities and
alpha within 1e-5."""
import dataclasses

import numpy as np
import pytest

from oracle import rnn_head as H
from oracle import spec_oracle as O
from speculative_decoding_draft_04_gb300 import workloads as W

from parity import GpuResult, LazyRows, assert_parity, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_draft_04_gb300 import build as B
    B.build()
    return t


def run_gpu(torch, w, ri):
    from speculative_decoding_draft_04_gb300 import engine
    d = engine.DeviceWorkload.from_workload(w)
    b = engine.Buffers.for_workload(d)
    h = engine.DeviceRnn.from_inputs(ri, d)
    engine.rnn_cycle(d, b, h)
    torch.cuda.synchronize()
    g = GpuResult(b.draft_tokens.cpu().numpy(), b.q_tok.cpu().numpy(), b.lse_q.cpu().numpy(),
                  b.accept_len.cpu().numpy(), b.out_tokens.cpu().numpy(), b.alpha.cpu().numpy(),
                  b.p_tok.cpu().numpy(), engine.status_words(b.dstatus),
                  engine.status_words(b.vstatus))
    a = h.a_rows.float().cpu().numpy().astype(np.float64)          # [gamma, B, r]
    return g, np.transpose(a, (1, 0, 2))


def run_oracle(w, ri):
    tgt, U = LazyRows(w.target, w.dtype), LazyRows(w.U, w.dtype)
    W1, W2, Wr = w.f64("W1"), w.f64("W2"), W.to_f64(ri.Wr, w.dtype)
    ds, vs, arows = [], [], []
    for b in range(w.B):
        d, v, a = H.rnn_cycle_request(tgt[b], U[b], W1, W2, Wr, ri.hproj[b].astype(np.float64),
                                      w.anchor[b], float(w.temperature[b]),
                                      w.u_draft[b].astype(np.float64), w.verify_len[b],
                                      w.u_accept[b].astype(np.float64), float(w.u_final[b]),
                                      w.dtype)
        ds.append(d)
        vs.append(v)
        arows.append(a)
    return O.CycleResult(ds, vs), np.stack(arows)


def check_factor_rows(g, res, a_gpu, a_ref):
    """a_j depends on x_j: compare each request up to its first token that
    differs from the oracle's."""
    for b in range(a_ref.shape[0]):
        same = np.flatnonzero(g.draft_tokens[b] != res.draft[b].tokens)
        upto = (same[0] + 1) if same.size else a_ref.shape[1]
        assert np.array_equal(a_gpu[b, :upto], a_ref[b, :upto]), b


@pytest.mark.parametrize("name,B,stress", [("C0", None, False), ("C0", None, True),
                                           ("C1", 12, False), ("C2", 24, False),
                                           ("C2", 16, True), ("C3", 4, False), ("C4", 6, False)])
def test_rnn_cycle_parity(torch, name, B, stress):
    spec = W.config(name)
    if stress:
        spec = W.stress(spec, w_sd=0.3 if name == "C0" else 0.1)
    w = W.make_workload(spec, 0, B=B)
    ri = W.make_rnn_inputs(spec, 0, B=B)
    g, a_gpu = run_gpu(torch, w, ri)
    assert (g.dstatus[0] & ~16) == 0 and (g.vstatus[0] & ~16) == 0, (g.dstatus, g.vstatus)
    res, a_ref = run_oracle(w, ri)
    check_factor_rows(g, res, a_gpu, a_ref)
    assert_parity(compare(w, g, res))


def test_rnn_reduces_to_the_markov_draft(torch):
    """W_o = [0 | kappa I] and h_o = 0: the RNN draft's factor rows are
    round(tanh(kappa W1[x_j])), so it must draw exactly what the Markov draft
    draws with W1' = round(tanh(kappa W1)) (both on the GPU)."""
    from speculative_decoding_draft_04_gb300 import engine
    spec = W.config("C2")
    w = W.make_workload(spec, 1, B=40)
    r, kappa = w.r, 20.0
    ri = W.make_rnn_inputs(spec, 1, B=40)
    Wr = W.to_f64(ri.Wr, "bf16")
    Wr[2 * r:, :] = 0.0
    Wr[2 * r:, r:] = kappa * np.eye(r)
    ri = dataclasses.replace(ri, Wr=W.bf16_round(Wr))
    ri.hproj[:, :, 2, :] = 0.0
    g, a_gpu = run_gpu(torch, w, ri)
    W1m = W.bf16_round(np.tanh(kappa * w.f64("W1")))
    wm = dataclasses.replace(w, W1=W1m)
    d = engine.DeviceWorkload.from_workload(wm)
    b = engine.Buffers.for_workload(d)
    engine.draft(d, b)
    torch.cuda.synchronize()
    assert np.array_equal(b.draft_tokens.cpu().numpy(), g.draft_tokens)
    assert np.array_equal(b.q_tok.cpu().numpy(), g.q_tok)
    prevs = np.concatenate([w.anchor[:, None], g.draft_tokens[:, :-1]], axis=1)
    assert np.array_equal(a_gpu, W.bf16_to_f64(W1m)[prevs])


def test_rnn_full_size_sampled(torch):
    """C2 at full batch through the same launch configuration, checked on a
    sample of requests against the oracle."""
    spec = W.config("C2")
    w = W.make_workload(spec, 2)
    ri = W.make_rnn_inputs(spec, 2)
    g, a_gpu = run_gpu(torch, w, ri)
    rows = list(range(0, w.B, 16))
    sub = w.subset(rows)
    subri = dataclasses.replace(ri, hproj=ri.hproj[rows])
    res, a_ref = run_oracle(sub, subri)
    gs = GpuResult(*(getattr(g, f.name)[rows] if isinstance(getattr(g, f.name), np.ndarray) and
                     getattr(g, f.name).shape[:1] == (w.B,) else getattr(g, f.name)
                     for f in dataclasses.fields(GpuResult)))
    check_factor_rows(gs, res, a_gpu[rows], a_ref)
    assert_parity(compare(sub, gs, res))
