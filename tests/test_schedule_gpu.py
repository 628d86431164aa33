"""GPU parity of the confidence head (spec_confidence) and the hardware-aware
prefix scheduler (spec_prefix_schedule) against the float64 oracle
(oracle/scheduler.py), and of the confidence-scheduled cycle (draft ->
confidence -> schedule -> verify with the scheduled lengths) against the
oracle's cycle at those lengths.

Bars: confidences bit-equal to the float64 value rounded to fp32, except
within 1e-12 (relative) of a rounding midpoint, where one ulp is allowed;
survival values, verify lengths, B, tau and Theta bit-exact given the
kernel's confidences (the oracle takes the scheduler's decisions in the
kernel's precision: fp32 survival, tau in 2^-36 units, float64 Theta)."""
import dataclasses
import json
import os

import numpy as np
import pytest

from oracle import scheduler as S
from speculative_decoding_draft_04_gb300 import workloads as W

from parity import assert_parity, compare, oracle_cycle

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
UNIT = 2.0 ** -S.TAU_UNIT_BITS
BAD_TOKEN, BAD_CONF = 1, 64


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_draft_04_gb300 import build as B
    B.build()
    return t


def _lib():
    from speculative_decoding_draft_04_gb300 import _lib as L
    return L


# ------------------------------------------------------------------ helpers

def run_confidence(torch, hidden, W1, w, anchor, tokens, dtype):
    from speculative_decoding_draft_04_gb300.engine import _dev_logits
    R, g, _ = hidden.shape
    dev = "cuda"
    conf = torch.empty((R, g), dtype=torch.float32, device=dev)
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    _lib().spec_confidence(_dev_logits(hidden, dtype, dev), _dev_logits(W1, dtype, dev),
                           torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(dev),
                           torch.from_numpy(np.ascontiguousarray(anchor, np.int32)).to(dev),
                           torch.from_numpy(np.ascontiguousarray(tokens, np.int32)).to(dev),
                           conf, st)
    torch.cuda.synchronize()
    return conf.cpu().numpy(), int(st[0].item())


def run_schedule(torch, conf, sps):
    R, g = conf.shape
    dev = "cuda"
    c = torch.from_numpy(np.ascontiguousarray(conf, np.float32)).to(dev)
    s = torch.from_numpy(np.ascontiguousarray(sps, np.float64)).to(dev)
    surv = torch.empty((R, g), dtype=torch.float32, device=dev)
    ell = torch.full((R,), -7, dtype=torch.int32, device=dev)
    tot = torch.empty(4, dtype=torch.int64, device=dev)
    th = torch.empty(1, dtype=torch.float64, device=dev)
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    ws = torch.empty(_lib().spec_schedule_workspace_bytes(R, g), dtype=torch.uint8, device=dev)
    _lib().spec_prefix_schedule(c, s, surv, ell, tot, th, st, ws)
    torch.cuda.synchronize()
    return (surv.cpu().numpy(), ell.cpu().numpy(), tot.cpu().numpy(), float(th.item()),
            int(st[0].item()))


def conf_far_mismatches(got32, ref64):
    """Entries where the kernel's fp32 confidence is not the rounded float64
    value and the float64 value is not within 1e-12 of a rounding midpoint."""
    ref32 = ref64.astype(np.float32)
    bad = np.flatnonzero(got32.ravel() != ref32.ravel())
    far = []
    for i in bad:
        g, r, x = np.float32(got32.flat[i]), ref32.flat[i], float(ref64.flat[i])
        adjacent = np.nextafter(r, g) == g
        mid = (float(g) + float(r)) / 2
        if not (adjacent and abs(x - mid) <= 1e-12 * abs(x)):
            far.append(int(i))
    return bad, far


def check_schedule(conf32, sps, got):
    surv, ell, tot, th, st = got
    a = S.survival(conf32)
    assert np.array_equal(surv.view(np.uint32), a.view(np.uint32))
    ell_o, B_o, tau_o, th_o = S.schedule(a, sps)
    assert np.array_equal(ell, ell_o), (np.flatnonzero(ell != ell_o)[:10], tot)
    assert tot[0] == B_o and tot[1] == tau_o and tot[2] == ell_o.sum()
    assert th == th_o
    return ell_o


# ------------------------------------------------------------------ confidence

@pytest.mark.parametrize("name", ["C0", "C1", "C2", "C3", "C4"])
def test_confidence_parity(torch, name):
    spec = W.config(name)
    w = W.make_workload(spec, 0)
    si = W.make_schedule_inputs(spec, 0)
    rng = np.random.default_rng(11)
    tokens = rng.integers(0, w.V, size=(w.B, w.gamma)).astype(np.int32)
    got, st = run_confidence(torch, si.hidden, w.W1, si.w, w.anchor, tokens, w.dtype)
    assert st == 0
    ref = S.confidences(W.to_f64(si.hidden, w.dtype), w.f64("W1"), si.w.astype(np.float64),
                        w.anchor, tokens)
    bad, far = conf_far_mismatches(got, ref)
    assert not far, (name, far[:5])
    assert len(bad) <= max(1, 1e-4 * got.size)
    assert np.max(np.abs(got - ref)) < 1e-6


@pytest.mark.parametrize("d,r,dtype", [(8, 16, "f32"), (264, 16, "bf16"), (4104, 256, "bf16"),
                                       (520, 64, "f32")])
def test_confidence_ragged_widths_and_extremes(torch, d, r, dtype):
    """Widths that leave lanes partly idle, and logits far in both tails
    (c = 0 and c = 1 in fp32)."""
    rng = np.random.default_rng(d + r)
    R, g, V = 37, 5, 3000
    hid = rng.normal(0, 1, size=(R, g, d))
    hid[:, :, 0] = rng.choice([-120.0, -30.0, 0.0, 30.0, 120.0], size=(R, g))
    st_ = (lambda x: W.bf16_round(x)) if dtype == "bf16" else (lambda x: x.astype(np.float32))
    hidden, W1 = st_(hid), st_(rng.normal(0, 0.05, size=(V, r)))
    w = np.concatenate([[1.0], rng.normal(0, 1 / np.sqrt(d), d - 1), rng.normal(0, 1.0, r)])
    w = w.astype(np.float32)
    anchor = rng.integers(0, V, R).astype(np.int32)
    tokens = rng.integers(0, V, (R, g)).astype(np.int32)
    got, st = run_confidence(torch, hidden, W1, w, anchor, tokens, dtype)
    assert st == 0
    ref = S.confidences(W.to_f64(hidden, dtype), W.to_f64(W1, dtype), w.astype(np.float64), anchor,
                        tokens)
    _, far = conf_far_mismatches(got, ref)
    assert not far
    assert np.any(got == 1.0) and np.any(got == 0.0)


def test_confidence_bad_token(torch):
    rng = np.random.default_rng(3)
    R, g, d, V, r = 4, 3, 64, 100, 16
    hidden = rng.normal(size=(R, g, d)).astype(np.float32)
    W1 = rng.normal(size=(V, r)).astype(np.float32)
    w = rng.normal(size=d + r).astype(np.float32) * 0.1
    anchor = np.array([1, 2, 3, 4], np.int32)
    tokens = rng.integers(0, V, (R, g)).astype(np.int32)
    tokens[2, 0] = V                                   # read by row 1 of request 2
    got, st = run_confidence(torch, hidden, W1, w, anchor, tokens, "f32")
    assert st & BAD_TOKEN
    assert np.isnan(got[2, 1]) and np.isfinite(np.delete(got.ravel(), 2 * g + 1)).all()


# ------------------------------------------------------------------ scheduler

def test_schedule_golden_cases(torch):
    cases = json.load(open(os.path.join(HERE, "golden", "schedule_worked.json")))["cases"]
    for case in cases:
        conf = np.asarray(case["conf"], np.float32)
        sps = np.asarray(case["sps"], np.float64)
        got = run_schedule(torch, conf, sps)
        check_schedule(conf, sps, got)
        assert list(got[1]) == case["ell"] and got[2][0] == case["B"]
        assert got[2][1] * UNIT == pytest.approx(case["tau"], abs=1e-6)


@pytest.mark.parametrize("R,g", [(1, 1), (1, 16), (3, 4), (32, 7), (128, 7), (64, 15), (256, 7),
                                 (1000, 5), (4096, 16)])
def test_schedule_parity_random(torch, R, g):
    rng = np.random.default_rng(R * 31 + g)
    for trial in range(3):
        conf = rng.beta(4, 1.5, size=(R, g)).astype(np.float32)
        knee = R * (1 + g * rng.uniform(0.1, 0.9))
        sps = W.cost_table(R, g) if trial == 0 else 1000.0 / np.sqrt(
            42.0 ** 2 + (np.arange(R * (1 + g) + 1) * 42.0 / knee) ** 2)
        ell = check_schedule(conf, sps, run_schedule(torch, conf, sps))
        if R * g >= 100:
            assert 0 < ell.sum() < R * g           # the curve stops the search inside the pool


def test_schedule_ties_and_exact_values(torch):
    R, g = 50, 6
    conf = np.full((R, g), 0.5, np.float32)
    conf[::7, 2] = 1.0                              # a survival plateau inside a row
    conf[::11, 0] = 0.0
    for m in (0, 1, 49, 50, 51, 137, R * g):
        sps = np.ones(R + m + 1)                    # the table ends after m admissions
        got = run_schedule(torch, conf, sps)
        ell = check_schedule(conf, sps, got)
        assert ell.sum() == min(m, R * g)
        assert got[2][3] == (2 if m < R * g else 0)


def test_schedule_decrease_stop_reason(torch):
    R, g = 20, 4
    conf = np.full((R, g), 0.9, np.float32)
    sps = 1.0 / np.arange(1, R * (1 + g) + 2, dtype=np.float64)   # SPS = 1/B: any a < 1 loses
    sps = np.concatenate([[1.0], sps])[: R * (1 + g) + 1]
    got = run_schedule(torch, conf, sps)
    check_schedule(conf, sps, got)
    assert got[1].sum() == 0 and got[2][3] == 1


def test_schedule_bad_confidences_count_as_zero(torch):
    rng = np.random.default_rng(9)
    R, g = 40, 7
    conf = rng.random((R, g)).astype(np.float32)
    conf[3, 2], conf[7, 0], conf[11, 5] = np.nan, -0.25, 1.5
    sps = W.cost_table(R, g)
    got = run_schedule(torch, conf, sps)
    assert got[4] & BAD_CONF
    clean = np.where((conf >= 0) & (conf <= 1), conf, 0).astype(np.float32)
    check_schedule(clean, sps, got)
    assert got[1][7] == 0


# ------------------------------------------------------------ scheduled cycle

@pytest.mark.parametrize("name,B", [("C0", None), ("C2", 48), ("C4", 40)])
def test_scheduled_cycle_parity(torch, name, B):
    from speculative_decoding_draft_04_gb300 import engine
    spec = W.config(name)
    w = W.make_workload(spec, 0, B=B)
    si = W.make_schedule_inputs(spec, 0, B=B)
    d = engine.DeviceWorkload.from_workload(w)
    b = engine.Buffers.for_workload(d)
    s = engine.DeviceSchedule.from_inputs(si, w.B, w.gamma, w.dtype)
    engine.scheduled_cycle(d, b, s)
    torch.cuda.synchronize()
    assert engine.status_words(s.status)[0] == 0
    tokens = b.draft_tokens.cpu().numpy()
    conf = s.conf.cpu().numpy()
    ref = S.confidences(W.to_f64(si.hidden, w.dtype), w.f64("W1"), si.w.astype(np.float64),
                        w.anchor, tokens)
    _, far = conf_far_mismatches(conf, ref)
    assert not far
    got = (s.survival.cpu().numpy(), s.verify_len.cpu().numpy(), s.totals.cpu().numpy(),
           float(s.theta.item()), 0)
    ell = check_schedule(conf, si.sps, got)
    w2 = dataclasses.replace(w, verify_len=ell.astype(np.int32))
    from parity import GpuResult
    g = GpuResult(tokens, b.q_tok.cpu().numpy(), b.lse_q.cpu().numpy(), b.accept_len.cpu().numpy(),
                  b.out_tokens.cpu().numpy(), b.alpha.cpu().numpy(), b.p_tok.cpu().numpy(),
                  engine.status_words(b.dstatus), engine.status_words(b.vstatus))
    assert_parity(compare(w2, g, oracle_cycle(w2)))


@pytest.mark.parametrize("name,B", [("C0", None), ("C1", None), ("C2", None), ("C3", 32), ("C4", 96)])
def test_schedule_from_the_oracles_own_confidences(torch, name, B):
    """The whole schedule derived from the ORACLE's confidences (float64 value
    rounded once to fp32), not from the kernel's: verify lengths, B, tau and
    Theta must equal the kernel's.  Where a kernel confidence differs from the
    oracle's by one ulp (within 1e-12 of a rounding midpoint), the two
    schedules are both computed and any change of l, B or Theta is reported."""
    from speculative_decoding_draft_04_gb300 import engine
    spec = W.config(name)
    w = W.make_workload(spec, 0, B=B)
    si = W.make_schedule_inputs(spec, 0, B=B)
    d = engine.DeviceWorkload.from_workload(w)
    b = engine.Buffers.for_workload(d)
    s = engine.DeviceSchedule.from_inputs(si, w.B, w.gamma, w.dtype)
    engine.scheduled_cycle(d, b, s)
    torch.cuda.synchronize()
    tokens = b.draft_tokens.cpu().numpy()
    conf = s.conf.cpu().numpy()
    ell_k, tot_k = s.verify_len.cpu().numpy(), s.totals.cpu().numpy()
    theta_k = float(s.theta.item())
    ref = S.confidences(W.to_f64(si.hidden, w.dtype), w.f64("W1"), si.w.astype(np.float64),
                        w.anchor, tokens)
    ref32 = ref.astype(np.float32)
    ell_o, B_o, tau_o, th_o = S.schedule(S.survival(ref32), si.sps)
    bad, far = conf_far_mismatches(conf, ref)
    assert not far
    same = (np.array_equal(ell_o, ell_k) and tot_k[0] == B_o and tot_k[1] == tau_o and th_o == theta_k)
    if len(bad) == 0:
        assert same, (name, np.flatnonzero(ell_o != ell_k)[:10], tot_k, B_o, tau_o, th_o, theta_k)
    else:
        print(f"{name}: {len(bad)} confidences one ulp from the oracle's (rounding midpoints); "
              f"schedule {'unchanged' if same else 'CHANGED'}: l diff at "
              f"{np.flatnonzero(ell_o != ell_k)[:10].tolist()}, B {tot_k[0]} vs {B_o}, "
              f"Theta {theta_k} vs {th_o}")
