"""A small run of the parity sweep (tests/parity_sweep.py) as a test: every
request of a few seeded full-size trials of C0, C1 and C2 — trials outside
the range of the committed sweep record — through the C ABI on the GPU, then
compared with the float64 oracle request by request under input checksums.

The token parity gate (VESSL blog, "수락 규칙": the emitted sequence must follow
the target, so the GPU's tokens must be the oracle's): mismatched requests
below 0.01 % and none away from a decision boundary.  At these sample sizes
(a few hundred requests per workload) that allows no mismatch at all; the
committed record (tests/parity_sweep_record.json) holds the full sweep of
10^4+ requests per workload."""
import argparse
import json
import os

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import parity_sweep as PS  # noqa: E402

CASES = [("C0", "5000:5200"), ("C1", "5000:5012"), ("C2", "5000:5006")]


@pytest.fixture(scope="module")
def sweep(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    d = tmp_path_factory.mktemp("sweep")
    for name, trials in CASES:
        PS.run_gpu(argparse.Namespace(config=name, trials=trials, out=str(d), threads=4))
    rec = os.path.join(str(d), "record.json")
    PS.run_compare(argparse.Namespace(dir=str(d), record=rec, workers=min(8, os.cpu_count() or 1),
                                      fresh=True))
    with open(rec) as f:
        return json.load(f)


@pytest.mark.parametrize("name,trials", CASES)
def test_small_sweep_meets_the_gate(sweep, name, trials):
    a, b = trials.split(":")
    r = sweep[f"{name}:{a}-{b}"]
    assert r["checksum_mismatch"] == 0
    assert r["trials"] == int(b) - int(a)
    assert r["rows"] >= 100
    assert r["far"] == 0, r["far_rows"]
    assert r["mismatched"] == 0, r["mismatched_rows"]
    assert max(r["q_err"], r["lse_err"], r["alpha_err"], r["ptok_err"]) <= 1e-5
    assert r["gate_met"]
