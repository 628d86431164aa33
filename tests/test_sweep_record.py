"""The committed record of the full parity sweep (tests/parity_sweep.py:
every request of many seeded full-size trials, GPU outputs compared with the
float64 oracle under input checksums) meets the token parity gate at its own
scale: at least 1000 trials of C0-C2 and 100 of C3/C4, at least 10^4
requests each, mismatched requests below 0.01 % with none away from a
decision boundary, identical inputs on both sides, and every probability
within 1e-5 of the oracle's."""
import json
import os

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
RECORD = os.path.join(HERE, "parity_sweep_record.json")
MIN_TRIALS = {"C0": 1000, "C1": 1000, "C2": 1000, "C3": 100, "C4": 100}


def _load():
    with open(RECORD) as f:
        return json.load(f)


@pytest.mark.parametrize("name", sorted(MIN_TRIALS))
def test_record_meets_the_gate(name):
    rec = _load()
    runs = [r for k, r in rec.items() if k.split(":")[0] == name]
    assert runs, f"no sweep of {name} in the record"
    trials = sum(r["trials"] for r in runs)
    rows = sum(r["rows"] for r in runs)
    mism = sum(r["mismatched"] for r in runs)
    assert trials >= MIN_TRIALS[name]
    assert rows >= 10_000
    assert all(r["checksum_mismatch"] == 0 for r in runs)
    assert all(r["far"] == 0 and not r["far_rows"] for r in runs)
    assert mism < 1e-4 * rows
    assert len([x for r in runs for x in r["mismatched_rows"]]) == mism
    for r in runs:
        assert max(r["q_err"], r["lse_err"], r["alpha_err"], r["ptok_err"]) <= 1e-5
        assert r["near"] <= r["rows"]
        assert r["gate_met"]
