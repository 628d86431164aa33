"""Host-side logic of bench.py (no GPU): the DRAM-traffic hook that reads a
committed ncu summary only while the kernel's sources are unchanged, the
clock-record summary that decides whether a timing is kept, and the
algorithmic byte counts behind the roofline figures."""
import hashlib
import tempfile
import types

import numpy as np

import bench


def _profile(root, kernel, config, traffic, sources, sha):
    d = root / "profiles"
    d.mkdir(exist_ok=True)
    (d / f"{kernel}_{config}.md").write_text(
        f"# {kernel}\n\n    traffic_bytes_per_launch: {traffic}\n"
        f"    sources: {' '.join(sources)}\n    source_sha256: {sha}\n")


def test_traffic_hook_follows_the_sources_hash(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "a.cu").write_text("kernel A\n")
    (tmp_path / "b.cuh").write_text("header B\n")
    sha = hashlib.sha256(b"kernel A\n" + b"header B\n").hexdigest()
    _profile(tmp_path, "k", "C2", 1234, ["a.cu", "b.cuh"], sha)
    assert bench.recorded_traffic("k", "C2") == 1234.0
    assert bench.recorded_traffic("k", "C1") is None            # no summary for that workload
    (tmp_path / "b.cuh").write_text("header B, edited\n")     # sources changed since the capture
    assert bench.recorded_traffic("k", "C2") is None
    _profile(tmp_path, "k", "C2", 1234, ["a.cu", "missing.cu"], sha)
    assert bench.recorded_traffic("k", "C2") is None


def _clock_summary(lines):
    c = bench.ClockSampler(0)
    c.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    c.f.write("\n".join(lines) + "\n")
    return c.summary()


def test_clock_summary_median_and_reasons():
    ok = "0, {sm}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {cap}"
    s = _clock_summary([ok.format(sm=2070, cap="Not Active"), ok.format(sm=2055, cap="Active"),
                        ok.format(sm=2070, cap="Not Active"), "garbage line",
                        "0, [N/A], 2070, 1, 0x0, a, b, c, d"])
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    hot = "0, 1500, 2070, 1400.0, 0x0, Not Active, Active, Not Active, Not Active"
    assert _clock_summary([hot])["reasons"] == ["hw_thermal_slowdown"]
    assert _clock_summary([])["reasons"] == ["no samples"]


def test_algorithmic_bytes():
    w = types.SimpleNamespace(B=3, gamma=4, V=100, r=16, dtype="bf16",
                              verify_len=np.array([0, 2, 4], np.int32))
    draft, verify, per = bench.algorithmic_bytes(w)
    s = 2
    assert draft == 3 * 4 * 100 * s + 16 * 100 * s
    # target rows j <= L_b, U rows j < L_b, W2 once
    assert verify == (1 + 3 + 5) * 100 * s + (0 + 2 + 4) * 100 * s + 16 * 100 * s
    assert per["draft_persistent"] == draft
    assert per["target_stats"] + per["verify_tile"] == verify
    w.dtype = "f32"
    assert bench.algorithmic_bytes(w)[0] == (3 * 4 * 100 + 16 * 100) * 4
