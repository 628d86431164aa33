"""The seeded generators: exact bf16 rounding, exact uniforms, reproducibility,
request sharding."""
import numpy as np
import pytest

from speculative_decoding_draft_04_gb300 import workloads as W


def test_bf16_round_is_nearest_even():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.normal(0, 3, 20000), rng.normal(0, 0.02, 20000),
                        [0.0, -0.0, 1.0, -2.5, 1e-30, 3.0e38]])
    bits = W.bf16_round(x)
    v = W.bf16_to_f64(bits)
    # neighbours one bf16 step below and above the chosen value
    up = W.bf16_to_f64((bits.astype(np.int32) + 1).astype(np.uint16))
    dn = W.bf16_to_f64((bits.astype(np.int32) - 1).astype(np.uint16))
    err = np.abs(x - v)
    assert np.all(err <= np.abs(x - up) + 0.0)
    ok_dn = np.isnan(dn) | (err <= np.abs(x - dn))
    assert np.all(ok_dn)
    # ties go to the even pattern: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7
    assert W.bf16_to_f64(W.bf16_round(np.array([1.0 + 2.0 ** -8])))[0] == 1.0
    assert W.bf16_to_f64(W.bf16_round(np.array([1.0 + 3 * 2.0 ** -8])))[0] == 1.0 + 2.0 ** -6


def test_uniforms_exact_and_open_interval():
    u = W.uniforms(np.random.default_rng(0), 100000)
    assert u.dtype == np.float32
    assert np.all(u > 0) and np.all(u < 1)
    m = u.astype(np.float64) / W.U23 - 0.5
    assert np.all(m == np.round(m))
    assert u.max() <= np.float32(1.0 - 2.0 ** -24)


def test_workload_reproducible_and_prefix_stable():
    spec = W.config("C2", V=1024, B=16)
    a = W.make_workload(spec, trial=3)
    b = W.make_workload(spec, trial=3)
    c = W.make_workload(spec, trial=3, B=5)
    for f in ("target", "U", "W1", "W2", "anchor", "temperature", "verify_len",
              "u_draft", "u_accept", "u_final"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
        if f in ("W1", "W2"):
            np.testing.assert_array_equal(getattr(a, f), getattr(c, f))
        else:
            np.testing.assert_array_equal(getattr(a, f)[:5], getattr(c, f))
    assert np.all((a.verify_len >= 1) & (a.verify_len <= 7))
    d = W.make_workload(spec, trial=4)
    assert not np.array_equal(a.u_draft, d.u_draft)


def test_zipf_target_shape():
    spec = W.config("C3", V=4096, B=2, gamma=2)
    w = W.make_workload(spec, trial=0)
    t = w.f64("target")
    # heavy head: the top 1% of tokens carry far more than 1% of the mass
    p = np.exp(t[0, 0] - t[0, 0].max())
    p /= p.sum()
    assert np.sort(p)[::-1][:41].sum() > 0.2
    assert set(np.unique(w.temperature)) <= {np.float32(0.6), np.float32(1.0)}


@pytest.mark.parametrize("B,world", [(128, 2), (7, 3), (1, 2), (256, 8)])
def test_shard_rows_partition(B, world):
    parts = [W.shard_rows(B, r, world) for r in range(world)]
    allr = np.concatenate(parts)
    np.testing.assert_array_equal(allr, np.arange(B))
    sizes = [len(p) for p in parts]
    assert max(sizes) - min(sizes) <= 1
