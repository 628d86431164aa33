"""Double-float arithmetic of the extended-precision re-decision path, checked
on the host: spec_df.cuh compiles as plain C++ (every step explicitly
rounded), and the same code runs on the GPU.  Pins: exact rational arithmetic
(fractions / decimal) and numpy's float64 exp."""
import os
import shutil
import subprocess
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if not cxx:
        pytest.skip("no C++ compiler")
    exe = str(tmp_path_factory.mktemp("df") / "df_probe")
    subprocess.run([cxx, "-O2", "-std=c++17", "-ffp-contract=off", "-o", exe,
                    os.path.join(HERE, "host", "df_probe.cpp")], check=True)

    def run(lines):
        out = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True,
                             check=True).stdout.split()
        v = np.array(out, float).reshape(-1, 2)
        return v[:, 0], v[:, 1]
    return run


def _split(x):
    """The double-float nearest each double (what the device's dd_from_double makes)."""
    hi = x.astype(np.float32).astype(np.float64)
    lo = (x - hi).astype(np.float32).astype(np.float64)
    return hi + lo


def test_exp_accuracy(probe):
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-60, 0.5, 20000), rng.uniform(-0.006, 0.006, 4000),
                        np.array([0.0, -1e-30, 1e-9, -0.00541, 0.00541, -59.9, -1.0, -0.5])])
    hi, lo = probe([f"exp {v:.17g}" for v in x])
    ref = np.exp(_split(x))
    rel = np.abs(hi + lo - ref) / ref
    assert rel.max() < 5e-14, (rel.max(), x[rel.argmax()])


def test_exp_tiny_and_underflow(probe):
    x = np.array([-70.0, -80.0, -90.0, -102.0, -103.0, -200.0, -1e30])
    hi, lo = probe([f"exp {v:.17g}" for v in x])
    ref = np.exp(_split(x))
    assert np.all(np.abs(hi + lo - ref) < 1e-30)           # negligible next to O(1) weights
    assert hi[-3:].tolist() == [0.0, 0.0, 0.0]


def test_exp_table_is_two_to_the_j_over_64(probe):
    getcontext().prec = 50
    hi, lo = probe(["tab"])
    for j in range(64):
        exact = Decimal(2) ** (Decimal(j) / 64)
        got = Decimal(float(hi[j])) + Decimal(float(lo[j]))
        assert abs(got - exact) / exact < Decimal("1e-14"), j


def _bf16(rng, n, scale):
    v = (rng.standard_normal(n) * scale).astype(np.float32)
    b = (v.view(np.uint32) + 0x8000) & 0xFFFF0000         # round to bf16 (ties away: fine for a test)
    return b.astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("n,scale", [(16, 1.0), (256, 0.02), (256, 3.0), (64, 1e-3)])
def test_compensated_dot_of_bf16_products(probe, n, scale):
    """Products of bf16 values are exact in fp32; TwoSum accumulation keeps
    every rounding error, so the double-float result is within 1e-13 of the
    sum of magnitudes (the bound used by the re-decision's error analysis)."""
    rng = np.random.default_rng(n)
    lines, exact, mags = [], [], []
    for _ in range(50):
        a, w = _bf16(rng, n, scale), _bf16(rng, n, 0.05)
        lines.append(f"dot {n} " + " ".join(f"{x:x}" for x in a.view(np.uint32)) + " " +
                     " ".join(f"{x:x}" for x in w.view(np.uint32)))
        prods = [Fraction(float(p)) * Fraction(float(q)) for p, q in zip(a, w)]
        exact.append(sum(prods, Fraction(0)))
        mags.append(sum(abs(p) for p in prods))
    hi, lo = probe(lines)
    for h, l, e, m in zip(hi, lo, exact, mags):
        err = abs(Fraction(float(h)) + Fraction(float(l)) - e)
        assert err <= Fraction(1, 10**13) * m + Fraction(1, 10**40), (float(err), float(m))


def test_mul_and_add_are_double_float_accurate(probe):
    rng = np.random.default_rng(7)
    a = _split(rng.uniform(-4, 4, 500))
    b = _split(rng.uniform(-4, 4, 500))
    ah, bh = a.astype(np.float32), b.astype(np.float32)
    al, bl = (a - ah).astype(np.float32), (b - bh).astype(np.float32)
    args = [f"{x:.9g} {y:.9g} {z:.9g} {t:.9g}" for x, y, z, t in zip(ah, al, bh, bl)]
    for op, f in (("mul", lambda x, y: x * y), ("add", lambda x, y: x + y)):
        hi, lo = probe([f"{op} {s}" for s in args])
        for i in range(len(a)):
            xa = Fraction(float(ah[i])) + Fraction(float(al[i]))
            xb = Fraction(float(bh[i])) + Fraction(float(bl[i]))
            ex = f(xa, xb)
            got = Fraction(float(hi[i])) + Fraction(float(lo[i]))
            scale = abs(xa) * abs(xb) if op == "mul" else abs(xa) + abs(xb)
            assert abs(got - ex) <= Fraction(1, 2**44) * scale, (op, i)


def test_reciprocal(probe):
    rng = np.random.default_rng(3)
    t = np.concatenate([rng.uniform(0.05, 8.0, 400), [0.6, 0.7, 1.0, 3.0, 1e-3, 1e3]]).astype(np.float32)
    hi, lo = probe([f"rcp {v:.9g}" for v in t])
    for i, v in enumerate(t):
        exact = 1 / Fraction(float(v))
        got = Fraction(float(hi[i])) + Fraction(float(lo[i]))
        assert abs(got - exact) <= exact / 2**46, (v, float(got), float(exact))


def test_log_of_double_float(probe):
    getcontext().prec = 50
    rng = np.random.default_rng(4)
    z = _split(np.concatenate([rng.uniform(0.5, 2.0, 300), 10 ** rng.uniform(-3, 6, 300)]))
    zh = z.astype(np.float32)
    zl = (z - zh).astype(np.float32)
    hi, _ = probe([f"log {a:.9g} {b:.9g}" for a, b in zip(zh, zl)])
    for i in range(len(z)):
        exact = (Decimal(float(zh[i])) + Decimal(float(zl[i]))).ln()
        bound = Decimal("3e-14") * (1 + abs(exact))          # the exponential's relative error, carried
        assert abs(Decimal(float(hi[i])) - exact) < bound, (float(z[i]), hi[i], float(exact))


@pytest.mark.parametrize("n", [8, 264, 4352])
def test_dot2_of_bf16_by_fp32_products(probe, n):
    """Dot2 over products of a bf16 and an fp32 value (the confidence head's
    w^T [h; e]): the products are not exact in fp32, TwoProd recovers them."""
    rng = np.random.default_rng(n + 1)
    lines, exact, mags = [], [], []
    for _ in range(20):
        a = _bf16(rng, n, 1.0)
        w = (rng.standard_normal(n) / np.sqrt(n)).astype(np.float32)
        lines.append(f"dot2 {n} " + " ".join(f"{x:x}" for x in a.view(np.uint32)) + " " +
                     " ".join(f"{x:x}" for x in w.view(np.uint32)))
        prods = [Fraction(float(p)) * Fraction(float(q)) for p, q in zip(a, w)]
        exact.append(sum(prods, Fraction(0)))
        mags.append(sum(abs(p) for p in prods))
    hi, lo = probe(lines)
    for h, l, e, m in zip(hi, lo, exact, mags):
        err = abs(Fraction(float(h)) + Fraction(float(l)) - e)
        assert err <= Fraction(1, 10**13) * m + Fraction(1, 10**40), (float(err), float(m))


def test_division(probe):
    rng = np.random.default_rng(8)
    a = _split(rng.uniform(-4, 4, 400))
    b = _split(np.concatenate([rng.uniform(0.5, 3.0, 300), -rng.uniform(1e-3, 1e3, 100)]))
    ah, bh = a.astype(np.float32), b.astype(np.float32)
    al, bl = (a - ah).astype(np.float32), (b - bh).astype(np.float32)
    hi, lo = probe([f"div {x:.9g} {y:.9g} {z:.9g} {t:.9g}" for x, y, z, t in zip(ah, al, bh, bl)])
    for i in range(len(a)):
        ex = (Fraction(float(ah[i])) + Fraction(float(al[i]))) / (Fraction(float(bh[i])) + Fraction(float(bl[i])))
        got = Fraction(float(hi[i])) + Fraction(float(lo[i]))
        assert abs(got - ex) <= abs(ex) / 2**44, i


def test_sigmoid(probe):
    """1/(1 + e^{-z}) to about 1e-13 relative over the whole fp32 range of c
    (pinned with 50-digit decimal arithmetic)."""
    getcontext().prec = 50
    rng = np.random.default_rng(9)
    z = _split(np.concatenate([rng.uniform(-8, 8, 2000), rng.uniform(-100, 100, 300),
                               [0.0, 1e-9, -1e-9, 17.0, -17.0, 30.0, -85.0]]))
    zh = z.astype(np.float32)
    zl = (z - zh).astype(np.float32)
    hi, lo = probe([f"sig {a:.9g} {b:.9g}" for a, b in zip(zh, zl)])
    for i in range(len(z)):
        x = Decimal(float(zh[i])) + Decimal(float(zl[i]))
        exact = 1 / (1 + (-x).exp())
        got = Decimal(float(hi[i])) + Decimal(float(lo[i]))
        # relative, down to the double-float's resolution near the fp32 minimum
        bound = max(Decimal("2e-13") * exact, Decimal("1e-44"))
        assert abs(got - exact) <= bound, (float(z[i]), float(got), float(exact))
    # the rounded float is the nearest float of the exact value (no midpoint is near here)
    c32 = (hi + lo).astype(np.float32)
    ref = 1 / (1 + np.exp(-z))
    assert np.mean(c32 == ref.astype(np.float32)) > 0.999


def test_tanh(probe):
    """tanh to about 1e-12 relative from 1e-8 to saturation (50-digit decimal pin)."""
    getcontext().prec = 50
    rng = np.random.default_rng(10)
    mag = np.concatenate([10 ** rng.uniform(-8, 1.7, 3000), [1e-4, 9.9e-5, 1.01e-4, 0.5, 30.0, 60.0]])
    z = _split(mag * rng.choice([-1.0, 1.0], size=mag.size))
    zh = z.astype(np.float32)
    zl = (z - zh).astype(np.float32)
    hi, lo = probe([f"tanh {a:.9g} {b:.9g}" for a, b in zip(zh, zl)])
    for i in range(len(z)):
        x = Decimal(float(zh[i])) + Decimal(float(zl[i]))
        e = (2 * x).exp()
        exact = (e - 1) / (e + 1)
        got = Decimal(float(hi[i])) + Decimal(float(lo[i]))
        assert abs(got - exact) <= Decimal("1e-12") * abs(exact), (float(x), float(got), float(exact))


def _bf16_nearest(v: Fraction) -> int:
    """Bit pattern of the bfloat16 nearest to v (ties to even), by brute force
    over the two neighbours of v's float32 truncation."""
    f = np.float32(float(v))
    bits = int(f.view(np.uint32)) & 0xFFFF0000
    cands = [bits, bits + 0x10000, bits - 0x10000]
    best = None
    for c in cands:
        cv = Fraction(float(np.uint32(c & 0xFFFFFFFF).view(np.float32)))
        d = abs(cv - v)
        key = (d, (c >> 16) & 1)
        if best is None or key < best[0]:
            best = (key, (c >> 16) & 0xFFFF)
    return best[1]


def test_bf16_rounding_of_double_floats(probe):
    """Nearest bfloat16 of hi + lo, including values whose hi sits exactly on a
    bfloat16 midpoint (lo then decides) and true ties (lo = 0)."""
    rng = np.random.default_rng(11)
    hs, ls = [], []
    for _ in range(3000):
        h = np.float32(rng.normal() * 10 ** rng.uniform(-3, 3))
        if rng.random() < 0.5:                       # force hi onto a midpoint
            h = np.uint32((int(h.view(np.uint32)) & 0xFFFF0000) | 0x8000).view(np.float32)
        ulp = float(np.spacing(np.float32(abs(h))))
        lo = np.float32(rng.choice([0.0, rng.uniform(-0.5, 0.5) * ulp]))
        hs.append(h)
        ls.append(lo)
    out = probe([f"bf16 {int(np.float32(h).view(np.uint32)):x} {int(np.float32(l).view(np.uint32)):x}"
                 for h, l in zip(hs, ls)])[0]
    for h, l, got in zip(hs, ls, out):
        v = Fraction(float(h)) + Fraction(float(l))
        assert int(got) == _bf16_nearest(v), (float(h), float(l))
