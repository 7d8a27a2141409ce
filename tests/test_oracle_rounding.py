"""Pins of the oracle's float32 evaluation order (CPU only).

Every bit-exact claim of the library rests on two pieces of float32
arithmetic in the oracle:

* the squared distance of the leaf loop of the query kernel ("Implementing ICP
  with CUDA-KDTree", section 3.2): dx = ref.x - q.x (likewise y, z) and
  d2 = dx*dx + dy*dy + dz*dz, read with C's left-to-right association,
  every operation rounded on its own (no fused multiply-add):
  d2 = fl(fl(fl(dx*dx) + fl(dy*dy)) + fl(dz*dz));
* the transform of section 2.1 / 3.3, p = R*s + t, read row by row the same
  way: p_a = fl(fl(fl(fl(R_a0*s_x) + fl(R_a1*s_y)) + fl(R_a2*s_z)) + t_a).

The expected values here come from neither float32 hardware nor the oracle:
each operation is carried out exactly on rationals and rounded to the nearest
float32, ties to even, by the definition of IEEE 754 binary32 (24-bit
significand, exponent range -126 .. 127, subnormals at 2^-149).  The inputs
are drawn (seeded) so that every other plausible reading -- another
association of the three-term sum, t added first or second, any fused
multiply-add contraction of a product into the following addition --
gives a different float32 on at least a handful of them; a re-associated or
contracted oracle therefore fails here.  A last test plants the contraction
mistake in a copy of the oracle built with -ffp-contract=fast and checks that
these pins catch it.
"""
from __future__ import annotations

import ctypes
import os
import platform
import shutil
import subprocess
import tempfile
from fractions import Fraction

import numpy as np
import pytest

from conftest import ROOT

# ------------------------------------------------------------ exact binary32

_TWO = Fraction(2)
_MAX_FINITE = (2 - Fraction(1, 2 ** 23)) * _TWO ** 127


def rnd(x: Fraction) -> Fraction:
    """x rounded to the nearest IEEE binary32 value, ties to even."""
    if x == 0:
        return Fraction(0)
    sign = 1 if x > 0 else -1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if _TWO ** e > a:
        e -= 1
    elif _TWO ** (e + 1) <= a:
        e += 1
    e = max(e, -126)                      # below 2^-126 the spacing stays 2^-149
    ulp = _TWO ** (e - 23)
    q = a / ulp
    n = q.numerator // q.denominator
    r = q - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    out = n * ulp
    if out > _MAX_FINITE:
        raise OverflowError("value rounds to infinity")
    return sign * out


def F(v) -> Fraction:
    """The exact value of a float32 (or float64) number."""
    return Fraction(float(v))


def add(a, b):
    return rnd(a + b)


def sub(a, b):
    return rnd(a - b)


def mul(a, b):
    return rnd(a * b)


def fma(a, b, c):
    """fl(a*b + c) with one rounding."""
    return rnd(a * b + c)


def as_f32(v: Fraction) -> np.float32:
    out = np.float32(float(v))
    assert Fraction(float(out)) == v, "not a float32 value"
    return out


def test_rounding_helper_against_known_values():
    # a few values fixed by the binary32 format itself
    assert rnd(Fraction(1, 3)) == Fraction(11184811, 2 ** 25)
    assert rnd(1 + Fraction(1, 2 ** 24)) == 1                       # tie -> even
    assert rnd(1 + Fraction(3, 2 ** 24)) == 1 + Fraction(2, 2 ** 23)  # tie -> even (up)
    assert rnd(1 + Fraction(1, 2 ** 24) + Fraction(1, 2 ** 60)) == 1 + Fraction(1, 2 ** 23)
    assert rnd(Fraction(3, 2 ** 150)) == Fraction(2, 2 ** 149)      # subnormal tie -> even
    assert rnd(Fraction(-5, 4)) == Fraction(-5, 4)
    assert rnd(_MAX_FINITE) == _MAX_FINITE
    with pytest.raises(OverflowError):
        rnd(_TWO ** 128)
    # agreement with an independent route on random products: numpy float64
    # holds the exact product of two float32 values, and one float32 cast of
    # it is a single correct rounding
    rng = np.random.default_rng(5)
    a = rng.standard_normal(500).astype(np.float32)
    b = rng.standard_normal(500).astype(np.float32)
    for x, y in zip(a, b):
        assert float(np.float32(np.float64(x) * np.float64(y))) == float(mul(F(x), F(y)))


# ------------------------------------------------------------ squared distance

def d2_reading(r, q):
    dx, dy, dz = (sub(F(r[k]), F(q[k])) for k in range(3))
    return add(add(mul(dx, dx), mul(dy, dy)), mul(dz, dz))


def d2_alternatives(r, q):
    """Other orders a re-associating or contracting implementation might use."""
    dx, dy, dz = (sub(F(r[k]), F(q[k])) for k in range(3))
    xx, yy, zz = mul(dx, dx), mul(dy, dy), mul(dz, dz)
    return {
        "x + (y + z)": add(xx, add(yy, zz)),
        "(x + z) + y": add(add(xx, zz), yy),
        "(y + z) + x": add(add(yy, zz), xx),
        "fma(dy, dy, xx) + zz": add(fma(dy, dy, xx), zz),
        "fma(dx, dx, yy) + zz": add(fma(dx, dx, yy), zz),
        "fma(dz, dz, xx + yy)": fma(dz, dz, add(xx, yy)),
        "fma(dz, dz, fma(dy, dy, xx))": fma(dz, dz, fma(dy, dy, xx)),
        "fma(dz, dz, fma(dx, dx, yy))": fma(dz, dz, fma(dx, dx, yy)),
    }


def _d2_cases(count=3000, seed=2024):
    """Query/reference pairs with coordinate offsets of mixed magnitudes (a
    near point on one axis, a far one on another): the three squares then
    differ in size and the order of their sum shows in the last bit."""
    rng = np.random.default_rng(seed)
    q = rng.uniform(-40, 40, (count, 3)).astype(np.float32)
    scale = 10.0 ** rng.uniform(-3, 1, (count, 3))
    r = (q + rng.standard_normal((count, 3)) * scale).astype(np.float32)
    return r, q


@pytest.fixture(scope="module")
def d2_pins():
    r, q = _d2_cases()
    want, refuted = [], {}
    for i in range(len(r)):
        v = d2_reading(r[i], q[i])
        want.append(v)
        for name, alt in d2_alternatives(r[i], q[i]).items():
            if alt != v:
                refuted.setdefault(name, []).append(i)
    return r, q, want, refuted


def test_distance_pins_discriminate(d2_pins):
    """Each alternative order disagrees with the reading on enough inputs that
    an oracle using it could not pass the next tests."""
    _, _, _, refuted = d2_pins
    for name in d2_alternatives(np.zeros(3, np.float32), np.ones(3, np.float32)):
        assert len(refuted.get(name, [])) >= 20, name


def test_oracle_distance_matches_the_reading_bit_for_bit(oracle_mod, d2_pins):
    r, q, want, _ = d2_pins
    got = oracle_mod.pair_dist2(r, q)            # dx = r - q, as the search
    exp = np.array([as_f32(v) for v in want], np.float32)
    np.testing.assert_array_equal(got.view(np.uint32), exp.view(np.uint32))
    # the same arithmetic inside the brute-force search and the tree search
    for i in range(0, len(r), 97):
        idx, d2 = oracle_mod.nn_brute(r[i:i + 1], q[i:i + 1])
        assert idx[0] == 0 and d2.view(np.uint32)[0] == exp.view(np.uint32)[i]
    tree = oracle_mod.KDTree(r[:1], 8)
    _, d2t = tree.query(q)
    exp0 = np.array([as_f32(d2_reading(r[0], q[i])) for i in range(len(q))], np.float32)
    np.testing.assert_array_equal(d2t.view(np.uint32), exp0.view(np.uint32))


# ------------------------------------------------------------ transform

def tf_reading(R, t, s):
    out = []
    for a in range(3):
        p = add(add(mul(F(R[a, 0]), F(s[0])), mul(F(R[a, 1]), F(s[1]))), mul(F(R[a, 2]), F(s[2])))
        out.append(add(p, F(t[a])))
    return out


def tf_alternatives(R, t, s):
    alts = {}
    for a in range(3):
        p0, p1, p2 = (mul(F(R[a, k]), F(s[k])) for k in range(3))
        e0, e1, e2 = (F(R[a, k]) * F(s[k]) for k in range(3))      # exact products
        ta = F(t[a])
        rows = {
            "p0 + (p1 + p2), + t": add(add(p0, add(p1, p2)), ta),
            "t first": add(add(add(ta, p0), p1), p2),
            "(p0 + p1) + (p2 + t)": add(add(p0, p1), add(p2, ta)),
            "fma p1 into p0": add(add(rnd(p0 + e1), p2), ta),
            "fma p2 into the sum": add(rnd(add(p0, p1) + e2), ta),
            "fma p1 and p2": add(rnd(rnd(p0 + e1) + e2), ta),
            "fma p0 into p1": add(add(rnd(e0 + p1), p2), ta),
            "fma chain from t": rnd(rnd(rnd(ta + e0) + e1) + e2),
        }
        for name, v in rows.items():
            alts.setdefault(name, []).append(v)
    return alts


def _tf_cases(count=1500, seed=77):
    """Rotations of random axis and angle, translations of metres, source
    points over a 40 m scene: the row terms then differ in size."""
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(count):
        axis = rng.standard_normal(3)
        axis /= np.linalg.norm(axis)
        ang = rng.uniform(-np.pi, np.pi)
        K = np.array([[0, -axis[2], axis[1]], [axis[2], 0, -axis[0]], [-axis[1], axis[0], 0]])
        R = np.eye(3) + np.sin(ang) * K + (1 - np.cos(ang)) * (K @ K)
        t = rng.uniform(-5, 5, 3)
        s = rng.uniform(-20, 20, 3) * 10.0 ** rng.uniform(-2, 0, 3)
        cases.append((R.astype(np.float32), t.astype(np.float32), s.astype(np.float32)))
    return cases


@pytest.fixture(scope="module")
def tf_pins():
    cases = _tf_cases()
    want, refuted = [], {}
    for i, (R, t, s) in enumerate(cases):
        v = tf_reading(R, t, s)
        want.append(v)
        for name, alt in tf_alternatives(R, t, s).items():
            if alt != v:
                refuted.setdefault(name, []).append(i)
    return cases, want, refuted


def test_transform_pins_discriminate(tf_pins):
    _, _, refuted = tf_pins
    names = tf_alternatives(np.eye(3, dtype=np.float32), np.zeros(3, np.float32), np.ones(3, np.float32))
    for name in names:
        assert len(refuted.get(name, [])) >= 20, name


def test_oracle_transform_matches_the_reading_bit_for_bit(oracle_mod, tf_pins):
    cases, want, _ = tf_pins
    for (R, t, s), v in zip(cases, want):
        got = oracle_mod.transform(R, t, s[None, :])[0]
        exp = np.array([as_f32(x) for x in v], np.float32)
        assert got.view(np.uint32).tolist() == exp.view(np.uint32).tolist()


# ------------------------------------------------------------ the build itself

def test_oracle_build_keeps_every_rounding():
    """The oracle must be compiled with contraction off (gcc contracts a*b + c
    into a fused multiply-add on aarch64 by default) and without fast-math."""
    import oracle
    import inspect
    src = inspect.getsource(oracle.build)
    assert '"-ffp-contract=off"' in src
    assert "-ffast-math" not in src.replace("-fno-fast-math", "")


def _fma_capable_flags():
    machine = platform.machine().lower()
    if machine in ("aarch64", "arm64"):
        return []
    if machine in ("x86_64", "amd64"):
        try:
            with open("/proc/cpuinfo") as f:
                if " fma" not in f.read():
                    return None
        except OSError:
            return None
        return ["-mfma"]
    return None


def test_pins_catch_a_contracted_oracle_build(d2_pins, tf_pins):
    """Planted mistake: the oracle's own source built with -ffp-contract=fast
    (and FMA instructions available) must disagree with the pins."""
    flags = _fma_capable_flags()
    if flags is None or shutil.which("gcc") is None:
        pytest.skip("no fused multiply-add on this host")
    src = os.path.join(ROOT, "oracle", "icp_oracle.c")
    with tempfile.TemporaryDirectory() as d:
        so = os.path.join(d, "libcontracted.so")
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=fast", *flags, "-fPIC", "-shared",
                               src, "-o", so, "-lm"])
        lib = ctypes.CDLL(so)
        P, i64 = ctypes.c_void_p, ctypes.c_int64
        lib.orc_pair_dist2.argtypes = [P, P, i64, P]
        lib.orc_transform.argtypes = [P, P, P, i64, P]
        r, q, want, _ = d2_pins
        r = np.ascontiguousarray(r)
        q = np.ascontiguousarray(q)
        got = np.empty(len(r), np.float32)
        lib.orc_pair_dist2(r.ctypes.data, q.ctypes.data, len(r), got.ctypes.data)
        exp = np.array([as_f32(v) for v in want], np.float32)
        d2_mismatch = int(np.sum(got.view(np.uint32) != exp.view(np.uint32)))
        cases, twant, _ = tf_pins
        tf_mismatch = 0
        for (R, t, s), v in zip(cases, twant):
            R9 = np.ascontiguousarray(R.reshape(9))
            s3 = np.ascontiguousarray(s.reshape(1, 3))
            out = np.empty(3, np.float32)
            lib.orc_transform(R9.ctypes.data, np.ascontiguousarray(t).ctypes.data, s3.ctypes.data, 1,
                              out.ctypes.data)
            tf_mismatch += int(np.any(out != np.array([as_f32(x) for x in v], np.float32)))
    assert d2_mismatch > 0, "a contracted build passed the distance pins"
    assert tf_mismatch > 0, "a contracted build passed the transform pins"
