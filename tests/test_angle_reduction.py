"""The kernels reduce the RoPE angle pos * inv_freq by 2 pi the Cody & Waite
way.  The indexer's query prep (csrc/indexer_common.cuh) splits 2 pi into two 26-bit
parts and an fp64 remainder; the cache-write kernels (csrc/cache_write.cu)
hold the angle as an exact fp32 pair and reduce it with a three-part fp32 2 pi
below 2^24, in fp64 above.  Checked here on the CPU against exact rational
arithmetic: the parts add up to 2 pi, the leading parts are short enough (or
the fused steps exact), and the reduced angle matches the exact remainder over
the positions and frequencies the path serves."""

import math
import os
import re
from fractions import Fraction

import numpy as np
import pytest

sympy = pytest.importorskip("sympy")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "dsa_sparse_mla_query_gb300", "csrc", "indexer_common.cuh")
SRC_CW = os.path.join(ROOT, "dsa_sparse_mla_query_gb300", "csrc", "cache_write.cu")


def constants(src=SRC, names=("kTwoPi1", "kTwoPi2", "kTwoPi3", "kInvTwoPi"), ctype="double"):
    text = open(src).read()
    out = {}
    suffix = "f" if ctype == "float" else ""
    for name in names:
        m = re.search(r"constexpr %s %s = (-?0x[0-9a-fA-F.]+p[+-]?\d+)%s;" % (ctype, name, suffix), text)
        assert m, name
        out[name] = float.fromhex(m.group(1))
    return out


TWO_PI = Fraction(str(sympy.N(2 * sympy.pi, 60)))


def significant_bits(x: float) -> int:
    m, _ = math.frexp(abs(x))
    f = Fraction(m)
    bits = 0
    while f.denominator != 1:
        f *= 2
        bits += 1
    return bits


def test_parts_sum_to_two_pi():
    c = constants()
    total = Fraction(c["kTwoPi1"]) + Fraction(c["kTwoPi2"]) + Fraction(c["kTwoPi3"])
    assert abs(total - TWO_PI) / TWO_PI < Fraction(1, 10**30)
    assert abs(Fraction(c["kInvTwoPi"]) * TWO_PI - 1) < Fraction(1, 2**52)


def test_leading_parts_have_26_bits():
    c = constants()
    assert significant_bits(c["kTwoPi1"]) <= 26
    assert significant_bits(c["kTwoPi2"]) <= 26


def reduce(th: float, c) -> float:
    # the kernel's steps; k * C1 and k * C2 are exact for |k| < 2^27, so the
    # first two products need no fused multiply-add to match it
    k = float(np.rint(th * c["kInvTwoPi"]))
    assert abs(k) < 2**27
    assert Fraction(k) * Fraction(c["kTwoPi1"]) == Fraction(k * c["kTwoPi1"])
    assert Fraction(k) * Fraction(c["kTwoPi2"]) == Fraction(k * c["kTwoPi2"])
    r = th - k * c["kTwoPi1"]
    r = r - k * c["kTwoPi2"]
    return r - k * c["kTwoPi3"]


def test_reduced_angle_matches_exact_remainder():
    c = constants()
    rng = np.random.default_rng(7)
    inv_freq = (10000.0 ** (-np.arange(32) / 32.0)).astype(np.float32)
    positions = np.concatenate([[0, 1, 2, 2047, 2048, 32767, 524287, 1 << 20, 1 << 24],
                                rng.integers(0, 1 << 22, 200)])
    worst = 0.0
    for pos in positions:
        for f in inv_freq[:: 5].tolist() + [1.0]:
            th = float(pos) * float(f)  # exact in fp64
            assert Fraction(th) == Fraction(int(pos)) * Fraction(f)
            r = reduce(th, c)
            exact = Fraction(th) - round(Fraction(th) / TWO_PI) * TWO_PI
            worst = max(worst, abs(float(Fraction(r) - exact)))
            assert abs(r) <= math.pi + 1e-9
    assert worst < 1e-12, worst


# --- the cache-write kernels -------------------------------------------------

def rne32(x: Fraction) -> Fraction:
    """x rounded to the nearest fp32 (ties to even), exactly; normal range only."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    assert -126 <= e < 128
    scaled = a / Fraction(2) ** (e - 23)  # in [2^23, 2^24)
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    return sign * Fraction(m) * Fraction(2) ** (e - 23)


def rint_even(x: Fraction) -> Fraction:
    f = x.numerator // x.denominator
    rem = x - f
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return Fraction(f)


def reduce32(pos: int, f: float, c):
    """The fp32 steps of the cache-write kernels' angle reduction, each fused
    multiply-add rounded once, with the exactness of the first step checked."""
    pf = Fraction(pos)
    F = Fraction(f)
    hi = rne32(pf * F)
    lo = rne32(pf * F - hi)
    assert hi + lo == pf * F  # the product's residual is exact
    k = rint_even(rne32(hi * Fraction(c["kInvTwoPiF"])))
    exact_r1 = hi - k * Fraction(c["kTwoPi1"])
    r = rne32(exact_r1)
    assert r == exact_r1, (pos, f)  # exact: |r| < 8 on a 2^-21 grid
    r = rne32(r - k * Fraction(c["kTwoPi2"]))
    r = rne32(r - k * Fraction(c["kTwoPi3"]))
    r = rne32(r + lo) if r + lo != 0 else Fraction(0)
    return r, k


def cw_constants():
    c = constants(SRC_CW, ("kTwoPi1", "kTwoPi2", "kTwoPi3", "kInvTwoPiF"), "float")
    c.update(constants(SRC_CW, ("kTwoPiHi", "kTwoPiMid", "kTwoPiLo", "kInvTwoPiD"), "double"))
    return c


def test_cache_write_parts_sum_to_two_pi():
    c = cw_constants()
    for name in c:
        if name in ("kTwoPi1", "kTwoPi2", "kTwoPi3", "kInvTwoPiF"):
            assert float(np.float32(c[name])) == c[name], name  # fp32 values
    t32 = Fraction(c["kTwoPi1"]) + Fraction(c["kTwoPi2"]) + Fraction(c["kTwoPi3"])
    assert abs(t32 - TWO_PI) / TWO_PI < Fraction(1, 2**70)
    assert abs(Fraction(c["kInvTwoPiF"]) * TWO_PI - 1) < Fraction(1, 2**24)
    t64 = Fraction(c["kTwoPiHi"]) + Fraction(c["kTwoPiMid"]) + Fraction(c["kTwoPiLo"])
    assert abs(t64 - TWO_PI) / TWO_PI < Fraction(1, 10**30)
    assert significant_bits(c["kTwoPiHi"]) <= 26 and significant_bits(c["kTwoPiMid"]) <= 26


def test_cache_write_fp32_reduction_matches_exact_remainder():
    c = cw_constants()
    rng = np.random.default_rng(11)
    inv_freq = (10000.0 ** (-np.arange(32) / 32.0)).astype(np.float32)
    positions = np.concatenate([[0, 1, 3, 4, 2047, 32767, 524287, (1 << 20) - 1, (1 << 24) - 1],
                                rng.integers(0, 1 << 24, 120)])
    worst = 0.0
    for pos in positions.tolist():
        for f in inv_freq[::4].tolist() + [1.0, float(np.float32(0.7498942))]:
            if abs(pos * f) >= 2**24:
                continue  # the kernels take the fp64 reduction there
            r, k = reduce32(pos, f, c)
            exact = Fraction(pos) * Fraction(f) - k * TWO_PI
            worst = max(worst, abs(float(r - exact)))
            assert abs(r) < 8
    assert worst < 3e-7, worst
