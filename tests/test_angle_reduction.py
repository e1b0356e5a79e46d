"""The query-prep kernel reduces the RoPE angle pos * inv_freq by 2 pi with a
Cody & Waite split of 2 pi into two 26-bit parts and an fp64 remainder (the
constants live in csrc/indexer.cu).  Checked here on the CPU against exact
rational arithmetic: the parts add up to 2 pi, the first two are short enough
for k * part to be exact, and the reduced angle matches the exact remainder
over the positions and frequencies the path serves."""

import math
import os
import re
from fractions import Fraction

import numpy as np
import pytest

sympy = pytest.importorskip("sympy")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "dsa_sparse_mla_query_gb300", "csrc", "indexer.cu")


def constants():
    text = open(SRC).read()
    out = {}
    for name in ("kTwoPi1", "kTwoPi2", "kTwoPi3", "kInvTwoPi"):
        m = re.search(r"constexpr double %s = (-?0x[0-9a-fA-F.]+p[+-]?\d+);" % name, text)
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
