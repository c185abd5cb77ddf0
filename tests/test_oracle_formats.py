"""Pins for the oracle's scalar formats (E2M1 values, E4M3 values, both encoders).

The E2M1 grid is the one in the quantization recipe; E4M3 values are checked
against torch's float8_e4m3fn; both encoders are checked against an exhaustive
exact-rational nearest search (tests/_exact.py) and against torch's own fp8 cast.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests import _exact as ex


def test_e2m1_values_are_the_grid():
    for c in range(16):
        mag = float(ex.GRID[c & 7])
        assert oracle.e2m1_value(c) == (-mag if c & 8 else mag)


def test_e4m3_values_match_torch():
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for byte in range(256):
        v = oracle.e4m3_value(byte)
        if np.isnan(ref[byte]):
            assert np.isnan(v), byte
        else:
            assert v == ref[byte], (byte, v, ref[byte])
    # largest finite value and smallest subnormal of OCP E4M3
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(1) == 2.0 ** -9


@pytest.mark.parametrize("den", [1.0, 6.0, 6.0 * float(np.float32(0.0123)), 2.0 ** -20, 6.0 * float(np.float32(3.3e-5))])
def test_e4m3_encode_exact_values_and_ties(den):
    vals = [Fraction(oracle.e4m3_value(b)) for b in range(127)]
    d = Fraction(den)
    for b in range(127):
        assert oracle.e4m3_encode_ratio(float(vals[b] * d), den) == b
    for b in range(126):
        mid = (vals[b] + vals[b + 1]) / 2
        even = b if b % 2 == 0 else b + 1
        assert oracle.e4m3_encode_ratio(float(mid * d), den) == even
        # a hair below / above the midpoint goes to the nearer neighbour
        lo = float(mid * d) * (1 - 2.0 ** -40)
        hi = float(mid * d) * (1 + 2.0 ** -40)
        assert oracle.e4m3_encode_ratio(lo, den) == b
        assert oracle.e4m3_encode_ratio(hi, den) == b + 1
    # saturation at 448
    assert oracle.e4m3_encode_ratio(float(Fraction(464) * d), den) == 0x7E
    assert oracle.e4m3_encode_ratio(float(Fraction(10 ** 6) * d), den) == 0x7E


def test_e4m3_encode_matches_torch_cast():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.uniform(0, 448, 4000), np.exp(rng.uniform(np.log(1e-4), np.log(448), 4000))]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode_ratio(float(x), 1.0) for x in v])
    assert (got == ref).all(), np.nonzero(got != ref)


def test_e4m3_encode_bruteforce_ratios():
    rng = np.random.default_rng(2)
    for _ in range(600):
        g = np.float32(np.exp(rng.uniform(np.log(1e-8), np.log(10.0))))
        num = np.float32(float(g) * 2688 * rng.uniform(0, 1.02))
        want = ex.nearest_even(Fraction(float(num)) / (6 * Fraction(float(g))), ex.E4M3)
        assert oracle.e4m3_encode_ratio(float(num), 6.0 * float(g)) == want


def test_e2m1_encode_bruteforce():
    rng = np.random.default_rng(3)
    for _ in range(3000):
        s = int(rng.integers(1, 127))
        g = np.float32(np.exp(rng.uniform(np.log(1e-6), np.log(1.0))))
        S = Fraction(oracle.e4m3_value(s)) * Fraction(float(g))
        x = np.float32(float(S) * rng.uniform(-7.0, 7.0))
        want = ex.nearest_even(abs(Fraction(float(x))) / S, ex.GRID) | (8 if np.signbit(x) else 0)
        assert oracle.e2m1_encode(float(x), float(S)) == want
    # every grid midpoint, both signs: ties to the even code
    for k in range(7):
        mid = (ex.GRID[k] + ex.GRID[k + 1]) / 2
        even = k if k % 2 == 0 else k + 1
        assert oracle.e2m1_encode(float(mid), 1.0) == even
        assert oracle.e2m1_encode(-float(mid), 1.0) == even | 8
    assert oracle.e2m1_encode(-0.0, 1.0) == 8 and oracle.e2m1_encode(0.0, 1.0) == 0
    assert oracle.e2m1_encode(1e9, 1.0) == 7 and oracle.e2m1_encode(0.3, 0.0) == 0


def test_e2m1_guided_is_a_neighbour():
    rng = np.random.default_rng(4)
    for _ in range(3000):
        x = float(np.float32(rng.uniform(-7, 7)))
        up = int(rng.integers(0, 2))
        c = oracle.e2m1_encode_guided(x, 1.0, up)
        a = abs(Fraction(x))
        assert (c >> 3) == int(np.signbit(x))
        mag = c & 7
        if a >= 6:
            assert mag == 7
            continue
        lo = max(k for k in range(8) if ex.GRID[k] <= a)
        if ex.GRID[lo] == a:
            assert mag == lo
        else:
            assert mag == (lo + 1 if up else lo)
    # exact grid values are kept whatever the mask says
    for k in range(8):
        for up in (0, 1):
            assert oracle.e2m1_encode_guided(float(ex.GRID[k]), 1.0, up) == k
