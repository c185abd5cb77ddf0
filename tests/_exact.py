"""Exhaustive, exact-rational brute force used to pin the oracle.

These helpers do not follow the oracle's method (walking midpoints); they
enumerate every candidate value with Python Fractions and take the argmin of
the exact distance, ties resolved to the even encoding. Decoding comes from
torch's float8_e4m3fn (a library routine) and the E2M1 grid printed in the
quantization recipe.
"""
from fractions import Fraction

import numpy as np
import torch

GRID = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4), Fraction(6)]


def e4m3_table():
    """Exact values of the 127 finite non-negative E4M3 bytes (0x00..0x7E), decoded by torch."""
    b = torch.arange(0, 127, dtype=torch.uint8)
    vals = b.view(torch.float8_e4m3fn).to(torch.float64).tolist()
    return [Fraction(v) for v in vals]


E4M3 = e4m3_table()


def nearest_even(target: Fraction, values):
    """Index of the value nearest to target; ties to the even index (values sorted ascending)."""
    best = None
    for i, v in enumerate(values):
        d = abs(target - v)
        if best is None or d < best[0] or (d == best[0] and i % 2 == 0):
            best = (d, i)
    return best[1]


def f32(x) -> Fraction:
    return Fraction(float(np.float32(x)))


def global_scale(amax) -> np.float32:
    """fp32 nearest to amax / 2688 (ties to even), by checking neighbouring fp32 values."""
    q = Fraction(float(np.float32(amax))) / 2688
    c = np.float32(float(q))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best = None
    for v in cands:
        d = abs(Fraction(float(v)) - q)
        even = (int(np.array(v, np.float32).view(np.uint32)) & 1) == 0
        if best is None or d < best[0] or (d == best[0] and even):
            best = (d, v)
    return np.float32(best[1])


def quantize_block(vals, g: np.float32, mask_bits=None):
    """Scale byte and codes of one 16-element block by exhaustive search."""
    g = Fraction(float(g))
    signs = [int(np.signbit(np.float64(v))) for v in vals]
    vals = [Fraction(float(v)) for v in vals]
    bamax = max(abs(v) for v in vals)
    if g == 0:
        s = 0
    else:
        s = nearest_even(bamax / (6 * g), E4M3)
    S = E4M3[s] * g
    codes = []
    for i, v in enumerate(vals):
        if S == 0:
            mag = 0
        elif mask_bits is None:
            mag = nearest_even(abs(v) / S, GRID)
        else:
            a = abs(v) / S
            if a >= 6:
                mag = 7
            else:
                lo = max(k for k in range(8) if GRID[k] <= a)
                mag = lo if (GRID[lo] == a or not mask_bits[i]) else lo + 1
        codes.append(mag | (8 if signs[i] else 0))
    return s, codes


def unpack(codes_u8: np.ndarray) -> np.ndarray:
    c = np.asarray(codes_u8, dtype=np.uint8)
    out = np.empty(c.shape[:-1] + (c.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = c & 15
    out[..., 1::2] = c >> 4
    return out


def pack(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def dequant_torch(codes_u8, scales_u8, g) -> np.ndarray:
    """deq = grid(code) * e4m3(scale) * g, with E4M3 decoded by torch, in float64."""
    c = unpack(codes_u8)
    grid = np.array([float(v) for v in GRID], np.float64)
    val = grid[c & 7] * np.where(c & 8, -1.0, 1.0)
    sc = torch.from_numpy(np.ascontiguousarray(scales_u8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return val * np.repeat(sc, 16, axis=-1) * float(g)
