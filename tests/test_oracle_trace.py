"""Pins of the oracle's TRACE record / cached-replay functions (CPU only).

Record: the rollout side keeps, per element, whether the plain NVFP4 rounding went up in magnitude
(TRACE summary, section "仕組みの工学的な理解"). Replay: the training side re-encodes from the cached
scale bytes and g with those rounding directions (section "TRACE の中心的なアイデア"). Each pin
checks the oracle against something it does not compute itself: hand-derived values, the exact
dequantization through torch, or the bracketing relations that define floor and ceiling codes.
"""
import numpy as np
import pytest

import oracle
import synth
from tests import _exact as ex

GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _bits(mask, n):
    return np.unpackbits(np.asarray(mask, np.uint32).view(np.uint8), bitorder="little")[:n]


# g = 2688 / 2688 = 1; the first block's amax is 6, so its scale byte is E4M3(1.0) = 0x38 and
# S = 1: every quotient is the value itself. The second block's amax 6.3 gives 6.3 / 6 = 1.05,
# nearest E4M3 1.0 (0x38) again, so 6.3 saturates to 6 (rounded down).
HAND_ROWS = [
    [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 0.6, 0.9, -0.9, 1.0, 0.0, -0.0, 2.9, 4.5],
    [6.3, 5.5, -5.5, 0.2, 0.3, 1.4, 1.6, 2.2, 2.6, 3.2, 3.9, 4.1, 0.1, 0.4, 0.55, 0.45],
]
# row 0: ties go to the even grid index: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2,
# 3.5 -> 4, 5 -> 4; 0.6 -> 0.5, 0.9 -> 1, 2.9 -> 3, 4.5 -> 4; 6, 1 and the zeros are on the grid.
# row 1: 6.3 -> 6 (saturated, down); 5.5 -> 6 (up); 0.2 -> 0; 0.3 -> 0.5; 1.4 -> 1.5; 1.6 -> 1.5;
# 2.2 -> 2; 2.6 -> 3; 3.2 -> 3; 3.9 -> 4; 4.1 -> 4; 0.1 -> 0; 0.4 -> 0.5; 0.55 -> 0.5; 0.45 -> 0.5
HAND_UP = [0, 1, 0, 1, 0, 1, 0, 0, 0, 1, 1, 0, 0, 0, 1, 0] + [0, 1, 1, 0, 1, 1, 0, 0, 1, 0, 1, 0, 0, 1, 0, 1]


def test_record_hand_block():
    x = np.array(HAND_ROWS, np.float32)
    codes, scales, g, mask = oracle.quantize_record(x, amax_in=2688.0)
    assert g == np.float32(1.0)
    assert scales.tolist() == [[0x38], [0x38]]
    assert _bits(mask, 32).tolist() == HAND_UP
    # the codes are the plain ones
    c_plain, s_plain, g_plain = oracle.quantize(x, amax_in=2688.0)
    assert np.array_equal(codes, c_plain) and np.array_equal(scales, s_plain) and g == g_plain
    mags = (ex.unpack(codes) & 7).reshape(2, 16)
    assert [GRID[m] for m in mags[0]] == [0, 1, 1, 2, 2, 4, 4, 6, 0.5, 1, 1, 1, 0, 0, 3, 4]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_record_bits_equal_exact_direction(dtype):
    """Bit i is set exactly where |deq(plain code)| > |x| (exact dequantization through torch)."""
    if dtype == "bf16":
        x = synth.heavy_tail_activation_bf16(24, 256, 5, 1)
        xv = synth.bf16_to_f32(x).astype(np.float64)
    else:
        x = synth.weight_f32(24, 256, 0.02, 5, 2, outlier_frac=0.02)
        xv = x.astype(np.float64)
    codes, scales, g, mask = oracle.quantize_record(x)
    up = np.abs(ex.dequant_torch(codes, scales, g)) > np.abs(xv)
    assert np.array_equal(_bits(mask, x.size).astype(bool), up.reshape(-1))
    assert 0.2 < up.mean() < 0.8


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_guided_with_record_gives_plain(dtype):
    """Rounding guided by the record reproduces the plain encoding (codes, scales and g)."""
    if dtype == "bf16":
        x = synth.activation_bf16(40, 160, 6, 1)
    else:
        x = synth.weight_f32(40, 160, 0.02, 6, 2, outlier_frac=0.01)
    codes, scales, g, mask = oracle.quantize_record(x)
    cg, sg, gg = oracle.quantize(x, mask=mask)
    assert np.array_equal(cg, codes) and np.array_equal(sg, scales) and gg == g
    # and so does the replay from the cache
    assert np.array_equal(oracle.quantize_cached(x, mask, scales, g), codes)


def test_record_split_over_threads_is_the_same():
    """Rows split across host threads own whole mask words (cols = 48: 2 rows per word boundary)."""
    x = synth.weight_f32(37, 48, 0.02, 9, 1)
    one = oracle.quantize_record(x, nthreads=1)
    many = oracle.quantize_record(x, nthreads=7)
    for a, b in zip(one, many):
        assert np.array_equal(np.asarray(a), np.asarray(b))


def test_cached_replay_of_updated_weights_brackets():
    """Cached scales and g applied to perturbed values: mask 0 gives the floor grid point of
    |x| / S and mask 1 the ceiling (exact grid points kept, 6 S and above saturating), and a mixed
    mask picks per element between those two."""
    x = synth.weight_f32(16, 128, 0.02, 11, 1)
    _, scales, g, rec = oracle.quantize_record(x)
    x2 = (x + synth.normal_f32(x.shape, 0.002, 11, 2)).astype(np.float32)  # one optimizer step later
    zeros, ones = np.zeros_like(rec), np.full_like(rec, 0xFFFFFFFF)
    lo = oracle.quantize_cached(x2, zeros, scales, g)
    hi = oracle.quantize_cached(x2, ones, scales, g)
    a = np.abs(x2.astype(np.float64))
    S = ex.dequant_torch(np.full((16, 64), 0x22, np.uint8), scales, g)  # code 2 is 1.0: dec(s) g
    dlo, dhi = np.abs(ex.dequant_torch(lo, scales, g)), np.abs(ex.dequant_torch(hi, scales, g))
    sat = a >= 6 * S
    grid = np.array(GRID)
    # floor: the largest grid point <= a; ceiling: the smallest grid point >= a (6 when saturated)
    fl = grid[np.searchsorted(grid, (a / S).clip(0, 6), side="right") - 1] * S
    ce = grid[np.minimum(np.searchsorted(grid, (a / S).clip(0, 6), side="left"), 7)] * S
    assert np.array_equal(dlo, np.where(sat, 6 * S, fl))
    assert np.array_equal(dhi, np.where(sat, 6 * S, ce))
    # signs follow x (also on zero codes)
    sg = (ex.unpack(lo) >> 3).reshape(x2.shape)
    assert np.array_equal(sg.astype(bool), np.signbit(x2))
    # a mixed mask: the record of the original weights
    mixed = oracle.quantize_cached(x2, rec, scales, g)
    bits = _bits(rec, x2.size).reshape(x2.shape).astype(bool)
    assert np.array_equal(ex.unpack(mixed).reshape(x2.shape),
                          np.where(bits, ex.unpack(hi).reshape(x2.shape), ex.unpack(lo).reshape(x2.shape)))


def test_cached_edge_cases():
    x = np.array([[1.0, -2.0] + [0.5] * 14], np.float32)
    mask = np.full(1, 0xFFFFFFFF, np.uint32)
    # g = 0 (or negative): every code is sign|0
    for g in (0.0, -1.0):
        c = ex.unpack(oracle.quantize_cached(x, mask, np.array([[0x38]], np.uint8), g)).reshape(-1)
        assert c[0] == 0 and c[1] == 8 and not (c & 7).any()
    # a byte above 0x7E reads as 0x7E (448)
    g = 2.0 ** -8
    c_hi = oracle.quantize_cached(x, mask, np.array([[0xFF]], np.uint8), g)
    c_7e = oracle.quantize_cached(x, mask, np.array([[0x7E]], np.uint8), g)
    assert np.array_equal(c_hi, c_7e)
    # byte 0x78 is 256, so S = 256 * 2^-8 = 1 exactly: 1.0, -2.0 and 0.5 are on the grid and
    # keep their codes whatever the mask
    c = ex.unpack(oracle.quantize_cached(x, mask, np.array([[0x78]], np.uint8), g)).reshape(-1)
    assert c[0] == 2 and c[1] == 8 | 4 and (c[2:] == 1).all()
