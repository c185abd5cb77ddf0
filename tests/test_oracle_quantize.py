"""Pins for the oracle's NVFP4 tensor quantization (plain and guided).

Hand-worked examples (tests/golden), an exhaustive exact-rational search on
small tensors, and invariants the definition fixes: exactness on
representable values, power-of-two scaling, sign symmetry, guided rounding
with the plain rounding's own decisions, the all-zero tensor.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from tests import _exact as ex

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_worked_examples.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)["examples"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", _golden(), ids=lambda c: c["name"])
def test_worked_examples(case, dtype):
    v = np.array([np.float32(s) for s in case["values"]], np.float32)
    x = v.reshape(1, -1) if dtype == "f32" else synth.bf16_bits(v).reshape(1, -1)
    codes, scales, g = oracle.quantize(x)
    assert float(g) == float(case["g"])
    assert scales.reshape(-1).tolist() == case["scales"]
    assert ex.unpack(codes).reshape(-1).tolist() == case["codes_" + dtype]


def test_global_scale_is_correctly_rounded():
    rng = np.random.default_rng(5)
    for a in np.exp(rng.uniform(np.log(1e-30), np.log(1e30), 2000)).astype(np.float32):
        assert oracle.global_scale(a) == ex.global_scale(a)
    assert oracle.global_scale(np.float32(2688.0)) == 1.0 and oracle.global_scale(np.float32(0.0)) == 0.0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_quantize_matches_exhaustive_search(dtype, seed):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((3, 64)) * np.exp(rng.uniform(-3, 3, (3, 1)))).astype(np.float32)
    w[0, :16] *= 1e-3  # a block far below the tensor amax (small scale bytes)
    x = w if dtype == "f32" else synth.bf16_bits(w)
    codes, scales, g = oracle.quantize(x)
    xv = w if dtype == "f32" else synth.bf16_to_f32(x)
    assert g == ex.global_scale(np.abs(xv).max())
    got = ex.unpack(codes)
    for r in range(3):
        for b in range(4):
            s, c = ex.quantize_block(xv[r, 16 * b:16 * b + 16], g)
            assert scales[r, b] == s
            assert got[r, 16 * b:16 * b + 16].tolist() == c


def test_guided_matches_exhaustive_search():
    rng = np.random.default_rng(7)
    w = rng.standard_normal((2, 64)).astype(np.float32)
    mask = synth.guided_mask(w.size, 3)
    codes, scales, g = oracle.quantize(w, mask=mask)
    bits = np.unpackbits(mask.view(np.uint8), bitorder="little")[: w.size].reshape(w.shape)
    got = ex.unpack(codes)
    for r in range(2):
        for b in range(4):
            s, c = ex.quantize_block(w[r, 16 * b:16 * b + 16], g, bits[r, 16 * b:16 * b + 16])
            assert scales[r, b] == s
            assert got[r, 16 * b:16 * b + 16].tolist() == c


def test_exact_on_representable_values():
    rng = np.random.default_rng(8)
    rows, cols = 4, 128
    g = np.float32(3.0 / 256)  # few significant bits: code * dec(s) * g is exact in fp32
    codes = rng.integers(0, 16, (rows, cols)).astype(np.uint8)
    scales = rng.integers(1, 127, (rows, cols // 16)).astype(np.uint8)
    # make every block hold its largest magnitude 6 once, and one block the scale 448,
    # so that the recovered block amax and tensor amax reproduce scales and g
    for r in range(rows):
        for b in range(cols // 16):
            codes[r, 16 * b + (r + b) % 16] = 7 | (codes[r, 16 * b] & 8)
    scales[0, 0] = 0x7E
    x = ex.dequant_torch(ex.pack(codes), scales, g).astype(np.float32)
    assert np.array_equal(x.astype(np.float64), ex.dequant_torch(ex.pack(codes), scales, g))  # exact in fp32
    c2, s2, g2 = oracle.quantize(x)
    assert g2 == ex.global_scale(np.abs(x).max())
    assert np.array_equal(s2, scales)
    assert g2 == g and np.array_equal(c2, ex.pack(codes))


@pytest.mark.parametrize("k", [-7, -1, 3, 12])
def test_power_of_two_scaling(k):
    x = synth.weight_f32(16, 256, 0.02, 0, 99, outlier_frac=0.02)
    c1, s1, g1 = oracle.quantize(x)
    c2, s2, g2 = oracle.quantize((x * np.float32(2.0 ** k)).astype(np.float32))
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)
    assert float(g2) == float(g1) * 2.0 ** k


def test_negation_flips_sign_bits_only():
    x = synth.weight_f32(16, 256, 0.02, 0, 98)
    c1, s1, g1 = oracle.quantize(x)
    c2, s2, g2 = oracle.quantize(-x)
    assert g1 == g2 and np.array_equal(s1, s2)
    assert np.array_equal(c2, c1 ^ 0x88)


def test_guided_with_plain_decisions_equals_plain():
    x = synth.weight_f32(32, 512, 0.02, 0, 97, outlier_frac=0.01)
    c, s, g = oracle.quantize(x)
    # the plain rounding went up (away from zero) wherever its magnitude exceeds the floor neighbour
    deq = ex.dequant_torch(c, s, g)
    up = (np.abs(deq) > np.abs(x.astype(np.float64))).reshape(-1)
    mask = np.packbits(up.astype(np.uint8), bitorder="little").view(np.uint32)
    cg, sg, gg = oracle.quantize(x, mask=mask)
    assert np.array_equal(cg, c) and np.array_equal(sg, s) and gg == g
    # an all-zero / all-one mask gives the floor / ceiling neighbour everywhere
    lo, _, _ = oracle.quantize(x, mask=np.zeros_like(mask))
    hi, _, _ = oracle.quantize(x, mask=np.full_like(mask, 0xFFFFFFFF))
    a = np.abs(x.astype(np.float64))
    dlo, dhi = np.abs(ex.dequant_torch(lo, s, g)), np.abs(ex.dequant_torch(hi, s, g))
    S = ex.dequant_torch(np.full_like(c, 0x22), s, g)  # code 2 is 1.0, so this is dec(s) * g per element
    sat = a >= 6 * S
    assert ((dlo <= a) | sat).all() and ((dhi >= a) | sat).all()
    step = (ex.unpack(hi).astype(int) & 7) - (ex.unpack(lo).astype(int) & 7)
    assert ((step == 0) | (step == 1)).all()


def test_zero_tensor():
    x = np.zeros((4, 32), np.float32)
    x[1, 3] = -0.0
    c, s, g = oracle.quantize(x)
    assert g == 0 and not s.any()
    u = ex.unpack(c)
    assert u[1, 3] == 8 and (np.delete(u.reshape(-1), 1 * 32 + 3) == 0).all()


def test_dequantize_matches_torch_decode():
    x = synth.weight_f32(8, 128, 0.02, 0, 96, outlier_frac=0.05)
    c, s, g = oracle.quantize(x)
    assert np.array_equal(oracle.dequantize(c, s, g), ex.dequant_torch(c, s, g))


def test_amax_override():
    x = synth.weight_f32(8, 64, 0.02, 0, 95)
    c1, s1, g1 = oracle.quantize(x)
    c2, s2, g2 = oracle.quantize(x, amax_in=float(np.abs(x).max()))
    assert g1 == g2 and np.array_equal(c1, c2) and np.array_equal(s1, s2)
    # a smaller amax saturates scale bytes at 0x7E
    _, s3, _ = oracle.quantize(x, amax_in=float(np.abs(x).max()) / 4)
    assert s3.max() == 0x7E
