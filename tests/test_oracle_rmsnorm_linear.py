"""Pins for the oracle's AQN RMSNorm, noise schedule and LoRA linear layers.

AQN RMSNorm (QeRL explainer, section "ゼロオーバーヘッド"): with no noise it is
torch's rms_norm; noise enters only through the weight (w + z); a constant row
has a closed form. The schedule (section "AQNの仕組み") has fixed endpoints and a
constant ratio. The linear layers are pinned to numpy matmuls of torch-decoded
weights, to an exact-rational brute force on tiny shapes, and to the special
cases B = 0, s = 0, zero codes, on-grid activations and per-expert groups.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from tests import _exact as ex


def _x(M, H, seed):
    return synth.activation_bf16(M, H, seed, 1)


def test_rmsnorm_without_noise_is_torch_rms_norm():
    x = _x(16, 384, 0)
    w = synth.aqn_weight(384, 0, 2)
    y = oracle.rmsnorm_aqn(x, w, None, 0.0, 1e-6)
    xt = torch.from_numpy(synth.bf16_to_f32(x).astype(np.float64))
    ref = F.rms_norm(xt, (384,), weight=torch.from_numpy(w.astype(np.float64)), eps=float(np.float32(1e-6))).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-15)
    # a zero noise vector is the same as no noise
    y0 = oracle.rmsnorm_aqn(x, w, np.zeros(384, np.float32), 0.3, 1e-6)
    np.testing.assert_array_equal(y0, y)


def test_noise_enters_through_the_weight_only():
    x = _x(8, 256, 1)
    w = synth.aqn_weight(256, 1, 2)
    eps = synth.aqn_eps(256, 1, 3)
    sigma = np.float32(0.01)
    y = oracle.rmsnorm_aqn(x, w, eps, sigma, 1e-6)
    w_noisy = (w.astype(np.float64) + float(sigma) * eps.astype(np.float64))
    y_ref = F.rms_norm(torch.from_numpy(synth.bf16_to_f32(x).astype(np.float64)), (256,),
                       weight=torch.from_numpy(w_noisy), eps=float(np.float32(1e-6))).numpy()
    np.testing.assert_allclose(y, y_ref, rtol=1e-13, atol=1e-15)
    # channel-wise additive noise is a row-wise multiplicative change: y - y0 = z * x * r
    y0 = oracle.rmsnorm_aqn(x, w, None, 0.0, 1e-6)
    xd = synth.bf16_to_f32(x).astype(np.float64)
    r = 1.0 / np.sqrt((xd ** 2).mean(axis=1, keepdims=True) + float(np.float32(1e-6)))
    np.testing.assert_allclose(y - y0, float(sigma) * eps.astype(np.float64) * xd * r, rtol=1e-9, atol=1e-15)


def test_constant_row_closed_form():
    c, H, delta = 1.5, 64, 0.25
    x = synth.bf16_bits(np.full((1, H), c, np.float32))
    w = np.linspace(0.5, 2, H).astype(np.float32)
    y = oracle.rmsnorm_aqn(x, w, None, 0.0, delta)
    np.testing.assert_allclose(y[0], w.astype(np.float64) * c / np.sqrt(c * c + delta), rtol=1e-15)


def test_sigma_schedule():
    s0, sK, K = 1e-2, 5e-4, 10
    sig = [oracle.aqn_sigma(s0, sK, k, K) for k in range(K + 1)]
    assert sig[0] == s0 and abs(sig[K] - sK) <= 1e-18
    ratios = [sig[k + 1] / sig[k] for k in range(K)]
    np.testing.assert_allclose(ratios, (sK / s0) ** (1 / K), rtol=1e-13)
    assert all(a > b for a, b in zip(sig, sig[1:]))  # large noise early, small late


def _weights(N, K, seed, outliers=0.0):
    W = synth.weight_f32(N, K, 0.02, seed, 5, outlier_frac=outliers)
    return oracle.quantize(W)


def test_linear_without_lora_is_a_matmul_of_the_decoded_weight():
    N, K, M = 48, 96, 5  # N != K catches a transposed operand
    codes, scales, g = _weights(N, K, 1, 0.05)
    x = _x(M, K, 2)
    A, B = synth.lora_factors(8, K, N, 2, 9)
    xd = synth.bf16_to_f32(x).astype(np.float64)
    ref = xd @ ex.dequant_torch(codes, scales, g).T
    np.testing.assert_allclose(oracle.lora_linear_w4a16(x, codes, scales, g, A, np.zeros_like(B), 2.0), ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.lora_linear_w4a16(x, codes, scales, g, A, B, 0.0), ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.lora_linear_w4a16(x, codes, scales, g, None, None, 2.0), ref, rtol=1e-12, atol=1e-12)


def test_zero_codes_leave_only_the_lora_branch():
    N, K, M, r, s = 40, 64, 3, 4, 2.0
    codes = np.zeros((N, K // 2), np.uint8)
    scales = np.full((N, K // 16), 0x38, np.uint8)
    x = _x(M, K, 3)
    A, B = synth.lora_factors(r, K, N, 3, 9)
    xd = synth.bf16_to_f32(x).astype(np.float64)
    ref = s * (xd @ synth.bf16_to_f32(A).astype(np.float64).T) @ synth.bf16_to_f32(B).astype(np.float64).T
    np.testing.assert_allclose(oracle.lora_linear_w4a16(x, codes, scales, np.float32(0.01), A, B, s), ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("seed", [0, 1])
def test_linear_exact_rational_brute_force(seed):
    M, N, K, r, s = 3, 5, 32, 2, 2.0
    codes, scales, g = _weights(N, K, 10 + seed, 0.1)
    x = _x(M, K, 11 + seed)
    A, B = synth.lora_factors(r, K, N, 12 + seed, 9)
    Y = oracle.lora_linear_w4a16(x, codes, scales, g, A, B, s)
    c, sc = ex.unpack(codes), scales
    G = Fraction(float(g))
    xf = [[Fraction(float(v)) for v in row] for row in synth.bf16_to_f32(x)]
    Af = [[Fraction(float(v)) for v in row] for row in synth.bf16_to_f32(A)]
    Bf = [[Fraction(float(v)) for v in row] for row in synth.bf16_to_f32(B)]
    for m in range(M):
        U = [sum(xf[m][k] * Af[j][k] for k in range(K)) for j in range(r)]
        for n in range(N):
            base = 0
            for k in range(K):
                code = int(c[n, k])
                val = ex.GRID[code & 7] * (-1 if code & 8 else 1)
                base += xf[m][k] * val * ex.E4M3[int(sc[n, k // 16])] * G
            exact = base + Fraction(s) * sum(U[j] * Bf[n][j] for j in range(r))
            assert abs(Fraction(Y[m, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 45) + Fraction(1, 2 ** 80)


def test_w4a4_on_grid_activations_equals_w4a16():
    # activations that are NVFP4-representable (with their own amax) quantize losslessly
    N, K, M = 32, 64, 4
    codes, scales, g = _weights(N, K, 20)
    rng = np.random.default_rng(21)
    xc = rng.integers(0, 16, (M, K)).astype(np.uint8)
    xs = rng.integers(0x20, 0x70, (M, K // 16)).astype(np.uint8)
    xc[:, ::16] = 7          # every block reaches 6 * its scale ...
    xs[0, 0] = 0x7E          # ... and one block has scale 448, so amax / 2688 == gx exactly
    gx = np.float32(2.0 ** -10)
    x_f = ex.dequant_torch(ex.pack(xc), xs, gx)
    x_bits = synth.bf16_bits(x_f.astype(np.float32))
    assert np.array_equal(synth.bf16_to_f32(x_bits).astype(np.float64), x_f)  # exact in bf16
    A, B = synth.lora_factors(4, K, N, 22, 9)
    y4, (qc, qs, qg) = oracle.lora_linear_w4a4(x_bits, codes, scales, g, A, B, 2.0)
    y16 = oracle.lora_linear_w4a16(x_bits, codes, scales, g, A, B, 2.0)
    assert np.array_equal(oracle.dequantize(qc, qs, qg), x_f)
    np.testing.assert_allclose(y4, y16, rtol=1e-13, atol=1e-15)


def test_grouped_rows_equal_per_expert_dense():
    E, K, N = 4, 64, 32
    tok, off = synth.moe_routing(24, E, 2, 0, 1)
    assert off[-1] == 48 and (np.diff(off) >= 0).all()
    X = _x(48, K, 30)
    Ws = [_weights(N, K, 40 + e) for e in range(E)]
    full = np.concatenate([oracle.lora_linear_w4a16(X[off[e]:off[e + 1]], *Ws[e], None, None, 0.0)
                           for e in range(E)])
    for e in range(E):
        rows = np.arange(off[e], off[e + 1])
        if len(rows):
            part = oracle.lora_linear_w4a16(X, *Ws[e], None, None, 0.0, rows=rows)
            np.testing.assert_array_equal(part, full[off[e]:off[e + 1]])
