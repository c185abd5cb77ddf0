"""Pins of the oracle's FP4 KV cache and decode attention (CPU only).

TRACE summary, section "実験結果と性能": rollouts with FP4 weights, activations and KV cache. Each
cached K/V row is NVFP4-encoded with a given per-tensor g; decode attention reads the dequantized
rows, out = softmax(scale q K^T) V, query head h on KV head h // (Hq // Hkv). The pins compare with
torch's own attention in float64 on independently dequantized caches, and with closed forms.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from tests import _exact as ex


def _cache(B, Lmax, Hkv, D, seed, g=np.float32(0.004)):
    k = synth.activation_bf16(B * Lmax * Hkv, D, seed, 1).reshape(B, Lmax, Hkv, D)
    v = synth.activation_bf16(B * Lmax * Hkv, D, seed, 2).reshape(B, Lmax, Hkv, D)
    kc, ks = oracle.kv_quantize(k, g)
    vc, vs = oracle.kv_quantize(v, g)
    return kc, ks, vc, vs


def _deq(codes, scales, g):
    """[B, L, H, D] dequantized through torch's E4M3 decoding (tests/_exact.py); g an fp32 value."""
    B, L, H, D2 = codes.shape
    return ex.dequant_torch(codes.reshape(-1, D2), scales.reshape(-1, D2 // 8), np.float32(g)).reshape(B, L, H, 2 * D2)


def test_kv_quantize_is_the_nvfp4_encoding():
    x = synth.activation_bf16(40, 128, 3, 1)
    a = oracle.amax(x)
    g = oracle.global_scale(a)
    c, s = oracle.kv_quantize(x.reshape(5, 8, 128), g)
    c2, s2, g2 = oracle.quantize(x)
    assert g2 == g and np.array_equal(c.reshape(40, 64), c2) and np.array_equal(s.reshape(40, 8), s2)


@pytest.mark.parametrize("B,Hq,Hkv,D,Lmax", [(2, 4, 2, 64, 9), (3, 7, 1, 128, 17), (1, 28, 4, 128, 33)])
def test_matches_torch_sdpa_in_float64(B, Hq, Hkv, D, Lmax):
    g = np.float32(0.004)  # the per-tensor scale is an fp32 value
    kc, ks, vc, vs = _cache(B, Lmax, Hkv, D, B * Hq)
    q = synth.activation_bf16(B * Hq, D, B * Hq, 3).reshape(B, Hq, D)
    lens = np.random.default_rng(B).integers(1, Lmax + 1, B).astype(np.int32)
    scale = 1.0 / np.sqrt(D)
    got = oracle.attention_decode(q, kc, ks, g, vc, vs, g, lens, scale)
    K, V = _deq(kc, ks, g), _deq(vc, vs, g)
    qd = torch.from_numpy(synth.bf16_to_f32(q).astype(np.float64))
    for b in range(B):
        L = int(lens[b])
        kb = torch.from_numpy(K[b, :L]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)  # [Hq, L, D]
        vb = torch.from_numpy(V[b, :L]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
        ref = F.scaled_dot_product_attention(qd[b][:, None, :], kb, vb, scale=scale)[:, 0, :].numpy()
        assert np.allclose(got[b], ref, rtol=1e-12, atol=1e-14), f"sequence {b}"


def test_one_token_returns_its_value_row():
    B, Hq, Hkv, D, Lmax = 2, 6, 3, 32, 4
    g = np.float32(0.01)
    kc, ks, vc, vs = _cache(B, Lmax, Hkv, D, 7, g)
    q = synth.activation_bf16(B * Hq, D, 7, 3).reshape(B, Hq, D)
    out = oracle.attention_decode(q, kc, ks, g, vc, vs, g, np.ones(B, np.int32), 0.2)
    V = _deq(vc, vs, g)
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(out[b, h], V[b, 0, h // 2])


def test_zero_query_averages_the_values():
    B, Hq, Hkv, D, Lmax = 1, 2, 1, 16, 6
    g = np.float32(0.01)
    kc, ks, vc, vs = _cache(B, Lmax, Hkv, D, 8, g)
    q = np.zeros((B, Hq, D), np.uint16)
    out = oracle.attention_decode(q, kc, ks, g, vc, vs, g, np.array([5], np.int32), 1.0)
    V = _deq(vc, vs, g)
    assert np.allclose(out[0, 0], V[0, :5, 0].mean(axis=0), rtol=1e-14, atol=1e-15)
    assert np.array_equal(out[0, 0], out[0, 1])


def test_rows_beyond_the_length_are_not_read():
    B, Hq, Hkv, D, Lmax = 2, 4, 2, 32, 8
    g = np.float32(0.01)
    kc, ks, vc, vs = _cache(B, Lmax, Hkv, D, 9, g)
    q = synth.activation_bf16(B * Hq, D, 9, 3).reshape(B, Hq, D)
    lens = np.array([3, 8], np.int32)
    a = oracle.attention_decode(q, kc, ks, g, vc, vs, g, lens, 0.3)
    kc2, vc2, ks2 = kc.copy(), vc.copy(), ks.copy()
    kc2[0, 3:] = 0x77
    vc2[0, 3:] = 0x11
    ks2[0, 3:] = 0x7E
    b = oracle.attention_decode(q, kc2, ks2, g, vc2, vs, g, lens, 0.3)
    assert np.array_equal(a, b)


def test_scale_and_per_tensor_scales_enter_as_stated():
    B, Hq, Hkv, D, Lmax = 1, 2, 2, 32, 5
    kc, ks, vc, vs = _cache(B, Lmax, Hkv, D, 10, 1.0)
    q = synth.activation_bf16(B * Hq, D, 10, 3).reshape(B, Hq, D)
    lens = np.array([5], np.int32)
    # doubling g_k is doubling the softmax scale; doubling g_v doubles the output
    a = oracle.attention_decode(q, kc, ks, 2.0, vc, vs, 1.0, lens, 0.05)
    b = oracle.attention_decode(q, kc, ks, 1.0, vc, vs, 1.0, lens, 0.1)
    assert np.allclose(a, b, rtol=1e-13)
    c = oracle.attention_decode(q, kc, ks, 1.0, vc, vs, 2.0, lens, 0.1)
    assert np.array_equal(c, 2 * b)
