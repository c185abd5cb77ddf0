"""The pins catch plausible mistakes in the oracle.

Each mutant is a copy of the oracle source with one planted mistake (a flipped
tie rule, a dropped sign, a missing factor, a swapped nibble, a transposed
index, ...), compiled to a temporary library on the CPU. A compact battery of
the same pins the other oracle tests use must fail for every mutant and pass
for the unmodified source.
"""
import os
import tempfile

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from tests import _exact as ex

SRC = os.path.join(os.path.dirname(oracle.__file__), "nvfp4_oracle.cpp")

MUTANTS = {
    "e4m3_tie_to_odd": ("return (b & 1) ? b + 1 : b;", "return (b & 1) ? b : b + 1;"),
    "e2m1_tie_down": ("if (a == t) return sign | ((k & 1) ? k + 1 : k);", "if (a == t) return sign | k;"),
    "e2m1_sign_dropped": ("  const int sign = std::signbit(x) ? 8 : 0;\n  if (S == 0.0) return sign;\n  const double a = std::fabs(x);\n  for",
                          "  const int sign = 0;\n  if (S == 0.0) return sign;\n  const double a = std::fabs(x);\n  for"),
    "scale_without_6": ("e4m3_encode_ratio(bamax, 6.0 * static_cast<double>(g))", "e4m3_encode_ratio(bamax, static_cast<double>(g))"),
    "g_over_448": ("return amax / 2688.0f;", "return amax / 448.0f;"),
    "nibbles_swapped": ("if ((idx & 1) == 0) byte", "if ((idx & 1) == 1) byte"),
    "e4m3_subnormal_exponent": ("std::ldexp(m / 8.0, -6)", "std::ldexp(m / 8.0, -7)"),
    "e4m3_saturates_to_nan": ("if (num >= 448.0 * den) return 0x7E;", "if (num >= 448.0 * den) return 0x7F;"),
    "guided_polarity": ("return sign | (up ? k + 1 : k);", "return sign | (up ? k : k + 1);"),
    "guided_exact_hit_dropped": ("if (a == kGrid[k] * S) return sign | k;\n", ""),
    "rms_sum_not_mean": ("ss / static_cast<double>(H)", "ss"),
    "rms_noise_dropped": ("(static_cast<double>(w[j]) + z)", "static_cast<double>(w[j])"),
    "rms_delta_dropped": ("+ static_cast<double>(delta))", ")"),
    "lora_scale_dropped": ("Y[m * N + n] = acc + s * lora;", "Y[m * N + n] = acc + lora;"),
    "lora_sign_flipped": ("Y[m * N + n] = acc + s * lora;", "Y[m * N + n] = acc - s * lora;"),
    "lora_B_transposed": ("U[m * r + j] * bf16_value(B[n * r + j])", "U[m * r + j] * bf16_value(B[(j * 5 + n) % 10])"),
    "dequant_block_index": ("scales[n * (K / 16) + k / 16]", "scales[n * (K / 16) + (k / 16 + 1) % (K / 16)]"),
    "gemm_operand_transposed": ("acc += xq[m * K + k] * wrow[k];", "acc += xq[m * K + k] * wrow[K - 1 - k];"),
    "record_bit_inverted": ("return kGrid[c & 7] * S > std::fabs(x) ? 1 : 0;", "return kGrid[c & 7] * S > std::fabs(x) ? 0 : 1;"),
    "record_grid_points_up": ("return kGrid[c & 7] * S > std::fabs(x) ? 1 : 0;", "return kGrid[c & 7] * S >= std::fabs(x) ? 1 : 0;"),
    "cached_scale_of_next_block": ("scales[r * nblk + b] > 0x7E ? 0x7E : scales[r * nblk + b]",
                                   "scales[r * nblk + (b + 1) % nblk] > 0x7E ? 0x7E : scales[r * nblk + (b + 1) % nblk]"),
    "cached_g_dropped": ("(g > 0.0f) ? e4m3_value(s) * static_cast<double>(g) : 0.0", "(g > 0.0f) ? e4m3_value(s) : 0.0"),
    "ais_ess_without_sqrt": ("const double a_ess = 1.0 / std::sqrt(1.0 + cv2);", "const double a_ess = 1.0 / (1.0 + cv2);"),
    "ais_signed_mismatch": ("sum_d += std::fabs(d);", "sum_d += d;"),
    "ais_ratio_inverted": ("static_cast<double>(logp_train[i]) - static_cast<double>(logp_rollout[i])",
                           "static_cast<double>(logp_rollout[i]) - static_cast<double>(logp_train[i])"),
    "ais_no_truncation": ("w[i] = std::fmin(std::exp(d), C);", "w[i] = std::exp(d);"),
    "ais_no_clip": ("std::fmin(1.0, std::fmax(0.0, a_ess - beta * a_var)) * a_mis", "(a_ess - beta * a_var) * a_mis"),
    "ais_mis_unsaturated": ("const double a_mis = std::fmin(1.0, dbar / delta);", "const double a_mis = dbar / delta;"),
    "ais_dsigma_raw_ratio": ("std::sqrt(vwa) / std::sqrt(va) - 1.0", "std::sqrt(vwa) / std::sqrt(va)"),
    "ais_rectified_weight": ("w_out[i] = 1.0 + alpha * (w[i] - 1.0);", "w_out[i] = alpha * w[i];"),
    "attn_gqa_modulo": ("const int64_t kvh = h / group, L = lens[b];", "const int64_t kvh = h % Hkv, L = lens[b];"),
    "attn_scale_dropped": ("sc[t] = scale * dot;", "sc[t] = dot;"),
    "attn_length_off_by_one": ("for (int64_t t = 0; t < L; ++t) acc += sc[t]", "for (int64_t t = 1; t < L; ++t) acc += sc[t]"),
    "attn_v_with_k_scales": ("acc += sc[t] * deq(vc, vs, gv,", "acc += sc[t] * deq(vc, ks, gv,"),
    "attn_unnormalised": ("out[(b * Hq + h) * D + d] = acc / den;", "out[(b * Hq + h) * D + d] = acc;"),
    "cached_mask_shifted": ("        const int up = (mask[idx / 32] >> (idx % 32)) & 1;\n        const int c = e2m1_encode_guided(load_elem",
                            "        const int up = (mask[idx / 32] >> ((idx + 1) % 32)) & 1;\n        const int c = e2m1_encode_guided(load_elem"),
}


def _battery(L):
    """Returns the names of the checks that fail for library L."""
    fails = []

    def check(name, fn):
        try:
            ok = fn()
        except AssertionError:
            ok = False
        if not ok:
            fails.append(name)

    # worked examples and exhaustive search on small blocks (plain + guided)
    import json
    with open(os.path.join(os.path.dirname(__file__), "golden", "nvfp4_worked_examples.json")) as f:
        golden = json.load(f)["examples"]

    def worked():
        for case in golden:
            v = np.array([np.float32(s) for s in case["values"]], np.float32).reshape(1, -1)
            c, s, g = oracle.quantize(v, L=L)
            if float(g) != float(case["g"]) or s.reshape(-1).tolist() != case["scales"]:
                return False
            if ex.unpack(c).reshape(-1).tolist() != case["codes_f32"]:
                return False
        return True
    check("worked", worked)

    def exhaustive(mask=False):
        rng = np.random.default_rng(0)
        w = (rng.standard_normal((3, 64)) * np.exp(rng.uniform(-3, 3, (3, 1)))).astype(np.float32)
        w[0, :16] *= 1e-3
        w[1, 5] = 0.0
        w[2, 7] = -0.0
        m = synth.guided_mask(w.size, 3) if mask else None
        c, s, g = oracle.quantize(w, mask=m, L=L)
        if g != ex.global_scale(np.abs(w).max()):
            return False
        bits = np.unpackbits(m.view(np.uint8), bitorder="little")[: w.size].reshape(w.shape) if mask else None
        got = ex.unpack(c)
        for r in range(3):
            for b in range(4):
                sb, cb = ex.quantize_block(w[r, 16 * b:16 * b + 16], g, None if bits is None else bits[r, 16 * b:16 * b + 16])
                if s[r, b] != sb or got[r, 16 * b:16 * b + 16].tolist() != cb:
                    return False
        return True
    check("exhaustive", exhaustive)
    check("exhaustive_guided", lambda: exhaustive(True))

    def e4m3_values():
        ref = torch.arange(127, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        return all(oracle.e4m3_value(b, L) == ref[b] for b in range(127))
    check("e4m3_values", e4m3_values)

    def e4m3_ties():
        vals = [oracle.e4m3_value(b, L) for b in range(127)]
        return all(oracle.e4m3_encode_ratio(0.5 * (vals[b] + vals[b + 1]), 1.0, L) == (b if b % 2 == 0 else b + 1)
                   for b in range(126))
    check("e4m3_ties", e4m3_ties)

    def saturation():
        return oracle.e4m3_encode_ratio(470.0, 1.0, L) == 0x7E
    check("saturation", saturation)

    def guided_exact():
        return all(oracle.e2m1_encode_guided(float(ex.GRID[k]), 1.0, 1, L) == k for k in range(8))
    check("guided_exact", guided_exact)

    def rmsnorm():
        x = synth.activation_bf16(4, 128, 0, 1)
        w = synth.aqn_weight(128, 0, 2)
        eps = synth.aqn_eps(128, 0, 3)
        y = oracle.rmsnorm_aqn(x, w, eps, 0.01, 1e-2, L=L)
        wn = w.astype(np.float64) + 0.01 * eps.astype(np.float64)
        xt = torch.from_numpy(synth.bf16_to_f32(x).astype(np.float64))
        ref = F.rms_norm(xt, (128,), weight=torch.from_numpy(wn),
                         eps=float(np.float32(1e-2))).numpy()
        return np.allclose(y, ref, rtol=1e-6, atol=1e-9)
    check("rmsnorm", rmsnorm)

    def record_hand():
        from tests.test_oracle_trace import HAND_ROWS, HAND_UP
        _, _, _, m = oracle.quantize_record(np.array(HAND_ROWS, np.float32), amax_in=2688.0, L=L)
        return np.unpackbits(m.view(np.uint8), bitorder="little")[:32].tolist() == HAND_UP
    check("record_hand", record_hand)

    def record_exact():
        x = synth.weight_f32(8, 64, 0.02, 3, 7, outlier_frac=0.05)
        c, s, g, m = oracle.quantize_record(x, L=L)
        up = np.abs(ex.dequant_torch(c, s, g)) > np.abs(x.astype(np.float64))
        return np.array_equal(np.unpackbits(m.view(np.uint8), bitorder="little")[: x.size].astype(bool),
                              up.reshape(-1))
    check("record_exact", record_exact)

    def cached_roundtrip():
        x = synth.weight_f32(6, 64, 0.02, 4, 7, outlier_frac=0.05)
        c, s, g, m = oracle.quantize_record(x, L=L)
        return np.array_equal(oracle.quantize_cached(x, m, s, g, L=L), c)
    check("cached_roundtrip", cached_roundtrip)

    def ais_cases():
        from tests import test_oracle_ais as T
        cases = [T.test_no_mismatch_is_vanilla_grpo, T.test_two_valued_weights_closed_form,
                 T.test_truncation_and_saturation, T.test_penalty_clips_at_zero,
                 lambda: T.test_variance_penalty_closed_form(3.0, 0.5, 0.25)]
        real = oracle.ais
        oracle.ais = lambda *a, **k: real(*a, **{**k, "L": L})
        try:
            for c in cases:
                c()
        finally:
            oracle.ais = real
        return True
    check("ais", ais_cases)

    def attention():
        from tests import test_oracle_attention as T
        real_a, real_q = oracle.attention_decode, oracle.kv_quantize
        oracle.attention_decode = lambda *a, **k: real_a(*a, **{**k, "L": L})
        oracle.kv_quantize = lambda *a, **k: real_q(*a, **{**k, "L": L})
        try:
            T.test_matches_torch_sdpa_in_float64(2, 4, 2, 64, 9)
            T.test_one_token_returns_its_value_row()
            T.test_scale_and_per_tensor_scales_enter_as_stated()
        finally:
            oracle.attention_decode, oracle.kv_quantize = real_a, real_q
        return True
    check("attention", attention)

    def linear():
        N, K, M, r = 5, 64, 3, 2
        W = synth.weight_f32(N, K, 0.02, 1, 5, outlier_frac=0.05)
        c, s, g = oracle.quantize(W, L=L)
        x = synth.activation_bf16(M, K, 2, 1)
        A, B = synth.lora_factors(r, K, N, 2, 9)
        xd = synth.bf16_to_f32(x).astype(np.float64)
        Ad, Bd = synth.bf16_to_f32(A).astype(np.float64), synth.bf16_to_f32(B).astype(np.float64)
        ref = xd @ ex.dequant_torch(c, s, g).T + 2.0 * (xd @ Ad.T) @ Bd.T
        got = oracle.lora_linear_w4a16(x, c, s, g, A, B, 2.0, L=L)
        return np.allclose(got, ref, rtol=1e-10, atol=1e-12)
    check("linear", linear)
    return fails


def _compile(text, tmp, name):
    src = os.path.join(tmp, name + ".cpp")
    with open(src, "w") as f:
        f.write(text)
    return oracle.lib(oracle.build(force=True, src=src, out=os.path.join(tmp, "lib" + name + ".so")))


def test_unmodified_oracle_passes_the_battery():
    assert _battery(oracle.lib()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    text = open(SRC).read()
    old, new = MUTANTS[name]
    assert text.count(old) >= 1, f"mutation site for {name} not found"
    mutated = text.replace(old, new, 1)
    with tempfile.TemporaryDirectory() as tmp:
        L = _compile(mutated, tmp, name)
        assert _battery(L) != [], f"planted mistake {name} went unnoticed"
