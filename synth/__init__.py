"""Seeded synthetic inputs for the NVFP4 rollout linear layer.

This module is the one thing the CUDA path and the CPU oracle share: it draws
the inputs (weights, activations, LoRA factors, AQN noise draws, guided
rounding masks, MoE routing) and nothing else. It holds none of the method's
arithmetic: no quantization, no normalisation, no GEMM.

Shapes and distributions follow the workloads the QeRL explainer and the TRACE
summary talk about (Qwen2.5 dense models, a 128-expert MoE); the pages print no
tensors, so every value here is synthetic and seeded.

All arrays are numpy. bf16 tensors are returned as uint16 bit patterns, rounded
to nearest-even from float32 (the usual bf16 cast).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "rng", "bf16_bits", "bf16_to_f32", "normal_f32", "normal_bf16", "weight_bf16",
    "weight_f32", "activation_bf16", "heavy_tail_activation_bf16", "lora_factors",
    "aqn_weight", "aqn_eps", "guided_mask", "moe_routing", "grpo_token_batch", "QWEN25_7B", "QWEN25_32B",
    "MOE", "GRPO_BATCH", "tiny_config",
]


def rng(seed: int, *stream: int) -> np.random.Generator:
    """A PCG64 generator keyed by (seed, stream ids): one independent stream per tensor."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed)] + [int(s) for s in stream])))


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even. Inputs must be finite."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_f32(shape, std: float, seed: int, *stream: int) -> np.ndarray:
    return (rng(seed, *stream).standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def normal_bf16(shape, std: float, seed: int, *stream: int) -> np.ndarray:
    return bf16_bits(normal_f32(shape, std, seed, *stream))


def _outlier_columns(cols: int, frac: float, seed: int, *stream: int) -> np.ndarray:
    n = int(round(frac * cols))
    return np.sort(rng(seed, *stream, 7).choice(cols, size=n, replace=False))


def weight_f32(rows: int, cols: int, std: float, seed: int, *stream: int,
               outlier_frac: float = 0.0, outlier_gain: float = 8.0) -> np.ndarray:
    """W ~ N(0, std^2), with a seeded set of round(frac*cols) columns multiplied by `outlier_gain`."""
    w = normal_f32((rows, cols), std, seed, *stream)
    if outlier_frac > 0:
        w[:, _outlier_columns(cols, outlier_frac, seed, *stream)] *= np.float32(outlier_gain)
    return w


def weight_bf16(rows: int, cols: int, std: float, seed: int, *stream: int,
                outlier_frac: float = 0.0, outlier_gain: float = 8.0) -> np.ndarray:
    return bf16_bits(weight_f32(rows, cols, std, seed, *stream,
                                outlier_frac=outlier_frac, outlier_gain=outlier_gain))


def activation_bf16(rows: int, cols: int, seed: int, *stream: int, std: float = 1.0) -> np.ndarray:
    return normal_bf16((rows, cols), std, seed, *stream)


def heavy_tail_activation_bf16(rows: int, cols: int, seed: int, *stream: int,
                               frac: float = 0.01, nu: int = 4) -> np.ndarray:
    """x ~ N(0,1) with round(frac*cols) seeded channels drawn from Student-t(nu) = Z / sqrt(chi2_nu / nu)."""
    x = normal_f32((rows, cols), 1.0, seed, *stream)
    ch = _outlier_columns(cols, frac, seed, *stream)
    if len(ch):
        g = rng(seed, *stream, 11)
        z = g.standard_normal(size=(rows, len(ch)))
        chi2 = g.chisquare(nu, size=(rows, len(ch)))
        x[:, ch] = (z / np.sqrt(chi2 / nu)).astype(np.float32)
    return bf16_bits(x)


def lora_factors(r: int, k: int, n: int, seed: int, *stream: int, std: float = 0.02):
    """LoRA A [r, k] and B [n, r], both ~N(0, std^2), bf16 bits."""
    return normal_bf16((r, k), std, seed, *stream, 1), normal_bf16((n, r), std, seed, *stream, 2)


def aqn_weight(h: int, seed: int, *stream: int, std: float = 0.1) -> np.ndarray:
    """RMSNorm weight w = 1 + N(0, std^2), fp32."""
    return (np.float32(1.0) + normal_f32((h,), std, seed, *stream)).astype(np.float32)


def aqn_eps(h: int, seed: int, *stream: int) -> np.ndarray:
    """Standard-normal draws for the AQN noise vector (the noise is sigma_k times these), fp32."""
    return normal_f32((h,), 1.0, seed, *stream)


def guided_mask(n_elements: int, seed: int, *stream: int) -> np.ndarray:
    """Bernoulli(1/2) rounding-direction bits: bit (i % 32) of word i // 32, as uint32 words."""
    words = (n_elements + 31) // 32
    return rng(seed, *stream).integers(0, 2**32, size=words, dtype=np.uint64).astype(np.uint32)


def moe_routing(tokens: int, experts: int, top_k: int, seed: int, *stream: int):
    """Synthetic top-k routing from N(0,1) router logits.

    Softmax is monotone, so the top-k of softmax(logits) is the top-k of the logits;
    ties go to the lower expert index. Returns (token_of_row, offsets): routed rows
    sorted stably by expert, `token_of_row[i]` the source token of row i, and
    int32 offsets[experts+1] with expert e owning rows [offsets[e], offsets[e+1]).
    """
    logits = rng(seed, *stream).standard_normal(size=(tokens, experts))
    order = np.argsort(-logits, axis=1, kind="stable")[:, :top_k]
    expert_of = order.reshape(-1)
    token_of = np.repeat(np.arange(tokens), top_k)
    perm = np.argsort(expert_of, kind="stable")
    counts = np.bincount(expert_of, minlength=experts)
    offsets = np.zeros(experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return token_of[perm].astype(np.int64), offsets


def grpo_token_batch(prompts: int, group: int, mean_len: int, seed: int, *stream: int, mismatch: float = 0.05,
                     max_tokens: int | None = None):
    """A GRPO training batch flattened to tokens: `prompts` prompts x `group` responses whose lengths
    are log-normal around mean_len (16 .. 4 mean_len); per response a Bernoulli reward (success rate
    uniform per prompt), normalised within its group, (r - mean) / (std + 1e-6), and broadcast to its
    tokens as the advantage; per token the rollout log-prob of the sampled token, -Exponential(0.4)
    (mostly confident tokens), and the training log-prob, that plus N(0, mismatch) noise capped at 0
    (the low-precision rollout's mismatch). Returns fp32 (logp_rollout, logp_train, adv), optionally
    cut to max_tokens."""
    g = rng(seed, *stream)
    n_resp = prompts * group
    lens = np.clip(np.rint(g.lognormal(np.log(mean_len) - 0.18, 0.6, n_resp)), 16, 4 * mean_len).astype(np.int64)
    p = np.repeat(g.uniform(0, 1, prompts), group)
    r = (g.uniform(0, 1, n_resp) < p).astype(np.float64).reshape(prompts, group)
    a = ((r - r.mean(axis=1, keepdims=True)) / (r.std(axis=1, keepdims=True) + 1e-6)).reshape(-1)
    adv = np.repeat(a, lens).astype(np.float32)
    n = adv.size
    lr = (-g.exponential(0.4, n)).astype(np.float32)
    lt = np.minimum(lr + g.normal(0.0, mismatch, n), 0.0).astype(np.float32)
    if max_tokens is not None:
        lr, lt, adv = lr[:max_tokens], lt[:max_tokens], adv[:max_tokens]
    return lr, lt, adv


# A GRPO batch of 64 prompts x 8 responses of ~8K tokens (about 4 M tokens; at most 4 Mi are kept).
GRPO_BATCH = {"prompts": 64, "group": 8, "mean_len": 8192, "tokens": 4 * 1024 * 1024}


# Model shapes (out_features, in_features) of one decoder layer's linears.
QWEN25_7B = {
    "hidden": 3584,
    "linears": {"q": (3584, 3584), "o": (3584, 3584), "gate": (18944, 3584),
                "up": (18944, 3584), "down": (3584, 18944)},
}
QWEN25_32B = {
    "hidden": 5120,
    "linears": {"q": (5120, 5120), "k": (1024, 5120), "v": (1024, 5120), "o": (5120, 5120),
                "gate": (27648, 5120), "up": (27648, 5120), "down": (5120, 27648)},
}
MOE = {"experts": 128, "hidden": 2048, "intermediate": 768, "tokens": 4096, "top_k": 8,
       "layers": 48, "guided_layers": list(range(36, 48))}


def tiny_config(seed: int = 0):
    """The tiny end-to-end case: W fp32 256x512 ~N(0,0.02); x bf16 8x512 ~N(0,1);
    RMSNorm w = 1+N(0,0.1), AQN sigma 0.01, delta 1e-6; LoRA r=16, A,B ~N(0,0.02), s=2."""
    return {
        "W": weight_f32(256, 512, 0.02, seed, 1),
        "x": activation_bf16(8, 512, seed, 2),
        "w": aqn_weight(512, seed, 3),
        "eps": aqn_eps(512, seed, 4),
        "sigma": 0.01, "delta": 1e-6,
        "A": normal_bf16((16, 512), 0.02, seed, 5),
        "B": normal_bf16((256, 16), 0.02, seed, 6),
        "r": 16, "s": 2.0,
    }
