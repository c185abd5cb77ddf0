"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same seeded inputs.

Quantization (codes, scale bytes, g) is compared bit for bit; RMSNorm and the
GEMMs within the tolerances of tests/_parity.py. Inputs come from synth; every
expected value comes from the oracle. Sizes span several tiles with ragged
tails, plus the full workload shapes (the 7B decode layer the benchmark times,
checked on every output; the larger ones on sampled rows).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import _parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    from nvfp4_quantized_rl_gb300 import _build
    _build.build()
    import nvfp4_quantized_rl_gb300 as m
    assert torch.cuda.is_available(), "GPU parity tests need a CUDA device"
    return m


def gpu_quantize(nv, x_np, mask=None, amax_in=None):
    x = P.dev_bf16(x_np) if x_np.dtype == np.uint16 else P.dev(x_np)
    m = None if mask is None else P.dev(mask.view(np.int32))
    a = None if amax_in is None else torch.tensor([amax_in], dtype=torch.float32, device="cuda")
    fn = nv.nvfp4_quantize if mask is None else (lambda t, **k: nv.nvfp4_quantize_guided(t, m, **k))
    c, s, g = fn(x, amax_in=a)
    torch.cuda.synchronize()
    return c.cpu().numpy(), s.cpu().numpy(), np.float32(g.cpu().numpy()[0])


def assert_quant_equal(got, want, what=""):
    (c1, s1, g1), (c2, s2, g2) = got, want
    assert np.float32(g1).view(np.uint32) == np.float32(g2).view(np.uint32), f"{what}: g {g1!r} vs {g2!r}"
    assert np.array_equal(s1, s2), f"{what}: {int((s1 != s2).sum())} scale bytes differ"
    assert np.array_equal(c1, c2), f"{what}: {int((c1 != c2).sum())} code bytes differ"


# ---------------------------------------------------------------- quantization

def test_quantize_tiny_fp32(nv):
    W = synth.tiny_config(0)["W"]
    assert_quant_equal(gpu_quantize(nv, W), oracle.quantize(W), "tiny fp32 256x512")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", [(1, 16), (37, 48), (300, 1040), (129, 4096)])
def test_quantize_ragged(nv, dtype, shape):
    W = synth.weight_f32(*shape, 0.02, 1, shape[0], outlier_frac=0.02)
    x = synth.bf16_bits(W) if dtype == "bf16" else W
    assert_quant_equal(gpu_quantize(nv, x), oracle.quantize(x), f"{dtype} {shape}")


def _edge_tensor():
    """Exact grid values, every E2M1 midpoint, +-0, zero blocks, tiny blocks (subnormal scale bytes)."""
    rng = np.random.default_rng(5)
    rows, cols = 64, 256
    g = np.float32(2.0 ** -6)
    x = np.zeros((rows, cols), np.float32)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float32)
    for r in range(rows):
        for b in range(cols // 16):
            s = np.float32(2.0 ** rng.integers(-9, 8))  # power-of-two block scales, some subnormal in E4M3
            vals = np.concatenate([mids, grid[1:], [0.0, 0.0]]) if (r + b) % 3 else rng.uniform(-7, 7, 16)
            vals = (vals * s * g).astype(np.float32) * np.where(rng.random(16) < 0.5, -1, 1).astype(np.float32)
            vals[0] = np.float32(6 * s * g)  # the block amax makes the scale byte exactly s
            x[r, 16 * b:16 * b + 16] = vals
    x[3] = 0.0
    x[4, :16] = -0.0
    x[0, 0] = np.float32(6 * 448 * g)  # tensor amax -> g exactly
    return x


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_quantize_edge_values(nv, dtype):
    x = _edge_tensor()
    x = synth.bf16_bits(x) if dtype == "bf16" else x
    want = oracle.quantize(x)
    assert_quant_equal(gpu_quantize(nv, x), want, "edge values")
    # saturation: a caller amax below the true one drives scale bytes to 0x7E and codes to 6
    a = float(np.float32(np.abs(synth.bf16_to_f32(x) if dtype == "bf16" else x).max()) / 5)
    assert_quant_equal(gpu_quantize(nv, x, amax_in=a), oracle.quantize(x, amax_in=a), "amax_in saturation")


def test_quantize_midpoints_with_general_scales(nv):
    """bf16 values exactly on E2M1 midpoints (and on grid points) of blocks whose E4M3 scale has a
    nonzero mantissa: every element is a rounding tie of the quotient x / (E4M3(s) g)."""
    rng = np.random.default_rng(11)
    rows, cols = 48, 512
    g = np.float32(2.0 ** -7)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    grid = np.array([.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    x = np.zeros((rows, cols), np.float32)
    for r in range(rows):
        for b in range(cols // 16):
            s = np.float32(2.0 ** int(rng.integers(-5, 7)) * (1 + int(rng.integers(0, 8)) / 8))
            vals = np.concatenate([[6.0], mids, grid[rng.integers(0, 7, 8)]])[:16].astype(np.float32)
            vals = vals * s * g * np.where(rng.random(16) < 0.5, -1, 1).astype(np.float32)
            x[r, 16 * b:16 * b + 16] = vals
    x[0, 0] = np.float32(6 * 448 * g)  # tensor amax -> g exactly
    xb = synth.bf16_bits(x)
    assert np.array_equal(synth.bf16_to_f32(xb), x)  # every value is exact in bf16
    assert_quant_equal(gpu_quantize(nv, xb), oracle.quantize(xb), "midpoint ties, general scales")


@pytest.mark.parametrize("M", [137, 150, 161, 231])
def test_quantize_bf16_next_to_midpoints(nv, M):
    """bf16 values next to every midpoint m E4M3(s) g (the three bf16 values nearest to it) in blocks of
    every normal scale byte s, with g = amax / 2688 for amax mantissas M: 231 = 11 * 21 makes g exact
    (m E4M3(s) g can then be a bf16 value: exact ties), 150 and 161 carry the factors 3 and 7 of 2688 / 2^7
    that put bf16 values within an fp32 rounding of m E4M3(s) g, 137 neither. The bf16 encoding rounds
    x times a reciprocal of E4M3(s) g with the hardware conversion: these are the values it must still
    decide exactly (codes, scales and g bit-exact against the oracle)."""
    rng = np.random.default_rng(M)
    amax = np.float32(M * 2.0 ** -4)
    g = float(np.float32(amax / np.float32(2688.0)))
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    blocks = []
    for b in range(0x08, 0x78):  # 6 E4M3(s) g stays below amax
        d = float(oracle.e4m3_value(b)) * g
        near = []
        for m in mids:
            c = int(synth.bf16_bits(np.array([m * d], np.float32))[0])
            near += [c - 1, c, c + 1]
        top = int(synth.bf16_bits(np.array([6.0 * d], np.float32))[0])
        vals = np.array(near + [top, top], np.uint16)  # 23 values: the block maximum in both blocks
        a, bb = np.concatenate([[top], vals[:15]]), np.concatenate([[top], vals[15:22], vals[:8]])
        for blk in (a, bb):
            blk = blk.astype(np.uint16) | (rng.integers(0, 2, 16) << 15).astype(np.uint16)
            blocks.append(rng.permutation(blk))
    amax_block = np.zeros(16, np.uint16)
    amax_block[3] = synth.bf16_bits(np.array([amax], np.float32))[0]
    blocks.append(amax_block)
    x = np.stack(blocks).reshape(-1, 64) if len(blocks) % 4 == 0 else np.stack(blocks + [np.zeros(16, np.uint16)] *
                                                                              (4 - len(blocks) % 4)).reshape(-1, 64)
    want = oracle.quantize(x)
    assert float(want[2]) == g
    assert_quant_equal(gpu_quantize(nv, x), want, f"bf16 next to midpoints, amax mantissa {M}")


def test_quantize_zero_tiny_and_huge(nv):
    z = np.zeros((8, 64), np.float32)
    z[2, 5] = -0.0
    assert_quant_equal(gpu_quantize(nv, z), oracle.quantize(z), "all zero")
    one = np.zeros((8, 64), np.float32)
    one[7, 63] = -3.0
    assert_quant_equal(gpu_quantize(nv, one), oracle.quantize(one), "single nonzero")
    tiny = (synth.weight_f32(16, 64, 1.0, 3, 1) * np.float32(1e-36)).astype(np.float32)  # g is subnormal
    assert_quant_equal(gpu_quantize(nv, tiny), oracle.quantize(tiny), "tiny g")
    huge = (synth.weight_f32(16, 64, 1.0, 3, 2) * np.float32(1e37)).astype(np.float32)
    assert_quant_equal(gpu_quantize(nv, huge), oracle.quantize(huge), "huge values")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_quantize_guided(nv, dtype):
    W = synth.weight_f32(200, 768, 0.02, 4, 1, outlier_frac=0.01)
    x = synth.bf16_bits(W) if dtype == "bf16" else W
    mask = synth.guided_mask(W.size, 4, 2)
    assert_quant_equal(gpu_quantize(nv, x, mask=mask), oracle.quantize(x, mask=mask), "guided")
    e = _edge_tensor()
    e = synth.bf16_bits(e) if dtype == "bf16" else e
    m2 = synth.guided_mask(e.size, 4, 3)
    assert_quant_equal(gpu_quantize(nv, e, mask=m2), oracle.quantize(e, mask=m2), "guided edge values")


def test_quantize_empty_is_a_noop(nv):
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    c, s, g = nv.nvfp4_quantize(x)
    torch.cuda.synchronize()
    assert c.shape == (0, 32) and s.shape == (0, 4)


def test_quantize_qwen7b_layer_full(nv):
    """All five weights of a Qwen2.5-7B-shaped layer (bf16, 1% outlier columns x8), every output byte."""
    for i, (name, (n, k)) in enumerate(synth.QWEN25_7B["linears"].items()):
        W = synth.weight_bf16(n, k, 0.02, 2, i, outlier_frac=0.01)
        assert_quant_equal(gpu_quantize(nv, W), oracle.quantize(W), f"7B {name}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_quantize_batch_mixed(nv, dtype):
    """nvfp4_quantize_batch on tensors of mixed sizes (so the fused encode + next-amax kernel runs
    with every share of the next tensor per iteration), an all-zero tensor, a tiny-g tensor and an
    empty one: each tensor's bytes equal the oracle's for that tensor alone."""
    mats = [synth.weight_f32(129, 4096, 0.02, 7, 1, outlier_frac=0.02), synth.weight_f32(300, 1040, 0.02, 7, 2),
            synth.weight_f32(37, 48, 1.0, 7, 3), np.zeros((8, 64), np.float32),
            (synth.weight_f32(16, 64, 1.0, 7, 4) * np.float32(1e-36)).astype(np.float32),
            synth.weight_f32(200, 2048, 0.05, 7, 5, outlier_frac=0.01), np.zeros((0, 64), np.float32),
            synth.weight_f32(1, 16, 3.0, 7, 6)]
    xs = [synth.bf16_bits(m) if dtype == "bf16" else m for m in mats]
    dev = [P.dev_bf16(x) if dtype == "bf16" else P.dev(x) for x in xs]
    codes, scales, gs = nv.nvfp4_quantize_batch(dev)
    torch.cuda.synchronize()
    for i, x in enumerate(xs):
        if x.shape[0] == 0:
            assert codes[i].shape == (0, 32)
            continue
        got = (codes[i].cpu().numpy(), scales[i].cpu().numpy(), np.float32(gs[i].cpu().numpy()[0]))
        assert_quant_equal(got, oracle.quantize(x), f"batch {dtype} tensor {i} {x.shape}")


def test_quantize_batch_qwen7b_layer(nv):
    """The weight refresh of the bench: all five Qwen2.5-7B-shaped weights in one batched call, every
    output byte against the oracle."""
    Ws = [synth.weight_bf16(n, k, 0.02, 2, i, outlier_frac=0.01)
          for i, (name, (n, k)) in enumerate(synth.QWEN25_7B["linears"].items())]
    codes, scales, gs = nv.nvfp4_quantize_batch([P.dev_bf16(W) for W in Ws])
    torch.cuda.synchronize()
    for i, W in enumerate(Ws):
        got = (codes[i].cpu().numpy(), scales[i].cpu().numpy(), np.float32(gs[i].cpu().numpy()[0]))
        assert_quant_equal(got, oracle.quantize(W), f"batch 7B weight {i}")


def test_quantize_moe_experts_guided(nv):
    """MoE expert weights (768x2048 gate/up, 2048x768 down); guided with a Bernoulli(1/2) mask, as for the
    deepest layers, and plain, on a seeded set of experts."""
    rng = np.random.default_rng(6)
    for e in rng.choice(128, 6, replace=False):
        for j, (n, k) in enumerate([(768, 2048), (768, 2048), (2048, 768)]):
            W = synth.weight_bf16(n, k, 0.02, 47, int(e), j)
            mask = synth.guided_mask(W.size, 47, int(e), j, 99)
            assert_quant_equal(gpu_quantize(nv, W, mask=mask), oracle.quantize(W, mask=mask), f"expert {e}.{j} guided")
            assert_quant_equal(gpu_quantize(nv, W), oracle.quantize(W), f"expert {e}.{j} plain")


def test_quantize_moe_guided_layers_sampled(nv):
    """Every guided layer of the MoE model (36..47 of 48): a seeded 1/32 of each layer's expert
    tensors (4 experts x gate, up, down), guided with that tensor's Bernoulli(1/2) mask, every block
    against the oracle."""
    cfg = synth.MOE
    H, I = cfg["hidden"], cfg["intermediate"]
    shapes = [(I, H), (I, H), (H, I)]
    for layer in cfg["guided_layers"]:
        experts = np.random.default_rng(1000 + layer).choice(cfg["experts"], 4, replace=False)
        for e in experts:
            for j, (n, k) in enumerate(shapes):
                W = synth.weight_bf16(n, k, 0.02, layer, int(e), j)
                mask = synth.guided_mask(W.size, layer, int(e), j, 99)
                assert_quant_equal(gpu_quantize(nv, W, mask=mask), oracle.quantize(W, mask=mask),
                                   f"layer {layer} expert {e}.{j} guided")


# ---------------------------------------------------------------- TRACE record and cached replay

def _mask_bits(words, n):
    return np.unpackbits(np.ascontiguousarray(words).view(np.uint8), bitorder="little")[:n]


def gpu_record(nv, x_np, fill=0):
    x = P.dev_bf16(x_np) if x_np.dtype == np.uint16 else P.dev(x_np)
    rec = torch.full(((x_np.size + 31) // 32,), fill, dtype=torch.int32, device="cuda")
    c, s, g, r = nv.nvfp4_quantize_record(x, record=rec)
    torch.cuda.synchronize()
    return (c.cpu().numpy(), s.cpu().numpy(), np.float32(g.cpu().numpy()[0])), r.cpu().numpy().view(np.uint32)


def gpu_cached(nv, x_np, mask, scales, g):
    x = P.dev_bf16(x_np) if x_np.dtype == np.uint16 else P.dev(x_np)
    gd = torch.tensor([np.float32(g)], dtype=torch.float32, device="cuda")
    c = nv.nvfp4_quantize_cached(x, P.dev(np.ascontiguousarray(mask).view(np.int32)), P.dev(scales), gd)
    torch.cuda.synchronize()
    return c.cpu().numpy()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", [(1, 16), (37, 48), (300, 1040), (129, 4096)])
def test_quantize_record_ragged(nv, dtype, shape):
    """Codes, scales and g as nvfp4_quantize; the record bit for bit; with an odd number of blocks
    the upper half of the last record word keeps its previous contents."""
    W = synth.weight_f32(*shape, 0.02, 12, shape[0], outlier_frac=0.02)
    x = synth.bf16_bits(W) if dtype == "bf16" else W
    got, rec = gpu_record(nv, x, fill=-0x5A5A5A5B)  # 0xA5A5A5A5
    c, s, g, m = oracle.quantize_record(x)
    assert_quant_equal(got, (c, s, g), f"record {dtype} {shape}")
    n = x.size
    assert np.array_equal(_mask_bits(rec, n), _mask_bits(m, n)), f"{dtype} {shape}: record bits differ"
    if (n // 16) % 2:
        assert rec[-1] >> 16 == 0xA5A5, "the unused half of the last record word was written"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_quantize_record_edge_values(nv, dtype):
    """Exact grid points, every midpoint (ties both ways), +-0, zero and subnormal-scale blocks."""
    e = _edge_tensor()
    x = synth.bf16_bits(e) if dtype == "bf16" else e
    got, rec = gpu_record(nv, x)
    c, s, g, m = oracle.quantize_record(x)
    assert_quant_equal(got, (c, s, g), f"record edge {dtype}")
    assert np.array_equal(_mask_bits(rec, x.size), _mask_bits(m, x.size))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_quantize_cached_replay(nv, dtype):
    """Replay from the rollout's cache: the same weights give the plain codes back; weights one
    update later, and a random mask, give the oracle's cached codes; degenerate caches (g = 0,
    negative g, bytes above 0x7E) follow the stated rules."""
    W = synth.weight_f32(200, 768, 0.02, 13, 1, outlier_frac=0.01)
    x = synth.bf16_bits(W) if dtype == "bf16" else W
    c, s, g, m = oracle.quantize_record(x)
    assert np.array_equal(gpu_cached(nv, x, m, s, g), c), "replay of the recorded weights"
    W2 = (W + synth.normal_f32(W.shape, 0.002, 13, 2)).astype(np.float32)
    x2 = synth.bf16_bits(W2) if dtype == "bf16" else W2
    assert np.array_equal(gpu_cached(nv, x2, m, s, g), oracle.quantize_cached(x2, m, s, g)), "updated weights"
    r = synth.guided_mask(W.size, 13, 3)
    assert np.array_equal(gpu_cached(nv, x2, r, s, g), oracle.quantize_cached(x2, r, s, g)), "random mask"
    s_odd = s.copy()
    s_odd[::7] = 0xFF
    s_odd[1::11] = 0x7F
    s_odd[2::13] = 0x00
    for gg in (g, np.float32(0.0), np.float32(-1.0)):
        assert np.array_equal(gpu_cached(nv, x2, r, s_odd, gg), oracle.quantize_cached(x2, r, s_odd, gg)), f"g={gg}"
    e = _edge_tensor()
    xe = synth.bf16_bits(e) if dtype == "bf16" else e
    ce, se, ge, me = oracle.quantize_record(xe)
    assert np.array_equal(gpu_cached(nv, xe, me, se, ge), ce), "edge values"


def _blocks_next_to_grid(M, seed):
    """bf16 blocks of every normal scale byte s whose elements are the three bf16 values nearest to each
    grid point G E4M3(s) g and each midpoint m E4M3(s) g, the block maximum 6 E4M3(s) g, random signs;
    g = amax / 2688 for the amax mantissa M (as in test_quantize_bf16_next_to_midpoints)."""
    rng = np.random.default_rng(seed)
    amax = np.float32(M * 2.0 ** -4)
    g = float(np.float32(amax / np.float32(2688.0)))
    pts = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    blocks = []
    for b in range(0x08, 0x78):  # 6 E4M3(s) g stays below amax
        d = float(oracle.e4m3_value(b)) * g
        near = []
        for p in pts:
            c = int(synth.bf16_bits(np.array([p * d], np.float32))[0])
            near += [c - 1, c, c + 1]
        top = int(synth.bf16_bits(np.array([6.0 * d], np.float32))[0])
        vals = np.array(near + near[:3], np.uint16)  # 45 values: three blocks of 15 beside the maximum
        for i in range(3):
            blk = np.concatenate([[top], vals[15 * i:15 * i + 15]]).astype(np.uint16)
            blk = blk | (rng.integers(0, 2, 16) << 15).astype(np.uint16)
            blocks.append(rng.permutation(blk))
    amax_block = np.zeros(16, np.uint16)
    amax_block[3] = synth.bf16_bits(np.array([amax], np.float32))[0]
    blocks.append(amax_block)
    blocks += [np.zeros(16, np.uint16)] * (-len(blocks) % 4)
    return np.stack(blocks).reshape(-1, 64), g


@pytest.mark.parametrize("M", [137, 150, 161, 231])
def test_quantize_guided_record_cached_next_to_grid_points(nv, M):
    """Guided, record and cached encodings of bf16 values next to every grid point and midpoint of
    every normal scale byte (see _blocks_next_to_grid): the bf16 path decides floor and ceiling from the
    hardware conversion of x times a reciprocal of E4M3(s) g, checked per scale byte against exactly
    these values (with M = 231 some of them lie on a grid point and the byte takes the compare form);
    codes, scales, g and record bits bit-exact against the oracle."""
    x, g = _blocks_next_to_grid(M, 40 + M)
    mask = synth.guided_mask(x.size, M, 1)
    want = oracle.quantize(x, mask=mask)
    assert float(want[2]) == g
    assert_quant_equal(gpu_quantize(nv, x, mask=mask), want, f"guided next to grid points, M {M}")
    got, rec = gpu_record(nv, x)
    c, s, gr, m = oracle.quantize_record(x)
    assert_quant_equal(got, (c, s, gr), f"record next to grid points, M {M}")
    assert np.array_equal(_mask_bits(rec, x.size), _mask_bits(m, x.size)), f"record bits, M {M}"
    assert np.array_equal(gpu_cached(nv, x, mask, s, gr), oracle.quantize_cached(x, mask, s, gr)), "cached"
    # given scale bytes one step off for a third of the blocks: the values then sit elsewhere on the grid
    s2 = s.copy().reshape(-1)
    rng = np.random.default_rng(M)
    pick = rng.random(s2.size) < 1 / 3
    s2[pick] = np.clip(s2[pick].astype(np.int32) + rng.choice([-1, 1], int(pick.sum())), 0, 0x7E).astype(np.uint8)
    s2 = s2.reshape(s.shape)
    assert np.array_equal(gpu_cached(nv, x, mask, s2, gr), oracle.quantize_cached(x, mask, s2, gr)), "cached, moved"


def test_quantize_guided_record_cached_subnormal_elements(nv):
    """Blocks that take the bf16 conversion form (a general g) whose other elements are bf16
    subnormals (2^-133 .. 2^-127), tiny normals and +-0 beside a normal block maximum: every nonzero
    element lies below the first grid point, so its floor is code 0 and its ceiling code 1, and the
    guided encoding must tell a subnormal from zero. Codes, scales, g and record bits bit-exact
    against the oracle; the cached mode with the recorded scales and a random mask."""
    rng = np.random.default_rng(77)
    rows, cols = 96, 512
    bits = np.zeros((rows, cols), np.uint16)
    sub = np.array([0x0001, 0x0002, 0x0007, 0x0040, 0x007F, 0x0080, 0x0081, 0x00FF, 0x0000], np.uint16)
    for r in range(rows):
        for b in range(cols // 16):
            top = synth.bf16_bits(np.array([rng.uniform(0.01, 1.5)], np.float32))[0]
            blk = np.concatenate([[top], rng.choice(sub, 15)]).astype(np.uint16)
            blk = blk | (rng.integers(0, 2, 16) << 15).astype(np.uint16)
            bits[r, 16 * b:16 * b + 16] = rng.permutation(blk)
    bits[0, 0] = synth.bf16_bits(np.array([1.7], np.float32))[0]  # amax 1.7: g = 1.7 / 2688, not a power of two
    mask = synth.guided_mask(bits.size, 77, 1)
    assert_quant_equal(gpu_quantize(nv, bits, mask=mask), oracle.quantize(bits, mask=mask), "guided, subnormals")
    got, rec = gpu_record(nv, bits)
    c, s, g, m = oracle.quantize_record(bits)
    assert_quant_equal(got, (c, s, g), "record, subnormals")
    assert np.array_equal(_mask_bits(rec, bits.size), _mask_bits(m, bits.size)), "record bits, subnormals"
    assert np.array_equal(gpu_cached(nv, bits, mask, s, g), oracle.quantize_cached(bits, mask, s, g)), "cached"


def test_trace_round_trip_gpu_only_qwen7b_gate(nv):
    """The full 7B gate weight (18944 x 3584 bf16): record, then replay from the GPU's own cache,
    gives the GPU's plain codes back; sampled rows of the record and of the codes match the oracle."""
    n, k = synth.QWEN25_7B["linears"]["gate"]
    W = synth.weight_bf16(n, k, 0.02, 14, 1, outlier_frac=0.01)
    x = P.dev_bf16(W)
    c, s, g, rec = nv.nvfp4_quantize_record(x)
    plain, _, _ = nv.nvfp4_quantize(x)
    replay = nv.nvfp4_quantize_cached(x, rec, s, g)
    torch.cuda.synchronize()
    assert torch.equal(replay, plain) and torch.equal(c, plain)
    rows = np.sort(np.random.default_rng(14).choice(n, 24, replace=False))
    gh = np.float32(g.cpu().numpy()[0])
    assert gh == oracle.global_scale(oracle.amax(W))
    rec_h = rec.cpu().numpy().view(np.uint32)
    for r in rows:
        cr, sr, gr, mr = oracle.quantize_record(W[r:r + 1], amax_in=oracle.amax(W))
        assert gr == gh
        assert np.array_equal(c[r].cpu().numpy(), cr[0]) and np.array_equal(s[r].cpu().numpy(), sr[0])
        assert np.array_equal(rec_h[r * k // 32:(r + 1) * k // 32], mr), f"row {r}: record bits differ"


# ---------------------------------------------------------------- FP4 KV cache and decode attention

def _kv_cache_dev(B, Lmax, Hkv, D=128, fill=0x5A):
    mk = lambda w: torch.full((B, Lmax, Hkv, w), fill, dtype=torch.uint8, device="cuda")
    return mk(D // 2), mk(D // 16), mk(D // 2), mk(D // 16)


def test_kv_append(nv):
    """New rows land bit-exactly (the oracle's encoding at the given g) at each sequence's position;
    a sequence whose position is outside the cache, and every other row, stay untouched."""
    B, Hkv, D, Lmax = 5, 4, 128, 7
    k = synth.activation_bf16(B * Hkv, D, 31, 1).reshape(B, Hkv, D)
    v = synth.heavy_tail_activation_bf16(B * Hkv, D, 31, 2).reshape(B, Hkv, D)
    pos = np.array([0, 6, 3, -1, 7], np.int32)  # the last two are outside [0, Lmax)
    gk, gv = np.float32(0.0021), np.float32(0.0047)
    kc, ks, vc, vs = _kv_cache_dev(B, Lmax, Hkv)
    nv.nvfp4_kv_append(P.dev_bf16(k), P.dev_bf16(v), P.dev(pos), P.dev(np.array([gk])), P.dev(np.array([gv])),
                       kc, ks, vc, vs)
    torch.cuda.synchronize()
    ck, sk = oracle.kv_quantize(k, gk)
    cv, sv = oracle.kv_quantize(v, gv)
    got = [t.cpu().numpy() for t in (kc, ks, vc, vs)]
    for b in range(B):
        for t in range(Lmax):
            written = t == pos[b]
            for arr, ref in zip(got, (ck, sk, cv, sv)):
                if written:
                    assert np.array_equal(arr[b, t], ref[b]), f"sequence {b} row {t}"
                else:
                    assert np.all(arr[b, t] == 0x5A), f"sequence {b} row {t} was written"


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,lens", [
    (3, 7, 1, 200, [1, 77, 200]),
    (4, 28, 4, 300, [300, 129, 64, 65]),
    (2, 16, 1, 2000, [1999, 640]),
    (2, 8, 2, 50, [0, 50]),
    (2, 40, 8, 130, [130, 66]),     # 5 query heads per KV head (Qwen2.5-32B grouping)
    (3, 9, 1, 257, [257, 1, 128]),  # 9 heads: two head tiles, the second nearly empty
])
def test_kv_decode_attention(nv, B, Hq, Hkv, Lmax, lens):
    """Cache built by nvfp4_kv_append one token at a time, attention against the oracle on the same
    cache bytes (ragged lengths, a single token, a length of 0, spans split across CTAs)."""
    D = 128
    g = np.float32(0.003)
    kc, ks, vc, vs = _kv_cache_dev(B, Lmax, Hkv, fill=0)
    gd = P.dev(np.array([g]))
    kall = synth.activation_bf16(B * Lmax * Hkv, D, 32, Hq).reshape(Lmax, B, Hkv, D)
    vall = synth.activation_bf16(B * Lmax * Hkv, D, 33, Hq).reshape(Lmax, B, Hkv, D)
    kd, vd = P.dev_bf16(kall), P.dev_bf16(vall)
    for t in range(Lmax):
        nv.nvfp4_kv_append(kd[t], vd[t], torch.full((B,), t, dtype=torch.int32, device="cuda"), gd, gd, kc, ks, vc, vs)
    q = synth.activation_bf16(B * Hq, D, 34, Hq).reshape(B, Hq, D)
    lens = np.array(lens, np.int32)
    scale = 1.0 / np.sqrt(D)
    out = nv.nvfp4_kv_decode_attention(P.dev_bf16(q), kc, ks, gd, vc, vs, gd, P.dev(lens), scale)
    torch.cuda.synchronize()
    caches = [t.cpu().numpy() for t in (kc, ks, vc, vs)]
    ck, sk = oracle.kv_quantize(kall.transpose(1, 0, 2, 3), g)
    assert np.array_equal(caches[0], ck) and np.array_equal(caches[1], sk), "cache bytes"
    got = P.host_bits(out)
    live = lens > 0
    ref = oracle.attention_decode(q[live], *(c[live] for c in caches[:2]), g, *(c[live] for c in caches[2:]), g,
                                  lens[live], scale)
    P.assert_gemm_close(got[live], ref, f"attention {B}x{Hq}/{Hkv} L={Lmax}")
    assert not got[~live].any(), "a sequence of length 0 gives zeros"


def _random_cache(B, Lmax, Hkv, lens, seed, fill):
    """Valid random NVFP4 rows (codes any byte, scale bytes 0x28..0x3F) below each length, `fill`
    bytes at and past it (0xFF: NaN scale bytes, -6 codes)."""
    rng = np.random.default_rng(seed)
    kc = rng.integers(0, 256, (B, Lmax, Hkv, 64), dtype=np.uint8)
    vc = rng.integers(0, 256, (B, Lmax, Hkv, 64), dtype=np.uint8)
    ks = rng.integers(0x28, 0x40, (B, Lmax, Hkv, 8), dtype=np.uint8)
    vs = rng.integers(0x28, 0x40, (B, Lmax, Hkv, 8), dtype=np.uint8)
    for b, n in enumerate(lens):
        for arr in (kc, vc, ks, vs):
            arr[b, n:] = fill
    return kc, ks, vc, vs


def test_kv_decode_attention_ignores_rows_past_length(nv):
    """Rows at and past each sequence's length hold NaN scale bytes and -6 codes (never written by
    nvfp4_kv_append): they must not reach the output, in full groups, ragged tails and spans."""
    B, Hq, Hkv, Lmax, D = 4, 28, 4, 300, 128
    lens = np.array([300, 129, 1, 64], np.int32)
    caches = _random_cache(B, Lmax, Hkv, lens, 37, 0xFF)
    g = np.float32(1.0 / 64)
    gd = P.dev(np.array([g]))
    q = synth.activation_bf16(B * Hq, D, 38, 1).reshape(B, Hq, D)
    dev = [torch.from_numpy(c).cuda() for c in caches]
    out = nv.nvfp4_kv_decode_attention(P.dev_bf16(q), dev[0], dev[1], gd, dev[2], dev[3], gd, P.dev(lens),
                                       1.0 / np.sqrt(D))
    torch.cuda.synchronize()
    got = P.host_bits(out)
    ref = oracle.attention_decode(q, caches[0], caches[1], g, caches[2], caches[3], g, lens, 1.0 / np.sqrt(D))
    assert np.all(np.isfinite(P.bf16_f64(got))), "rows past the length leaked into the output"
    P.assert_gemm_close(got, ref, "NaN-filled rows past the lengths")


@pytest.mark.parametrize("qmag", [2.0 ** -60, 2.0 ** 40, 0.0])
def test_kv_decode_attention_query_magnitudes(nv, qmag):
    """q scaled far from 1 (scores near 0: a near-uniform average; scores huge: one token wins) and
    q = 0 (the exact average of V): the power-of-two scaling of q must keep every result."""
    B, Hq, Hkv, Lmax, D = 2, 7, 1, 200, 128
    lens = np.array([200, 77], np.int32)
    caches = _random_cache(B, Lmax, Hkv, lens, 39, 0)
    g = np.float32(1.0 / 64)
    gd = P.dev(np.array([g]))
    q = synth.bf16_bits((P.bf16_f64(synth.activation_bf16(B * Hq, D, 40, 1)) * qmag).astype(np.float32))
    q = q.reshape(B, Hq, D)
    dev = [torch.from_numpy(c).cuda() for c in caches]
    out = nv.nvfp4_kv_decode_attention(P.dev_bf16(q), dev[0], dev[1], gd, dev[2], dev[3], gd, P.dev(lens),
                                       1.0 / np.sqrt(D))
    torch.cuda.synchronize()
    got = P.host_bits(out)
    ref = oracle.attention_decode(q, caches[0], caches[1], g, caches[2], caches[3], g, lens, 1.0 / np.sqrt(D))
    P.assert_gemm_close(got, ref, f"q x {qmag}")


def test_kv_decode_attention_qwen7b_sampled(nv):
    """Qwen2.5-7B decode at full size: 64 sequences, 28 query / 4 KV heads, 128 dims, an 8192-token
    cache of random valid NVFP4 bytes (scale bytes 0x28..0x3F), lengths 4096..8192; three sampled
    sequences against the oracle."""
    B, Hq, Hkv, D, Lmax = 64, 28, 4, 128, 8192
    gen = torch.Generator(device="cuda").manual_seed(35)
    codes = lambda: torch.randint(0, 256, (B, Lmax, Hkv, D // 2), generator=gen, device="cuda", dtype=torch.int32).to(torch.uint8)
    scl = lambda: torch.randint(0x28, 0x40, (B, Lmax, Hkv, D // 16), generator=gen, device="cuda", dtype=torch.int32).to(torch.uint8)
    kc, ks, vc, vs = codes(), scl(), codes(), scl()
    g = np.float32(1.0 / 64)
    gd = P.dev(np.array([g]))
    lens = np.random.default_rng(35).integers(4096, Lmax + 1, B).astype(np.int32)
    q = synth.activation_bf16(B * Hq, D, 36, 1).reshape(B, Hq, D)
    out = nv.nvfp4_kv_decode_attention(P.dev_bf16(q), kc, ks, gd, vc, vs, gd, P.dev(lens), 1.0 / np.sqrt(D))
    torch.cuda.synchronize()
    got = P.host_bits(out)
    for b in np.random.default_rng(36).choice(B, 3, replace=False):
        cb = [t[b:b + 1].cpu().numpy() for t in (kc, ks, vc, vs)]
        ref = oracle.attention_decode(q[b:b + 1], cb[0], cb[1], g, cb[2], cb[3], g, lens[b:b + 1], 1.0 / np.sqrt(D))
        P.assert_gemm_close(got[b:b + 1], ref, f"sequence {b}")


# ---------------------------------------------------------------- AIS mixing coefficient

AIS_ABS = ("alpha", "alpha_ess", "alpha_mis", "alpha_var", "cv2", "dsigma")  # dimensionless: 1e-5 absolute
AIS_REL = ("dbar", "mean_w")                                                 # 1e-5 relative


def gpu_ais(nv, lr, lt, adv, C, delta, gamma, beta):
    st, w = nv.ais_mixing(P.dev(lr), P.dev(lt), P.dev(adv), C, delta, gamma, beta)
    torch.cuda.synchronize()
    return dict(zip(nv.AIS_STATS, st.cpu().numpy().tolist())), w.cpu().numpy()


def assert_ais_close(got, want, C, what=""):
    (sg, wg), (sr, wr) = got, want
    for k in AIS_ABS:
        assert abs(sg[k] - sr[k]) <= 1e-5, f"{what}: {k} {sg[k]!r} vs {sr[k]!r}"
    for k in AIS_REL:
        assert abs(sg[k] - sr[k]) <= 1e-5 * abs(sr[k]) + 1e-12, f"{what}: {k} {sg[k]!r} vs {sr[k]!r}"
    err = np.abs(wg.astype(np.float64) - wr)
    assert err.max(initial=0.0) <= 1e-5 * (1 + C), f"{what}: weight error {err.max()}"


@pytest.mark.parametrize("n", [1, 3, 5, 1000, 4099, 65537, 300001])
def test_ais_sizes(nv, n):
    lr, lt, adv = synth.grpo_token_batch(8, 8, 512, 21, n, max_tokens=n)
    if lr.size < n:  # short batches: repeat the generated tokens
        reps = -(-n // lr.size)
        lr, lt, adv = (np.tile(a, reps)[:n].copy() for a in (lr, lt, adv))
    args = (2.0, 0.05, 0.5, 1.0)
    assert_ais_close(gpu_ais(nv, lr, lt, adv, *args), oracle.ais(lr, lt, adv, *args), 2.0, f"n={n}")


def test_ais_grpo_batch_full(nv):
    """The full GRPO batch (64 prompts x 8 responses of ~8K tokens, ~4 M tokens), every weight,
    for parameters where each factor of alpha is active."""
    b = synth.GRPO_BATCH
    lr, lt, adv = synth.grpo_token_batch(b["prompts"], b["group"], b["mean_len"], 22, max_tokens=b["tokens"])
    for args in [(2.0, 0.05, 0.5, 1.0), (1.05, 0.01, 1e-4, 0.5), (5.0, 1.0, 2e-3, 3.0)]:
        assert_ais_close(gpu_ais(nv, lr, lt, adv, *args), oracle.ais(lr, lt, adv, *args), args[0], f"{args}")


def test_ais_degenerate_batches(nv):
    """No mismatch (alpha = 0: every weight exactly 1), constant advantages (dsigma = 0), every
    ratio above C (all weights C), and a penalty that clips alpha to 0."""
    lr, lt, adv = synth.grpo_token_batch(4, 8, 256, 23, max_tokens=5000)
    st, w = gpu_ais(nv, lr, lr, adv, 2.0, 0.05, 0.5, 1.0)
    assert st["alpha"] == 0.0 and st["dbar"] == 0.0 and np.all(w == 1.0)
    const = np.full_like(adv, 0.75)
    assert_ais_close(gpu_ais(nv, lr, lt, const, 2.0, 0.05, 0.5, 1.0), oracle.ais(lr, lt, const, 2.0, 0.05, 0.5, 1.0),
                     2.0, "constant advantages")
    hi = (lr + 3.0).astype(np.float32)
    st, w = gpu_ais(nv, lr, hi, adv, 2.0, 0.05, 100.0, 1.0)
    assert st["mean_w"] == 2.0 and st["cv2"] == 0.0 and np.all(w == np.float32(1 + st["alpha"] * 1.0))
    clip = gpu_ais(nv, lr, (lr + np.float32(np.log(4.0))).astype(np.float32), adv, 100.0, 0.01, 0.5, 2.0)
    assert clip[0]["alpha"] == 0.0 and np.all(clip[1] == 1.0)


# ---------------------------------------------------------------- RMSNorm with AQN

def gpu_rmsnorm(nv, x, w, eps, sigma, delta):
    y = nv.rmsnorm_aqn(P.dev_bf16(x), P.dev(w), None if eps is None else P.dev(eps), sigma, delta)
    torch.cuda.synchronize()
    return P.host_bits(y)


def test_rmsnorm_tiny(nv):
    c = synth.tiny_config(0)
    s = np.float32(c["sigma"])
    y = gpu_rmsnorm(nv, c["x"], c["w"], c["eps"], s, c["delta"])
    P.assert_rmsnorm_close(y, oracle.rmsnorm_aqn(c["x"], c["w"], c["eps"], s, c["delta"]), "tiny")


def test_rmsnorm_schedule_qwen7b_decode(nv):
    x = synth.activation_bf16(64, 3584, 7, 1)
    w = synth.aqn_weight(3584, 7, 2)
    eps = synth.aqn_eps(3584, 7, 3)
    for k in range(11):
        s = np.float32(nv.aqn_sigma(1e-2, 5e-4, k, 10))
        y = gpu_rmsnorm(nv, x, w, eps, s, 1e-6)
        P.assert_rmsnorm_close(y, oracle.rmsnorm_aqn(x, w, eps, s, 1e-6), f"k={k}")


@pytest.mark.parametrize("shape", [(1, 8), (3, 520), (4096, 3584), (256, 5120), (8192, 5120)])
def test_rmsnorm_shapes(nv, shape):
    M, H = shape
    x = synth.activation_bf16(M, H, 8, M)
    w = synth.aqn_weight(H, 8, 2)
    eps = synth.aqn_eps(H, 8, 3)
    y = gpu_rmsnorm(nv, x, w, eps, np.float32(3e-3), 1e-6)
    P.assert_rmsnorm_close(y, oracle.rmsnorm_aqn(x, w, eps, np.float32(3e-3), 1e-6), f"{shape}")
    y0 = gpu_rmsnorm(nv, x, w, None, 0.0, 1e-6)
    P.assert_rmsnorm_close(y0, oracle.rmsnorm_aqn(x, w, None, 0.0, 1e-6), f"{shape} no noise")


# ---------------------------------------------------------------- LoRA linear

def _weights(n, k, seed, *stream, std=0.02, outliers=0.01, mask=None):
    W = synth.weight_bf16(n, k, std, seed, *stream, outlier_frac=outliers)
    return oracle.quantize(W, mask=mask)


@pytest.mark.parametrize("noise", [True, False], ids=["aqn", "plain"])
@pytest.mark.parametrize("shape", [(1, 16), (3, 528), (64, 3584), (4096, 3584), (300, 4096), (8192, 5120)])
def test_rmsnorm_quantize(nv, shape, noise):
    """rmsnorm_aqn_quantize: y within the RMSNorm tolerance of the oracle, and codes, scales and g
    exactly the oracle's quantization of that y (4096 x 3584 and 300 x 4096 take the fused
    on-chip kernel, 8192 x 5120 the fallback). Both paths also give rmsnorm_aqn's y bit for bit
    (same per-row partition and summation order)."""
    M, H = shape
    x = synth.heavy_tail_activation_bf16(M, H, 41, M) if M >= 64 else synth.activation_bf16(M, H, 41, M)
    w = synth.aqn_weight(H, 41, 2)
    eps = synth.aqn_eps(H, 41, 3) if noise else None
    sig = np.float32(3e-3) if noise else np.float32(0.0)
    xd, wd, ed = P.dev_bf16(x), P.dev(w), None if eps is None else P.dev(eps)
    y, c, sc, g = nv.rmsnorm_aqn_quantize(xd, wd, ed, sig, 1e-6)
    y_alone = nv.rmsnorm_aqn(xd, wd, ed, sig, 1e-6)
    torch.cuda.synchronize()
    yb = P.host_bits(y)
    P.assert_rmsnorm_close(yb, oracle.rmsnorm_aqn(x, w, eps, sig, 1e-6), f"{shape} y")
    assert np.array_equal(yb, P.host_bits(y_alone)), f"{shape}: y differs from rmsnorm_aqn"
    got = (c.cpu().numpy(), sc.cpu().numpy(), np.float32(g.cpu().numpy()[0]))
    assert_quant_equal(got, oracle.quantize(yb), f"{shape} quantized y")


def gpu_linear(nv, w4a4, x, q, A, B, s, offsets=None):
    codes, scales, g = q
    fn = nv.nvfp4_lora_linear_w4a4 if w4a4 else nv.nvfp4_lora_linear
    gd = P.dev(np.atleast_1d(np.asarray(g, np.float32)))
    kw = {}
    if offsets is not None:
        kw = dict(group_offsets=P.dev(offsets.astype(np.int32)), num_groups=len(offsets) - 1)
    y = fn(P.dev_bf16(x), P.dev(codes), P.dev(scales), gd, None if A is None else P.dev_bf16(A),
           None if B is None else P.dev_bf16(B), s, **kw)
    torch.cuda.synchronize()
    return P.host_bits(y)


def ref_linear(w4a4, x, q, A, B, s, rows=None):
    if w4a4:
        return oracle.lora_linear_w4a4(x, *q, A, B, s, rows=rows)[0]
    return oracle.lora_linear_w4a16(x, *q, A, B, s, rows=rows)


@pytest.mark.parametrize("w4a4", [False, True], ids=["w4a16", "w4a4"])
def test_linear_tiny(nv, w4a4):
    c = synth.tiny_config(0)
    q = oracle.quantize(c["W"])
    y = gpu_linear(nv, w4a4, c["x"], q, c["A"], c["B"], c["s"])
    P.assert_gemm_close(y, ref_linear(w4a4, c["x"], q, c["A"], c["B"], c["s"]), "tiny")


@pytest.mark.parametrize("w4a4", [False, True], ids=["w4a16", "w4a4"])
@pytest.mark.parametrize("M,N,K,r,s", [(100, 384, 768, 32, 2.0), (1, 128, 256, 0, 2.0), (65, 256, 512, 16, 0.0),
                                       (200, 640, 1024, 64, 0.5), (200, 384, 1024, 128, 1.0), (64, 256, 512, 128, 2.0),
                                       (130, 384, 768, 48, 1.0), (70, 256, 512, 112, 0.5)])
def test_linear_multi_tile_ragged(nv, w4a4, M, N, K, r, s):
    q = _weights(N, K, 11, M, N)
    x = synth.heavy_tail_activation_bf16(M, K, 12, M) if w4a4 else synth.activation_bf16(M, K, 12, M)
    A, B = synth.lora_factors(r, K, N, 13, M) if r else (None, None)
    y = gpu_linear(nv, w4a4, x, q, A, B, s)
    P.assert_gemm_close(y, ref_linear(w4a4, x, q, A, B, s), f"{M}x{N}x{K} r={r}")


@pytest.mark.parametrize("M,N,K,r,s", [(300, 9728, 512, 64, 2.0), (256, 9728, 512, 0, 1.0), (200, 9728, 256, 48, 0.5),
                                       (260, 256, 16384, 32, 1.0), (129, 384, 16384, 16, 2.0)])
def test_linear_256_token_tiles(nv, M, N, K, r, s):
    """W4A16 with more than 128 tokens at LoRA ranks up to 64 on 256-token tiles (taken when those
    fill half the SMs, 76 column tiles here, or K has 64 stages or more, split over a cluster here):
    the LoRA branch folded into the accumulator as hi + lo of c U, token tiles past M, r = 48 in a
    zero-padded 64-rank box, no LoRA at all."""
    q = _weights(N, K, 21, M, N)
    x = synth.activation_bf16(M, K, 22, M)
    A, B = synth.lora_factors(r, K, N, 23, M) if r else (None, None)
    y = gpu_linear(nv, False, x, q, A, B, s)
    P.assert_gemm_close(y, ref_linear(False, x, q, A, B, s), f"{M}x{N}x{K} r={r}")


@pytest.mark.parametrize("case", ["zero_weight", "small_scales"])
def test_linear_256_token_tiles_edge_weights(nv, case):
    """256-token tiles on an all-zero weight tensor (g = 0: the folded LoRA term enters with c = s and
    the output scale is 1, Y = s (x A^T) B^T) and on weights whose block scale bytes are zero or E4M3
    subnormals (the general dequant branch)."""
    M, N, K, r, s = 200, 9728, 256, 32, 2.0
    if case == "zero_weight":
        q = oracle.quantize(np.zeros((N, K), np.uint16))
        assert q[2] == 0.0
    else:
        W = synth.weight_bf16(N, K, 0.02, 91, 15)
        W[5] = 0
        amax = float(np.abs(synth.bf16_to_f32(W)).max())
        q = oracle.quantize(W, amax_in=amax * 2.0 ** 15)
        assert (q[1] <= 7).all() and (q[1] == 0).any()
    x = synth.activation_bf16(M, K, 92, 0)
    A, B = synth.lora_factors(r, K, N, 93, 0)
    y = gpu_linear(nv, False, x, q, A, B, s)
    P.assert_gemm_close(y, ref_linear(False, x, q, A, B, s), case)


def test_linear_empty_is_a_noop(nv):
    q = _weights(128, 256, 1)
    x = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    y = nv.nvfp4_lora_linear(x, P.dev(q[0]), P.dev(q[1]), P.dev(np.atleast_1d(q[2])))
    torch.cuda.synchronize()
    assert y.shape == (0, 128)


@pytest.mark.parametrize("w4a4", [False, True], ids=["w4a16", "w4a4"])
@pytest.mark.parametrize("shift", [15, 17])
def test_linear_small_scale_bytes(nv, w4a4, shift):
    """Weights quantized against a per-tensor amax 2^shift above their own, so that almost every block
    scale byte is zero or an E4M3 subnormal (0x00..0x07; the all-zero rows of W too), and the output
    is made of those blocks alone: the dequantization of small scale bytes is what the GEMM bar sees."""
    M, N, K, r = 96, 384, 1024, 32
    W = synth.weight_bf16(N, K, 0.02, 81, shift)
    W[5] = 0  # all-zero rows: scale byte 0
    W[200] = 0
    amax = float(np.abs(synth.bf16_to_f32(W)).max())
    q = oracle.quantize(W, amax_in=amax * 2.0 ** shift)
    sb = q[1]
    assert (sb <= 7).all() and (sb == 0).any() and len(np.unique(sb)) >= 3, np.unique(sb)
    x = synth.activation_bf16(M, K, 82, shift)
    A, B = synth.lora_factors(r, K, N, 83, shift)
    y = gpu_linear(nv, w4a4, x, q, A, B, 0.5)
    P.assert_gemm_close(y, ref_linear(w4a4, x, q, A, B, 0.5), f"small weight scales (2^-{shift})")


def test_w4a4_small_activation_scale_bytes(nv):
    """W4A4 with activations whose per-tensor amax sits in row 0 while every other row is 2^16 smaller:
    the activation quantizer gives those rows zero or subnormal block scale bytes, which the block-scaled
    MMA must decode exactly. Rows 1.. are compared on their own (row 0 dominates the output's rms)."""
    M, N, K = 130, 256, 512
    x = synth.bf16_to_f32(synth.activation_bf16(M, K, 84, 0))
    x[1:] *= np.float32(2.0 ** -16)
    x[7] = 0.0
    xb = synth.bf16_bits(x)
    q = _weights(N, K, 85, 0)
    gx = oracle.global_scale(oracle.amax(xb))
    _, xs = oracle.quantize_rows_given_g(xb, gx, np.arange(M))
    assert (xs[1:] <= 7).mean() > 0.99 and (xs[1:] == 0).any(), np.unique(xs[1:])
    y = gpu_linear(nv, True, xb, q, None, None, 0.0)
    ref = ref_linear(True, xb, q, None, None, 0.0)
    P.assert_gemm_close(y[:1], ref[:1], "row 0 (normal scales)")
    P.assert_gemm_close(y[1:], ref[1:], "rows 1.. (subnormal activation scales)")


@pytest.mark.parametrize("w4a4", [False, True], ids=["w4a16", "w4a4"])
@pytest.mark.parametrize("M,K,r", [(1300, 1280, 16), (1300, 1280, 112), (2048, 768, 48), (1025, 512, 128)])
def test_linear_prefill_sized_lora_down(nv, w4a4, M, K, r):
    """From 1024 rows the LoRA down-projection runs on the tensor cores in 128-row tiles with K split
    over a cluster; ragged row tiles, ranks from 16 to 128, plain U (W4A16) and hi/lo (W4A4) outputs.
    Sampled rows, the first and last included."""
    N = 256
    q = _weights(N, K, 96, M, r)
    x = synth.heavy_tail_activation_bf16(M, K, 97, r) if w4a4 else synth.activation_bf16(M, K, 97, r)
    A, B = synth.lora_factors(r, K, N, 98, M)
    y = gpu_linear(nv, w4a4, x, q, A, B, 1.5)
    rows = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(99).choice(M, 62, replace=False)]))
    P.assert_gemm_close(y[rows], ref_linear(w4a4, x, q, A, B, 1.5, rows=rows), f"M={M} K={K} r={r}")


@pytest.mark.parametrize("r", [48, 96])
def test_w4a4_lora_rank_not_a_multiple_of_64(nv, r):
    """The W4A4 kernel runs the LoRA up-projection in 64-rank slices; ranks that leave the last slice
    partly empty (its columns past r read as zeros) over several row and column tiles."""
    M, N, K, s = 150, 512, 768, 1.5
    q = _weights(N, K, 86, r)
    x = synth.heavy_tail_activation_bf16(M, K, 87, r)
    A, B = synth.lora_factors(r, K, N, 88, r)
    y = gpu_linear(nv, True, x, q, A, B, s)
    P.assert_gemm_close(y, ref_linear(True, x, q, A, B, s), f"r={r}")


def test_w4a4_lora_with_zero_alpha(nv):
    """alpha = g_x g_w = 0 with a LoRA branch. An all-zero weight tensor (g_w = 0): Y = s (x A^T) B^T
    alone. An all-zero activation tensor (g_x = 0, U = 0): Y = 0."""
    M, N, K, r, s = 140, 256, 512, 32, 2.0
    q = oracle.quantize(np.zeros((N, K), np.uint16))
    assert np.float32(q[2]) == 0
    x = synth.activation_bf16(M, K, 89, 0)
    A, B = synth.lora_factors(r, K, N, 89, 1)
    y = gpu_linear(nv, True, x, q, A, B, s)
    P.assert_gemm_close(y, ref_linear(True, x, q, A, B, s), "zero weights: LoRA branch alone")
    q2 = _weights(N, K, 89, 2)
    y0 = gpu_linear(nv, True, np.zeros((M, K), np.uint16), q2, A, B, s)
    assert not (y0 & 0x7FFF).any(), "zero activations must give zero outputs"


def _clear_status(nv):
    st, word = nv.device_status(clear=True)
    return st, word


def test_w4a4_lora_tiny_alpha_in_range(nv):
    """Weights ~1e-20 (g_w ~1e-23): the LoRA branch enters the accumulator scaled by s / alpha ~1e25,
    still within range; the result stays within the GEMM bar and no status bit is set."""
    M, N, K, r, s = 130, 384, 512, 32, 2.0
    assert _clear_status(nv)[0] == 0
    q = _weights(N, K, 90, 0, std=1e-20)
    x = synth.activation_bf16(M, K, 90, 1)
    A, B = synth.lora_factors(r, K, N, 90, 2)
    y = gpu_linear(nv, True, x, q, A, B, s)
    P.assert_gemm_close(y, ref_linear(True, x, q, A, B, s), "weights ~1e-20")
    assert _clear_status(nv) == (0, 0)


def test_w4a4_lora_scale_out_of_range_sets_status(nv):
    """Weights ~1e-30 put s / alpha above 2^100: the call sets the range bit of the device status word
    (NVFP4RL_ERR_RANGE, bit 5) and the context keeps working."""
    M, N, K, r = 130, 256, 512, 16
    assert _clear_status(nv)[0] == 0
    q = _weights(N, K, 95, 0, std=1e-30, outliers=0.0)
    x = synth.activation_bf16(M, K, 95, 1)
    A, B = synth.lora_factors(r, K, N, 95, 2)
    gpu_linear(nv, True, x, q, A, B, 2.0)
    assert _clear_status(nv) == (9, 32)
    assert _clear_status(nv) == (0, 0)
    q2 = _weights(N, K, 95, 3)
    y = gpu_linear(nv, True, x, q2, A, B, 2.0)
    P.assert_gemm_close(y, ref_linear(True, x, q2, A, B, 2.0), "after the range report")


@pytest.mark.parametrize("M,N,K,r", [(300, 384, 1024, 32), (130, 256, 512, 0), (200, 640, 1024, 128),
                                     (4096, 3584, 3584, 32)])
def test_w4a4_quantized_activations(nv, M, N, K, r):
    """nvfp4_lora_linear_w4a4_quantized on the NVFP4 output of rmsnorm_aqn_quantize: within the GEMM bar
    of the oracle's W4A4 on the normalized activations y, and the same bits as nvfp4_lora_linear_w4a4(y)
    (which quantizes y itself, to the same codes)."""
    x = synth.heavy_tail_activation_bf16(M, K, 91, M)
    w = synth.aqn_weight(K, 91, 2)
    eps = synth.aqn_eps(K, 91, 3)
    q = _weights(N, K, 92, M)
    A, B = synth.lora_factors(r, K, N, 93, M) if r else (None, None)
    yd, xc, xs, xg = nv.rmsnorm_aqn_quantize(P.dev_bf16(x), P.dev(w), P.dev(eps), np.float32(3e-3), 1e-6)
    gd = P.dev(np.atleast_1d(np.asarray(q[2], np.float32)))
    Ad, Bd = (None, None) if not r else (P.dev_bf16(A), P.dev_bf16(B))
    cd, sd = P.dev(q[0]), P.dev(q[1])
    out = nv.nvfp4_lora_linear_w4a4_quantized(yd if r else None, xc, xs, xg, cd, sd, gd, Ad, Bd, 2.0)
    ref_call = nv.nvfp4_lora_linear_w4a4(yd, cd, sd, gd, Ad, Bd, 2.0)
    torch.cuda.synchronize()
    got = P.host_bits(out)
    assert np.array_equal(got, P.host_bits(ref_call)), "differs from the quantize-on-the-fly call"
    y = P.host_bits(yd)
    rows = None if M <= 512 else np.sort(np.random.default_rng(94).choice(M, 48, replace=False))
    want = ref_linear(True, y, q, A, B, 2.0, rows=rows)
    P.assert_gemm_close(got if rows is None else got[rows], want, f"{M}x{N}x{K} r={r}")


def test_linear_qwen7b_decode_full(nv):
    """The 7B decode layer the benchmark times: M=64 bf16 tokens, every linear, r=32, every output."""
    x = synth.activation_bf16(64, 3584, 21, 0)
    x_int = synth.activation_bf16(64, 18944, 21, 1)
    for i, (name, (n, k)) in enumerate(synth.QWEN25_7B["linears"].items()):
        q = _weights(n, k, 2, i)
        A, B = synth.lora_factors(32, k, n, 22, i)
        xi = x_int if k == 18944 else x
        y = gpu_linear(nv, False, xi, q, A, B, 2.0)
        P.assert_gemm_close(y, ref_linear(False, xi, q, A, B, 2.0), f"7B {name}")


def test_w4a4_qwen7b_prefill_sampled(nv):
    """W4A4 at M=4096 with heavy-tailed channels; sampled rows (g_x still over all of x)."""
    x = synth.heavy_tail_activation_bf16(4096, 3584, 31, 0)
    x_int = synth.heavy_tail_activation_bf16(4096, 18944, 31, 1)
    rows = np.sort(np.random.default_rng(32).choice(4096, 48, replace=False))
    for i, (name, (n, k)) in enumerate(synth.QWEN25_7B["linears"].items()):
        if name in ("o", "up"):
            continue  # same shapes as q and gate
        q = _weights(n, k, 2, i)
        A, B = synth.lora_factors(32, k, n, 33, i)
        xi = x_int if k == 18944 else x
        y = gpu_linear(nv, True, xi, q, A, B, 2.0)
        P.assert_gemm_close(y[rows], ref_linear(True, xi, q, A, B, 2.0, rows=rows), f"7B W4A4 {name}")


@pytest.fixture(scope="module")
def qwen32b_layer():
    """The seven bf16 weights of one Qwen2.5-32B-shaped layer (~N(0, 0.015)) and the oracle's NVFP4
    encoding of each, shared by the quantization and the linear parity tests."""
    out = {}
    for i, (name, (n, k)) in enumerate(synth.QWEN25_32B["linears"].items()):
        W = synth.weight_bf16(n, k, 0.015, 3, i)
        out[name] = (W, oracle.quantize(W))
    return out


def test_quantize_qwen32b_layer_full(nv, qwen32b_layer):
    """Standalone nvfp4_quantize of all seven 32B-shaped weights (q, k, v, o, gate, up, down), every
    output byte against the oracle."""
    for name, (W, want) in qwen32b_layer.items():
        assert_quant_equal(gpu_quantize(nv, W), want, f"32B {name}")


def test_qwen32b_decode_and_prefill_sampled(nv, qwen32b_layer):
    """All seven 32B-shaped linears (r = 64): W4A16 at M = 256 and W4A4 at M = 8192, sampled rows."""
    rows256 = np.arange(0, 256, 8)
    rows8k = np.sort(np.random.default_rng(41).choice(8192, 24, replace=False))
    xs = {}
    for i, (name, (W, q)) in enumerate(qwen32b_layer.items()):
        n, k = W.shape
        if k not in xs:
            xs[k] = (synth.activation_bf16(256, k, 40, k), synth.heavy_tail_activation_bf16(8192, k, 40, k + 1))
        x256, x8k = xs[k]
        A, B = synth.lora_factors(64, k, n, 42, i)
        y = gpu_linear(nv, False, x256, q, A, B, 2.0)
        P.assert_gemm_close(y[rows256], ref_linear(False, x256, q, A, B, 2.0, rows=rows256), f"32B M=256 {name}")
        y = gpu_linear(nv, True, x8k, q, A, B, 2.0)
        P.assert_gemm_close(y[rows8k], ref_linear(True, x8k, q, A, B, 2.0, rows=rows8k), f"32B M=8192 {name}")


# ---------------------------------------------------------------- grouped (MoE) W4A4

def _grouped_ref(x, qs, offsets, rows):
    """Per-expert dense oracle on the sampled rows (the grouped definition)."""
    out = []
    gx = oracle.global_scale(oracle.amax(x))
    xc, xs = oracle.quantize_rows_given_g(x, gx, rows)
    xq = oracle.dequantize(xc, xs, gx)
    for i, r in enumerate(rows):
        e = int(np.searchsorted(offsets, r, side="right") - 1)
        out.append(oracle.linear(xq[i:i + 1], None, *qs[e], None, None, 0.0)[0])
    return np.stack(out)


def _stack(qs):
    return (np.stack([q[0] for q in qs]), np.stack([q[1] for q in qs]), np.array([q[2] for q in qs], np.float32))


def test_grouped_small_with_empty_experts(nv):
    E, N, K = 8, 256, 512
    tok, off = synth.moe_routing(96, E, 2, 5, 1)
    off = off.copy()
    # force expert 3 to be empty
    counts = np.diff(off)
    counts[4] += counts[3]
    counts[3] = 0
    off[1:] = np.cumsum(counts)
    x = synth.activation_bf16(int(off[-1]), K, 51, 0)
    qs = [_weights(N, K, 52, e) for e in range(E)]
    y = gpu_linear(nv, True, x, _stack(qs), None, None, 0.0, offsets=off)
    rows = np.arange(int(off[-1]))
    P.assert_gemm_close(y, _grouped_ref(x, qs, off, rows), "grouped small")


def test_grouped_moe_layer_sampled(nv):
    """One MoE layer: 4096 tokens top-8 over 128 experts (32768 routed rows); guided-quantized expert
    weights of the deepest layer; gate/up (768x2048) and down (2048x768); sampled rows."""
    cfg = synth.MOE
    E, H, I = cfg["experts"], cfg["hidden"], cfg["intermediate"]
    _, off = synth.moe_routing(cfg["tokens"], E, cfg["top_k"], 47, 0)
    M = int(off[-1])
    rows = np.sort(np.random.default_rng(61).choice(M, 64, replace=False))
    for j, (n, k) in enumerate([(I, H), (H, I)]):
        qs = []
        for e in range(E):
            W = synth.weight_bf16(n, k, 0.02, 47, e, j)
            qs.append(oracle.quantize(W, mask=synth.guided_mask(W.size, 47, e, j, 99)))
        x = synth.activation_bf16(M, k, 62, j)
        y = gpu_linear(nv, True, x, _stack(qs), None, None, 0.0, offsets=off)
        P.assert_gemm_close(y[rows], _grouped_ref(x, qs, off, rows), f"MoE {'gate' if j == 0 else 'down'}")
