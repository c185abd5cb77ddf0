"""The allocation-free W4A16 entry point (nvfp4_lora_linear_noalloc) against the workspace one.

Callers that cannot allocate device memory (code inside another framework's memory planner,
runtimes that forbid cudaMalloc, processes that must not grow their device footprint after
start-up) use nvfp4_lora_linear_noalloc, whose scratch is a fixed array inside the library.
Through the C ABI, two calls in a row on the same inputs must each give exactly the bits of
nvfp4_lora_linear with a torch-allocated workspace (both reduce split-K partials in a fixed
order), and both must lie within the GEMM tolerance of the oracle. The second call runs on the
array the first one left behind. The file is named to be collected last.
"""
import ctypes

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
    assert torch.cuda.is_available()
    return m


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


# decode (64 tokens, 7B q/o shape), tiny tiles, no LoRA with a ragged M, and rank 128 at M > 64
# (64-token tiles over four row tiles)
@pytest.mark.parametrize("M,N,K,r", [(64, 3584, 3584, 32), (8, 256, 512, 16), (33, 640, 1024, 0),
                                     (200, 384, 1024, 128)])
def test_noalloc_matches_workspace_entry_point(nv, M, N, K, r):
    W = synth.weight_bf16(N, K, 0.02, 71, N, K, outlier_frac=0.01)
    qc, qs, qg = oracle.quantize(W)
    codes, scales, gd = P.dev(qc), P.dev(qs), P.dev(np.atleast_1d(qg))
    x_np = synth.activation_bf16(M, K, 72, M)
    x = P.dev_bf16(x_np)
    A, B, a_np, b_np = None, None, None, None
    if r:
        a_np, b_np = synth.lora_factors(r, K, N, 73, M)
        A, B = P.dev_bf16(a_np), P.dev_bf16(b_np)
    L = nv.lib()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # the workspace entry point
    wsb = nv.workspace_bytes(nv.OP_LINEAR_W4A16, M, N, K, r)
    assert 0 < wsb <= L.nvfp4rl_noalloc_scratch_bytes()
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    y_ws = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    assert L.nvfp4_lora_linear(_ptr(x), M, K, _ptr(codes), _ptr(scales), _ptr(gd), N, _ptr(A), _ptr(B), r, 2.0,
                               None, 0, _ptr(y_ws), _ptr(ws), wsb, st) == 0
    torch.cuda.synchronize()
    ws_bits = P.host_bits(y_ws)
    ref = oracle.lora_linear_w4a16(x_np, qc, qs, qg, a_np, b_np, 2.0)
    P.assert_gemm_close(ws_bits, ref, "workspace entry point vs oracle")
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert L.nvfp4_lora_linear_noalloc(_ptr(x), M, K, _ptr(codes), _ptr(scales), _ptr(gd), N, _ptr(A), _ptr(B),
                                           r, 2.0, _ptr(y), st) == 0
        torch.cuda.synchronize()
        got = P.host_bits(y)
        assert np.array_equal(got, ws_bits), \
            f"noalloc call {call + 1}: {int((got != ws_bits).sum())} outputs differ from the workspace call"
        P.assert_gemm_close(got, ref, f"noalloc call {call + 1} vs oracle")


def test_noalloc_rejects_problems_beyond_its_scratch(nv):
    L = nv.lib()
    cap = L.nvfp4rl_noalloc_scratch_bytes()
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # U = bf16(x A^T) of 32768 tokens at rank 128 is 8 MiB, more than the fixed array
    M, N, K, r = 32768, 1024, 256, 128
    assert nv.workspace_bytes(nv.OP_LINEAR_W4A16, M, N, K, r) > cap
    assert L.nvfp4_lora_linear_noalloc(p, M, K, p, p, p, N, p, p, r, 1.0, p, st) == 4  # NVFP4RL_ERR_WORKSPACE
    # a rank the linear does not take is reported as such, before the scratch is considered
    assert L.nvfp4_lora_linear_noalloc(p, 8, K, p, p, p, N, p, p, 136, 1.0, p, st) == 3  # UNSUPPORTED_SHAPE
