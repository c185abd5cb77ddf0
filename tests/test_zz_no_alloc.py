"""The allocation-free W4A16 entry point (nvfp4_lora_linear_noalloc) against the workspace one.

Callers that cannot allocate device memory use nvfp4_lora_linear_noalloc, whose scratch is a
fixed array inside the library. Through the C ABI, two calls in a row on the same inputs must
each match nvfp4_lora_linear (given a torch-allocated workspace) within the GEMM tolerance of
the parity tests; the second call runs on the array the first one left behind. The file is
named to be collected last.
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


@pytest.mark.parametrize("M,N,K,r", [(64, 3584, 3584, 32), (8, 256, 512, 16), (33, 640, 1024, 0)])
def test_noalloc_matches_workspace_entry_point(nv, M, N, K, r):
    W = synth.weight_bf16(N, K, 0.02, 71, N, K, outlier_frac=0.01)
    qc, qs, qg = oracle.quantize(W)
    codes, scales, gd = P.dev(qc), P.dev(qs), P.dev(np.atleast_1d(qg))
    x = P.dev_bf16(synth.activation_bf16(M, K, 72, M))
    A, B = (None, None)
    if r:
        a_np, b_np = synth.lora_factors(r, K, N, 73, M)
        A, B = P.dev_bf16(a_np), P.dev_bf16(b_np)
    L = nv.lib()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # the workspace entry point
    wsb = nv.workspace_bytes(nv.OP_LINEAR_W4A16, M, N, K, r)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    y_ref = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    assert L.nvfp4_lora_linear(_ptr(x), M, K, _ptr(codes), _ptr(scales), _ptr(gd), N, _ptr(A), _ptr(B), r, 2.0,
                               None, 0, _ptr(y_ref), _ptr(ws), wsb, st) == 0
    assert L.nvfp4rl_noalloc_scratch_bytes() >= wsb
    ref = P.bf16_f64(P.host_bits(y_ref))
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert L.nvfp4_lora_linear_noalloc(_ptr(x), M, K, _ptr(codes), _ptr(scales), _ptr(gd), N, _ptr(A), _ptr(B),
                                           r, 2.0, _ptr(y), st) == 0
        torch.cuda.synchronize()
        P.assert_gemm_close(P.host_bits(y), ref, f"noalloc call {call + 1}")


def test_noalloc_rejects_problems_beyond_its_scratch(nv):
    L = nv.lib()
    cap = L.nvfp4rl_noalloc_scratch_bytes()
    # rank 136 (> 128) takes the general path, whose fp32 accumulator (M*N*4 bytes) exceeds the array
    M, N, K, r = 8192, 1024, 256, 136
    assert nv.workspace_bytes(nv.OP_LINEAR_W4A16, M, N, K, r) > cap
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.nvfp4_lora_linear_noalloc(p, M, K, p, p, p, N, p, p, r, 1.0, p, st) == 4  # NVFP4RL_ERR_WORKSPACE
