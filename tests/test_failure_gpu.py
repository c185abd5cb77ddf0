"""The device-side failure path: a bounded wait that runs out is reported to the host through the
library's status word, and the CUDA context stays usable (no fault, no hang: the self-test kernel
waits 1 ms on a barrier that nothing completes, then returns)."""
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
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def test_bounded_wait_timeout_is_reported_and_the_context_survives(nv):
    L = nv.lib()
    word = ctypes.c_uint32(0)
    assert L.nvfp4rl_device_status(ctypes.byref(word), 1) == 0    # clean start (and cleared)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.nvfp4rl_selftest_wait_timeout(stream) == 0           # launched
    st = L.nvfp4rl_device_status(ctypes.byref(word), 1)           # synchronizes, reads, clears
    assert st == 6 and word.value == 1                            # NVFP4RL_ERR_TIMEOUT, producer bit
    assert L.nvfp4rl_device_status(ctypes.byref(word), 0) == 0 and word.value == 0
    # the context still runs the library's kernels correctly
    W = synth.weight_bf16(64, 256, 0.02, 5, 1, outlier_frac=0.02)
    c, s, g = nv.nvfp4_quantize(P.dev_bf16(W))
    torch.cuda.synchronize()
    rc, rs, rg = oracle.quantize(W)
    assert np.array_equal(c.cpu().numpy(), rc) and np.array_equal(s.cpu().numpy(), rs)
    assert np.float32(g.cpu().numpy()[0]) == np.float32(rg)
