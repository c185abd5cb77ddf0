"""Python binding of libnvfp4rl.so, the NVFP4 rollout-linear C ABI (include/nvfp4rl.h).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels. PyTorch provides device memory (outputs and workspaces are torch
tensors) and the current CUDA stream. The library must have been built
(``nvfp4_quantized_rl_gb300._build.build()`` or ``__graft_entry__.build()``);
importing the binding does not build it, and every call fails loudly when the
library or a GPU is missing -- there is no CPU fallback.

Functions carry the C names: nvfp4_amax, nvfp4_quantize, nvfp4_quantize_guided,
nvfp4_quantize_record, nvfp4_quantize_cached, nvfp4_quantize_batch, nvfp4_kv_append,
nvfp4_kv_decode_attention, ais_mixing, aqn_sigma, rmsnorm_aqn, rmsnorm_aqn_quantize, nvfp4_lora_linear,
nvfp4_lora_linear_w4a4.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

LIB_PATH = _build.LIB

OK = 0
BF16, F32 = 0, 1
(OP_QUANTIZE, OP_LINEAR_W4A16, OP_LINEAR_W4A4, OP_QUANTIZE_BATCH, OP_RMSNORM_QUANTIZE, OP_AIS, OP_KV_ATTENTION,
 OP_LINEAR_W4A4_QUANTIZED) = (0, 1, 2, 3, 4, 5, 6, 7)

_lock = threading.Lock()
_lib = None

# Every symbol include/nvfp4rl.h declares, with its C signature.
_SIGNATURES = None


def _signatures():
    c = ctypes
    p, i32, i64, f32, f64, sz = c.c_void_p, c.c_int32, c.c_int64, c.c_float, c.c_double, c.c_size_t
    return {
        "nvfp4_amax": (c.c_int, [p, i32, i64, p, p]),
        "nvfp4_quantize": (c.c_int, [p, i32, i64, i64, p, p, p, p, p, sz, p]),
        "nvfp4_quantize_guided": (c.c_int, [p, i32, i64, i64, p, p, p, p, p, p, sz, p]),
        "nvfp4_quantize_record": (c.c_int, [p, i32, i64, i64, p, p, p, p, p, p, sz, p]),
        "nvfp4_quantize_cached": (c.c_int, [p, i32, i64, i64, p, p, p, p, p]),
        "nvfp4_kv_append": (c.c_int, [p, p, i64, i64, i64, p, p, p, p, p, p, p, i64, p]),
        "nvfp4_kv_decode_attention": (c.c_int, [p, p, p, p, p, p, p, p, i64, i64, i64, i64, i64, c.c_float, p, p,
                                                 sz, p]),
        "ais_mixing": (c.c_int, [p, p, p, i64, c.c_float, c.c_float, c.c_float, c.c_float, p, p, p, sz, p]),
        "nvfp4_quantize_batch": (c.c_int, [i32, p, p, p, i32, p, p, p, p, sz, p]),
        "aqn_sigma": (f64, [f64, f64, i64, i64]),
        "rmsnorm_aqn": (c.c_int, [p, i64, i64, p, p, f32, f32, p, p]),
        "rmsnorm_aqn_quantize": (c.c_int, [p, i64, i64, p, p, f32, f32, p, p, p, p, p, sz, p]),
        "nvfp4_lora_linear": (c.c_int, [p, i64, i64, p, p, p, i64, p, p, i32, f32, p, i32, p, p, sz, p]),
        "nvfp4_lora_linear_w4a4": (c.c_int, [p, i64, i64, p, p, p, i64, p, p, i32, f32, p, i32, p, p, sz, p]),
        "nvfp4_lora_linear_noalloc": (c.c_int, [p, i64, i64, p, p, p, i64, p, p, i32, f32, p, p]),
        "nvfp4_lora_linear_w4a4_quantized": (c.c_int, [p, p, p, p, i64, i64, p, p, p, i64, p, p, i32, f32, p, i32, p,
                                                       p, sz, p]),
        "nvfp4rl_noalloc_scratch_bytes": (sz, []),
        "nvfp4rl_workspace_bytes": (sz, [i32, i64, i64, i64, i32, i32]),
        "nvfp4rl_status_string": (c.c_char_p, [c.c_int]),
        "nvfp4rl_device_status": (c.c_int, [p, i32]),
        "nvfp4rl_selftest_wait_timeout": (c.c_int, [p]),
        "nvfp4rl_kernel_launches": (c.c_uint64, []),
    }


class Nvfp4rlError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libnvfp4rl.so is not built ({LIB_PATH}); run nvfp4_quantized_rl_gb300._build.build()")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _signatures().items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().nvfp4rl_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != OK:
        raise Nvfp4rlError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t, stream=None):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return ctypes.c_void_p(stream.cuda_stream)


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("nvfp4rl works on CUDA tensors only (no CPU path)")


def workspace_bytes(op: int, M: int, N: int, K: int, r: int = 0, groups: int = 0) -> int:
    return int(lib().nvfp4rl_workspace_bytes(op, M, N, K, r, groups))


def kernel_launches() -> int:
    return int(lib().nvfp4rl_kernel_launches())


def device_status(clear: bool = True) -> int:
    word = ctypes.c_uint32(0)
    st = lib().nvfp4rl_device_status(ctypes.byref(word), 1 if clear else 0)
    return st, int(word.value)


def aqn_sigma(sigma0: float, sigmaK: float, k: int, K: int) -> float:
    """AQN exponential schedule sigma_k = sigma0 * (sigmaK / sigma0)^(k / K) (host)."""
    return float(lib().aqn_sigma(float(sigma0), float(sigmaK), int(k), int(K)))


def _empty(shape, dtype, device):
    import torch
    return torch.empty(shape, dtype=dtype, device=device)


def _bits16(t):
    """bf16 tensors are passed as their bit patterns; any 2-byte dtype view works."""
    import torch
    if t is None:
        return None
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"expected a bf16 tensor, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t


def nvfp4_amax(x, out=None, stream=None):
    """max |x| of a bf16 or fp32 CUDA tensor (numel multiple of 16) -> fp32 [1]."""
    import torch
    _require_cuda(x)
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    dt = BF16 if x.dtype == torch.bfloat16 else F32 if x.dtype == torch.float32 else None
    if dt is None:
        raise TypeError("x must be bf16 or fp32")
    out = _empty((1,), torch.float32, x.device) if out is None else out
    _check(lib().nvfp4_amax(_ptr(x), dt, x.numel(), _ptr(out), _stream(x, stream)), "nvfp4_amax")
    return out


def nvfp4_quantize(x, amax_in=None, codes=None, scales=None, g=None, workspace=None, stream=None):
    """NVFP4 block quantization of a 2-D bf16 or fp32 CUDA tensor -> (codes u8 [R, C/2], scales u8 [R, C/16], g f32 [1])."""
    return _quantize(x, None, amax_in, codes, scales, g, workspace, stream)


def nvfp4_quantize_guided(x, mask, amax_in=None, codes=None, scales=None, g=None, workspace=None, stream=None):
    """Guided NVFP4 quantization: mask (int32/uint32 words, bit i%32 of word i//32) picks the rounding direction."""
    return _quantize(x, mask, amax_in, codes, scales, g, workspace, stream)


def nvfp4_quantize_record(x, amax_in=None, codes=None, scales=None, g=None, record=None, workspace=None,
                          stream=None):
    """nvfp4_quantize plus the record of its rounding directions -> (codes, scales, g, record int32
    [ceil(R*C/32)]): bit i%32 of word i//32 is 1 where element i was rounded up in magnitude."""
    import torch
    rows, cols = x.shape if x.dim() == 2 else (0, 0)
    record = _empty(((rows * cols + 31) // 32,), torch.int32, x.device) if record is None else record
    codes, scales, g = _quantize(x, None, amax_in, codes, scales, g, workspace, stream, record=record)
    return codes, scales, g, record


def nvfp4_quantize_cached(x, mask, scales, g, codes=None, stream=None):
    """Codes of x from a cache: the given scale bytes and g (CUDA tensors) with the rounding
    directions of mask, in one pass -> codes u8 [R, C/2]."""
    import torch
    _require_cuda(x, mask, scales, g)
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D tensor")
    dt = {torch.bfloat16: BF16, torch.float32: F32}.get(x.dtype)
    if dt is None:
        raise TypeError("x must be bf16 or fp32")
    rows, cols = x.shape
    codes = _empty((rows, cols // 2), torch.uint8, x.device) if codes is None else codes
    st = lib().nvfp4_quantize_cached(_ptr(x), dt, rows, cols, _ptr(mask), _ptr(scales), _ptr(g), _ptr(codes),
                                     _stream(x, stream))
    _check(st, "nvfp4_quantize_cached")
    return codes


def nvfp4_kv_append(k, v, pos, gk, gv, k_codes, k_scales, v_codes, v_scales, stream=None):
    """Writes one token's keys and values per sequence (bf16 [B, Hkv, D]) into an NVFP4 KV cache at
    rows pos [B] (int32): caches are uint8 [B, Lmax, Hkv, D/2] codes and [B, Lmax, Hkv, D/16] scales;
    gk, gv fp32 [1] CUDA tensors."""
    _require_cuda(k, v, pos, gk, gv, k_codes, k_scales, v_codes, v_scales)
    _bits16(k)
    _bits16(v)
    B, Hkv, D = k.shape
    Lmax = k_codes.shape[1]
    st = lib().nvfp4_kv_append(_ptr(k), _ptr(v), B, Hkv, D, _ptr(pos), _ptr(gk), _ptr(gv), _ptr(k_codes),
                               _ptr(k_scales), _ptr(v_codes), _ptr(v_scales), Lmax, _stream(k, stream))
    _check(st, "nvfp4_kv_append")


def nvfp4_kv_decode_attention(q, k_codes, k_scales, gk, v_codes, v_scales, gv, lens, scale, out=None,
                              workspace=None, stream=None):
    """One decode step of attention over an NVFP4 KV cache: q bf16 [B, Hq, 128] -> out bf16 [B, Hq, 128]."""
    import torch
    _require_cuda(q, k_codes, k_scales, gk, v_codes, v_scales, gv, lens, out, workspace)
    _bits16(q)
    B, Hq, D = q.shape
    Lmax, Hkv = k_codes.shape[1], k_codes.shape[2]
    out = _empty((B, Hq, D), torch.bfloat16, q.device) if out is None else out
    need = workspace_bytes(OP_KV_ATTENTION, B, Hkv, Lmax)
    if workspace is None and need > 0:
        workspace = _empty((need,), torch.uint8, q.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().nvfp4_kv_decode_attention(_ptr(q), _ptr(k_codes), _ptr(k_scales), _ptr(gk), _ptr(v_codes),
                                         _ptr(v_scales), _ptr(gv), _ptr(lens), B, Hq, Hkv, D, Lmax, float(scale),
                                         _ptr(out), _ptr(workspace), wsb, _stream(q, stream))
    _check(st, "nvfp4_kv_decode_attention")
    return out


AIS_STATS = ("alpha", "alpha_ess", "alpha_mis", "alpha_var", "dbar", "cv2", "dsigma", "mean_w")


def ais_mixing(logp_rollout, logp_train, adv, C: float, delta: float, gamma: float, beta: float, weights=True,
               w_out=None, stats=None, workspace=None, stream=None):
    """AIS correction of a token batch (fp32 CUDA tensors of n elements) -> (stats fp64 [8] in the order
    of AIS_STATS, rectified weights fp32 [n] or None when weights is False)."""
    import torch
    _require_cuda(logp_rollout, logp_train, adv, w_out, stats, workspace)
    for t in (logp_rollout, logp_train, adv):
        if t.dtype != torch.float32 or not t.is_contiguous() or t.numel() != logp_rollout.numel():
            raise ValueError("log-probs and advantages must be contiguous fp32 tensors of one size")
    n = logp_rollout.numel()
    dev = logp_rollout.device
    if weights and w_out is None:
        w_out = _empty((n,), torch.float32, dev)
    stats = _empty((8,), torch.float64, dev) if stats is None else stats
    if workspace is None:
        workspace = _empty((workspace_bytes(OP_AIS, 0, 0, 0),), torch.uint8, dev)
    st = lib().ais_mixing(_ptr(logp_rollout), _ptr(logp_train), _ptr(adv), n, float(C), float(delta), float(gamma),
                          float(beta), _ptr(w_out) if weights else None, _ptr(stats), _ptr(workspace),
                          workspace.numel() * workspace.element_size(), _stream(logp_rollout, stream))
    _check(st, "ais_mixing")
    return stats, (w_out if weights else None)


def nvfp4_quantize_batch(xs, codes=None, scales=None, g=None, workspace=None, stream=None):
    """NVFP4 quantization of a list of contiguous 2-D CUDA tensors of one dtype (bf16 or fp32) in one
    call, each with its own g -> (codes list, scales list, g list); outputs may be given as lists."""
    import torch
    xs = list(xs)
    n = len(xs)
    if n == 0:
        return [], [], []
    _require_cuda(*xs)
    dt = {torch.bfloat16: BF16, torch.float32: F32}.get(xs[0].dtype)
    if dt is None or any(t.dtype != xs[0].dtype for t in xs):
        raise TypeError("all tensors must be bf16, or all fp32")
    for t in xs:
        if t.dim() != 2 or not t.is_contiguous():
            raise ValueError("every tensor must be contiguous and 2-D")
    dev = xs[0].device
    codes = [_empty((t.shape[0], t.shape[1] // 2), torch.uint8, dev) for t in xs] if codes is None else list(codes)
    scales = [_empty((t.shape[0], t.shape[1] // 16), torch.uint8, dev) for t in xs] if scales is None else list(scales)
    g = [_empty((1,), torch.float32, dev) for _ in xs] if g is None else list(g)
    if workspace is None:
        workspace = _empty((workspace_bytes(OP_QUANTIZE_BATCH, n, 0, 0),), torch.uint8, dev)
    P = ctypes.c_void_p * n
    I64 = ctypes.c_int64 * n
    st = lib().nvfp4_quantize_batch(n, P(*[t.data_ptr() for t in xs]), I64(*[t.shape[0] for t in xs]),
                                    I64(*[t.shape[1] for t in xs]), dt, P(*[t.data_ptr() for t in codes]),
                                    P(*[t.data_ptr() for t in scales]), P(*[t.data_ptr() for t in g]), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(xs[0], stream))
    _check(st, "nvfp4_quantize_batch")
    return codes, scales, g


def _quantize(x, mask, amax_in, codes, scales, g, workspace, stream, record=None):
    import torch
    _require_cuda(x, mask, amax_in, record)
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D tensor")
    if x.dtype == torch.bfloat16:
        dt = BF16
    elif x.dtype == torch.float32:
        dt = F32
    else:
        raise TypeError("x must be bf16 or fp32")
    rows, cols = x.shape
    dev = x.device
    codes = _empty((rows, cols // 2), torch.uint8, dev) if codes is None else codes
    scales = _empty((rows, cols // 16), torch.uint8, dev) if scales is None else scales
    g = _empty((1,), torch.float32, dev) if g is None else g
    if workspace is None and amax_in is None:
        workspace = _empty((workspace_bytes(OP_QUANTIZE, 0, 0, 0),), torch.uint8, dev)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    L = lib()
    if record is not None:
        st = L.nvfp4_quantize_record(_ptr(x), dt, rows, cols, _ptr(codes), _ptr(scales), _ptr(g), _ptr(record),
                                     _ptr(amax_in), _ptr(workspace), wsb, _stream(x, stream))
        _check(st, "nvfp4_quantize_record")
    elif mask is None:
        st = L.nvfp4_quantize(_ptr(x), dt, rows, cols, _ptr(codes), _ptr(scales), _ptr(g), _ptr(amax_in),
                              _ptr(workspace), wsb, _stream(x, stream))
        _check(st, "nvfp4_quantize")
    else:
        st = L.nvfp4_quantize_guided(_ptr(x), dt, rows, cols, _ptr(mask), _ptr(codes), _ptr(scales), _ptr(g),
                                     _ptr(amax_in), _ptr(workspace), wsb, _stream(x, stream))
        _check(st, "nvfp4_quantize_guided")
    return codes, scales, g


def rmsnorm_aqn(x, w, eps=None, sigma: float = 0.0, delta: float = 1e-6, out=None, stream=None):
    """y = (w + sigma*eps) * x / sqrt(mean(x^2) + delta), bf16 x [M, H] -> bf16 y."""
    import torch
    _require_cuda(x, w, eps)
    _bits16(x)
    M, H = x.shape
    out = _empty((M, H), torch.bfloat16, x.device) if out is None else out
    st = lib().rmsnorm_aqn(_ptr(x), M, H, _ptr(w), _ptr(eps), float(sigma), float(delta), _ptr(out), _stream(x, stream))
    _check(st, "rmsnorm_aqn")
    return out


def rmsnorm_aqn_quantize(x, w, eps=None, sigma: float = 0.0, delta: float = 1e-6, out=None, codes=None, scales=None,
                         g=None, workspace=None, stream=None):
    """rmsnorm_aqn of bf16 x [M, H] and the NVFP4 quantization of its output in one call
    -> (y bf16 [M, H], codes u8 [M, H/2], scales u8 [M, H/16], g f32 [1])."""
    import torch
    _require_cuda(x, w, eps)
    _bits16(x)
    M, H = x.shape
    dev = x.device
    out = _empty((M, H), torch.bfloat16, dev) if out is None else out
    codes = _empty((M, H // 2), torch.uint8, dev) if codes is None else codes
    scales = _empty((M, H // 16), torch.uint8, dev) if scales is None else scales
    g = _empty((1,), torch.float32, dev) if g is None else g
    if workspace is None:
        workspace = _empty((workspace_bytes(OP_RMSNORM_QUANTIZE, 0, 0, 0),), torch.uint8, dev)
    st = lib().rmsnorm_aqn_quantize(_ptr(x), M, H, _ptr(w), _ptr(eps), float(sigma), float(delta), _ptr(out),
                                    _ptr(codes), _ptr(scales), _ptr(g), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(x, stream))
    _check(st, "rmsnorm_aqn_quantize")
    return out, codes, scales, g


def _linear(fn_name, op, x, codes, scales, g, A, B, s, group_offsets, num_groups, out, workspace, stream):
    import torch
    _require_cuda(x, codes, scales, g, A, B, group_offsets)
    _bits16(x), _bits16(A), _bits16(B)
    M, K = x.shape
    N = codes.shape[-2]
    r = 0 if A is None else A.shape[0]
    G = 0 if group_offsets is None else (num_groups if num_groups else group_offsets.numel() - 1)
    out = _empty((M, N), torch.bfloat16, x.device) if out is None else out
    if workspace is None:
        workspace = _empty((max(workspace_bytes(op, M, N, K, r, G), 16),), torch.uint8, x.device)
    wsb = workspace.numel() * workspace.element_size()
    st = getattr(lib(), fn_name)(_ptr(x), M, K, _ptr(codes), _ptr(scales), _ptr(g), N, _ptr(A), _ptr(B), r,
                                 float(s), _ptr(group_offsets), G, _ptr(out), _ptr(workspace), wsb, _stream(x, stream))
    _check(st, fn_name)
    return out


def nvfp4_lora_linear(x, codes, scales, g, A=None, B=None, s: float = 1.0, out=None, workspace=None, stream=None):
    """W4A16: Y = x deq(W)^T + s (x A^T) B^T (bf16 x [M, K]; codes [N, K/2], scales [N, K/16], g [1])."""
    return _linear("nvfp4_lora_linear", OP_LINEAR_W4A16, x, codes, scales, g, A, B, s, None, 0, out, workspace, stream)


def nvfp4_lora_linear_w4a4(x, codes, scales, g, A=None, B=None, s: float = 1.0, group_offsets=None,
                           num_groups: int = 0, out=None, workspace=None, stream=None):
    """W4A4: x quantized on the fly (per-tensor g_x); grouped when group_offsets (int32 [G+1]) is given,
    with codes [G, N, K/2], scales [G, N, K/16], g [G]."""
    return _linear("nvfp4_lora_linear_w4a4", OP_LINEAR_W4A4, x, codes, scales, g, A, B, s, group_offsets,
                   num_groups, out, workspace, stream)


def nvfp4_lora_linear_w4a4_quantized(x, x_codes, x_scales, x_g, codes, scales, g, A=None, B=None, s: float = 1.0,
                                     group_offsets=None, num_groups: int = 0, out=None, workspace=None, stream=None):
    """W4A4 on activations already in NVFP4 (x_codes [M, K/2], x_scales [M, K/16], x_g [1], e.g. from
    rmsnorm_aqn_quantize); x is the bf16 activation the LoRA branch reads (may be None without LoRA)."""
    import torch
    _require_cuda(x_codes, x_scales, x_g, codes, scales, g, A, B, group_offsets, x)
    _bits16(x), _bits16(A), _bits16(B)
    M, K2 = x_codes.shape
    K = 2 * K2
    N = codes.shape[-2]
    r = 0 if A is None else A.shape[0]
    G = 0 if group_offsets is None else (num_groups if num_groups else group_offsets.numel() - 1)
    out = _empty((M, N), torch.bfloat16, x_codes.device) if out is None else out
    if workspace is None:
        workspace = _empty((max(workspace_bytes(OP_LINEAR_W4A4_QUANTIZED, M, N, K, r, G), 16),), torch.uint8,
                           x_codes.device)
    wsb = workspace.numel() * workspace.element_size()
    st = lib().nvfp4_lora_linear_w4a4_quantized(_ptr(x), _ptr(x_codes), _ptr(x_scales), _ptr(x_g), M, K, _ptr(codes),
                                                _ptr(scales), _ptr(g), N, _ptr(A), _ptr(B), r, float(s),
                                                _ptr(group_offsets), G, _ptr(out), _ptr(workspace), wsb,
                                                _stream(x_codes, stream))
    _check(st, "nvfp4_lora_linear_w4a4_quantized")
    return out


def nvfp4_lora_linear_noalloc(x, codes, scales, g, A=None, B=None, s: float = 1.0, out=None, stream=None):
    """W4A16 LoRA linear without a workspace argument, for callers that cannot allocate device memory:
    the library's fixed 4 MiB device array serves as scratch (see include/nvfp4rl.h). Outputs are still
    the caller's (allocated here with torch only when `out` is None)."""
    import torch
    _require_cuda(x, codes, scales, g, A, B)
    _bits16(x), _bits16(A), _bits16(B)
    M, K = x.shape
    N = codes.shape[-2]
    r = 0 if A is None else A.shape[0]
    out = _empty((M, N), torch.bfloat16, x.device) if out is None else out
    st = lib().nvfp4_lora_linear_noalloc(_ptr(x), M, K, _ptr(codes), _ptr(scales), _ptr(g), N, _ptr(A), _ptr(B), r,
                                         float(s), _ptr(out), _stream(x, stream))
    _check(st, "nvfp4_lora_linear_noalloc")
    return out
