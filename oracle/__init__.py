"""CPU oracle for the NVFP4 rollout linear layer -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package. It wraps ``nvfp4_oracle.cpp``, a plain single-threaded
C++ restatement of the method (exact-table E2M1/E4M3 encoding, exact fp64
dequantization, fp64 accumulation). It shares no code with the CUDA library.

Python here only marshals arrays and splits independent rows (quantize,
RMSNorm) or output columns (GEMM) across host threads; ctypes releases the GIL
during each call, so the splits run in parallel without changing any result.
Every arithmetic step lives in the C++ file, which cites what it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.cpp")
_LIBDIR = os.path.join(_HERE, "lib")
_LIB = os.path.join(_LIBDIR, "libnvfp4_oracle.so")
_lock = threading.Lock()
_lib = None

BF16, F32 = 0, 1


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle with plain IEEE double/float arithmetic (no fast-math, no FMA contraction)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
                           "-shared", "-fPIC", "-o", tmp, src])
    os.replace(tmp, out)
    return out


def _declare(lib):
    d, i, f = ctypes.c_double, ctypes.c_int, ctypes.c_float
    i64, i32, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    sig = {
        "oracle_e2m1_value": (d, [i]),
        "oracle_e4m3_value": (d, [i]),
        "oracle_e4m3_encode_ratio": (i, [d, d]),
        "oracle_e2m1_encode": (i, [d, d]),
        "oracle_e2m1_encode_guided": (i, [d, d, i]),
        "oracle_amax": (f, [p, i, i64, i64]),
        "oracle_global_scale": (f, [f]),
        "oracle_quantize_rows": (None, [p, i, i64, i64, i64, f, p, p]),
        "oracle_quantize_guided_rows": (None, [p, i, i64, i64, i64, f, p, p, p]),
        "oracle_dequantize_rows": (None, [p, p, f, i64, i64, i64, p]),
        "oracle_quantize_record_rows": (None, [p, i, i64, i64, i64, f, p, p, p]),
        "oracle_e2m1_round_up": (i, [d, d]),
        "oracle_quantize_cached_rows": (None, [p, i, i64, i64, i64, f, p, p, p]),
        "oracle_ais": (None, [i64, p, p, p, d, d, d, d, p, p]),
        "oracle_attention_decode": (None, [p, p, p, f, p, p, f, p, i64, i64, i64, i64, i64, d, p]),
        "oracle_aqn_sigma": (d, [d, d, i64, i64]),
        "oracle_rmsnorm_aqn_rows": (None, [p, i64, i64, i64, p, p, f, f, p]),
        "oracle_lora_down": (None, [p, i64, i64, p, i32, p]),
        "oracle_linear_cols": (None, [p, i64, i64, p, p, f, i64, i64, i64, p, p, i32, d, p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def lib(path: str | None = None):
    """The loaded oracle library (built on first use)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def threads() -> int:
    return max(1, int(os.environ.get("ORACLE_THREADS", os.cpu_count() or 1)))


def _split(n: int, parts: int):
    parts = max(1, min(parts, n))
    step = (n + parts - 1) // parts
    return [(a, min(n, a + step)) for a in range(0, n, step)]


def _parallel(fn, n: int, nthreads: int | None = None):
    chunks = _split(n, nthreads or threads())
    if len(chunks) <= 1:
        for a, b in chunks:
            fn(a, b)
        return
    with ThreadPoolExecutor(len(chunks)) as ex:
        list(ex.map(lambda ab: fn(*ab), chunks))


# ---- scalar formats ---------------------------------------------------------------

def e2m1_value(code: int, L=None) -> float:
    return (L or lib()).oracle_e2m1_value(int(code))


def e4m3_value(byte: int, L=None) -> float:
    return (L or lib()).oracle_e4m3_value(int(byte))


def e4m3_encode_ratio(num: float, den: float, L=None) -> int:
    return (L or lib()).oracle_e4m3_encode_ratio(float(num), float(den))


def e2m1_encode(x: float, S: float, L=None) -> int:
    return (L or lib()).oracle_e2m1_encode(float(x), float(S))


def e2m1_encode_guided(x: float, S: float, up: int, L=None) -> int:
    return (L or lib()).oracle_e2m1_encode_guided(float(x), float(S), int(up))


# ---- tensors ------------------------------------------------------------------------

def _dtype_code(x: np.ndarray) -> int:
    if x.dtype == np.uint16:
        return BF16
    if x.dtype == np.float32:
        return F32
    raise TypeError("x must be bf16 bits (uint16) or float32")


def amax(x: np.ndarray, L=None, nthreads=None) -> np.float32:
    L = L or lib()
    x = np.ascontiguousarray(x)
    dt, n = _dtype_code(x), x.size
    parts = []
    _parallel(lambda a, b: parts.append(L.oracle_amax(_ptr(x), dt, a, b)), n, nthreads)
    return np.float32(max(parts) if parts else 0.0)


def global_scale(a: float, L=None) -> np.float32:
    return np.float32((L or lib()).oracle_global_scale(float(a)))


def quantize(x: np.ndarray, mask: np.ndarray | None = None, amax_in: float | None = None,
             L=None, nthreads=None):
    """NVFP4 encoding of a 2-D bf16-bits or fp32 array: (codes [rows, cols/2] u8, scales [rows, cols/16] u8, g f32)."""
    L = L or lib()
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    assert cols % 16 == 0
    dt = _dtype_code(x)
    a = amax(x, L, nthreads) if amax_in is None else np.float32(amax_in)
    g = global_scale(a, L)
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // 16), np.uint8)
    if mask is None:
        fn = lambda r0, r1: L.oracle_quantize_rows(_ptr(x), dt, cols, r0, r1, float(g), _ptr(codes), _ptr(scales))
    else:
        mask = np.ascontiguousarray(mask, dtype=np.uint32)
        assert mask.size * 32 >= rows * cols
        fn = lambda r0, r1: L.oracle_quantize_guided_rows(_ptr(x), dt, cols, r0, r1, float(g), _ptr(mask),
                                                          _ptr(codes), _ptr(scales))
    _parallel(fn, rows, nthreads)
    return codes, scales, g


def e2m1_round_up(x: float, S: float, L=None) -> int:
    return (L or lib()).oracle_e2m1_round_up(float(x), float(S))


def _rows_per_part(rows: int, cols: int, nthreads):
    """Row split whose part boundaries fall on 32-element mask words (each part owns whole words)."""
    step = 32 // np.gcd(cols, 32)
    parts = _split((rows + step - 1) // step, nthreads or threads())
    return [(a * step, min(rows, b * step)) for a, b in parts]


def quantize_record(x: np.ndarray, amax_in: float | None = None, L=None, nthreads=None):
    """Plain NVFP4 encoding plus the record of its rounding directions (TRACE rollout side):
    (codes, scales, g, mask) with mask bit i%32 of word i/32 set when element i was rounded up in
    magnitude."""
    L = L or lib()
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    assert cols % 16 == 0
    dt = _dtype_code(x)
    a = amax(x, L, nthreads) if amax_in is None else np.float32(amax_in)
    g = global_scale(a, L)
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // 16), np.uint8)
    mask = np.zeros((rows * cols + 31) // 32, np.uint32)
    chunks = _rows_per_part(rows, cols, nthreads)
    fn = lambda r0, r1: L.oracle_quantize_record_rows(_ptr(x), dt, cols, r0, r1, float(g), _ptr(codes),
                                                      _ptr(scales), _ptr(mask))
    if len(chunks) <= 1:
        for r0, r1 in chunks:
            fn(r0, r1)
    else:
        with ThreadPoolExecutor(len(chunks)) as ex:
            list(ex.map(lambda ab: fn(*ab), chunks))
    return codes, scales, g, mask


def quantize_cached(x: np.ndarray, mask: np.ndarray, scales: np.ndarray, g: float, L=None, nthreads=None):
    """Codes of x from a TRACE cache: the recorded scale bytes and g, rounding directions from mask."""
    L = L or lib()
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    assert cols % 16 == 0
    dt = _dtype_code(x)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    mask = np.ascontiguousarray(mask, dtype=np.uint32)
    assert scales.size == rows * cols // 16 and mask.size * 32 >= rows * cols
    codes = np.zeros((rows, cols // 2), np.uint8)
    fn = lambda r0, r1: L.oracle_quantize_cached_rows(_ptr(x), dt, cols, r0, r1, float(np.float32(g)),
                                                      _ptr(scales), _ptr(mask), _ptr(codes))
    _parallel(fn, rows, nthreads)
    return codes


def kv_quantize(x_bits: np.ndarray, g: float, L=None):
    """NVFP4 encoding of KV rows (bf16 bits [..., D], D % 16 == 0) with a given per-tensor g:
    (codes [..., D/2], scales [..., D/16])."""
    L = L or lib()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    D = x.shape[-1]
    rows = x.size // D
    codes = np.zeros(x.shape[:-1] + (D // 2,), np.uint8)
    scales = np.zeros(x.shape[:-1] + (D // 16,), np.uint8)
    _parallel(lambda r0, r1: L.oracle_quantize_rows(_ptr(x), BF16, D, r0, r1, float(np.float32(g)), _ptr(codes),
                                                    _ptr(scales)), rows)
    return codes, scales


def attention_decode(q_bits, k_codes, k_scales, gk, v_codes, v_scales, gv, lens, scale, L=None):
    """Decode attention over an NVFP4 KV cache in fp64: q [B, Hq, D] bf16 bits; caches [B, Lmax, Hkv, D/2]
    codes and [B, Lmax, Hkv, D/16] scales; lens [B] -> out [B, Hq, D] float64."""
    L = L or lib()
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    B, Hq, D = q.shape
    Lmax, Hkv = k_codes.shape[1], k_codes.shape[2]
    kc, ks, vc, vs = (np.ascontiguousarray(a, dtype=np.uint8) for a in (k_codes, k_scales, v_codes, v_scales))
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    assert Hq % Hkv == 0 and D % 16 == 0 and lens.size == B and np.all((lens > 0) & (lens <= Lmax))
    out = np.zeros((B, Hq, D))

    def part(b0, b1):
        L.oracle_attention_decode(_ptr(q[b0:b1]), _ptr(kc[b0:b1]), _ptr(ks[b0:b1]), float(np.float32(gk)),
                                  _ptr(vc[b0:b1]), _ptr(vs[b0:b1]), float(np.float32(gv)), _ptr(lens[b0:b1]),
                                  b1 - b0, Hq, Hkv, D, Lmax, float(scale), _ptr(out[b0:b1]))
    _parallel(part, B)
    return out


AIS_STATS = ("alpha", "alpha_ess", "alpha_mis", "alpha_var", "dbar", "cv2", "dsigma", "mean_w")


def ais(logp_rollout, logp_train, adv, C: float, delta: float, gamma: float, beta: float, L=None):
    """AIS mixing coefficient over a batch of tokens (fp32 inputs): (stats dict, rectified weights f64)."""
    L = L or lib()
    lr = np.ascontiguousarray(logp_rollout, dtype=np.float32)
    lt = np.ascontiguousarray(logp_train, dtype=np.float32)
    a = np.ascontiguousarray(adv, dtype=np.float32)
    n = lr.size
    assert lt.size == n and a.size == n
    stats = np.full(8, np.nan)
    w = np.zeros(n)
    L.oracle_ais(n, _ptr(lr), _ptr(lt), _ptr(a), float(C), float(delta), float(gamma), float(beta), _ptr(stats),
                 _ptr(w))
    return dict(zip(AIS_STATS, stats.tolist())), w


def quantize_rows_given_g(x: np.ndarray, g: float, rows, mask: np.ndarray | None = None, L=None):
    """Codes and scales of selected rows only, for a given per-tensor g (used for sampled parity)."""
    L = L or lib()
    x = np.ascontiguousarray(x)
    n_rows, cols = x.shape
    dt = _dtype_code(x)
    rows = np.asarray(rows, dtype=np.int64)
    codes = np.zeros((len(rows), cols // 2), np.uint8)
    scales = np.zeros((len(rows), cols // 16), np.uint8)
    for i, r in enumerate(rows):
        sub = np.ascontiguousarray(x[r:r + 1])
        c, s = codes[i:i + 1], scales[i:i + 1]
        if mask is None:
            L.oracle_quantize_rows(_ptr(sub), dt, cols, 0, 1, float(g), _ptr(c), _ptr(s))
        else:
            # the mask is indexed by the flat element index of the full tensor
            words = np.ascontiguousarray(mask[(r * cols) // 32:((r + 1) * cols + 31) // 32], dtype=np.uint32)
            assert (r * cols) % 32 == 0, "guided row sampling needs cols*row aligned to 32 elements"
            L.oracle_quantize_guided_rows(_ptr(sub), dt, cols, 0, 1, float(g), _ptr(words), _ptr(c), _ptr(s))
    return codes, scales


def dequantize(codes: np.ndarray, scales: np.ndarray, g: float, L=None, nthreads=None) -> np.ndarray:
    L = L or lib()
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    rows, cols = codes.shape[0], codes.shape[1] * 2
    out = np.empty((rows, cols), np.float64)
    _parallel(lambda a, b: L.oracle_dequantize_rows(_ptr(codes), _ptr(scales), float(g), cols, a, b, _ptr(out)),
              rows, nthreads)
    return out


def aqn_sigma(sigma0: float, sigmaK: float, k: int, K: int, L=None) -> float:
    return (L or lib()).oracle_aqn_sigma(float(sigma0), float(sigmaK), int(k), int(K))


def rmsnorm_aqn(x: np.ndarray, w: np.ndarray, eps: np.ndarray | None, sigma: float, delta: float,
                L=None, nthreads=None) -> np.ndarray:
    """y = (w + sigma*eps) * x / sqrt(mean(x^2) + delta) in fp64; x bf16 bits [M, H]."""
    L = L or lib()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    M, H = x.shape
    w = np.ascontiguousarray(w, dtype=np.float32)
    eps = None if eps is None else np.ascontiguousarray(eps, dtype=np.float32)
    y = np.empty((M, H), np.float64)
    _parallel(lambda a, b: L.oracle_rmsnorm_aqn_rows(_ptr(x), H, a, b, _ptr(w), _ptr(eps), float(sigma),
                                                     float(delta), _ptr(y)), M, nthreads)
    return y


def bf16_rows_f64(x_bits: np.ndarray) -> np.ndarray:
    """bf16 bits -> float64 (exact)."""
    return (np.ascontiguousarray(x_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def linear(xq: np.ndarray, xl: np.ndarray | None, codes: np.ndarray, scales: np.ndarray, g: float,
           A: np.ndarray | None, B: np.ndarray | None, s: float, L=None, nthreads=None) -> np.ndarray:
    """Y = xq deq(W)^T + s (xl A^T) B^T in fp64. xq, xl: [rows, K] float64; A [r, K], B [N, r] bf16 bits."""
    L = L or lib()
    xq = np.ascontiguousarray(xq, dtype=np.float64)
    nrows, K = xq.shape
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    N = codes.shape[0]
    r = 0 if A is None else A.shape[0]
    U = np.zeros((nrows, max(r, 1)), np.float64)
    Bc = None
    if r:
        xl = np.ascontiguousarray(xl, dtype=np.float64)
        A = np.ascontiguousarray(A, dtype=np.uint16)
        Bc = np.ascontiguousarray(B, dtype=np.uint16)
        L.oracle_lora_down(_ptr(xl), nrows, K, _ptr(A), r, _ptr(U))
    Y = np.empty((nrows, N), np.float64)
    _parallel(lambda a, b: L.oracle_linear_cols(_ptr(xq), nrows, K, _ptr(codes), _ptr(scales), float(g), N, a, b,
                                                _ptr(U), _ptr(Bc), r, float(s), _ptr(Y)), N, nthreads)
    return Y


def lora_linear_w4a16(x_bits, codes, scales, g, A, B, s, rows=None, L=None, nthreads=None):
    """W4A16 LoRA linear on bf16 activations (selected rows, default all)."""
    x_bits = np.asarray(x_bits)
    sel = x_bits if rows is None else x_bits[np.asarray(rows)]
    xd = bf16_rows_f64(sel)
    return linear(xd, xd, codes, scales, g, A, B, s, L, nthreads)


def lora_linear_w4a4(x_bits, codes, scales, g, A, B, s, rows=None, L=None, nthreads=None):
    """W4A4: the base GEMM takes deq(quantize(x)) with one per-tensor g_x over all of x;
    the LoRA branch takes the unquantized bf16 x."""
    L = L or lib()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    gx = global_scale(amax(x_bits, L, nthreads), L)
    rows = np.arange(x_bits.shape[0]) if rows is None else np.asarray(rows)
    xc, xs = quantize_rows_given_g(x_bits, gx, rows, L=L)
    xq = dequantize(xc, xs, gx, L, nthreads)
    xl = bf16_rows_f64(x_bits[rows])
    return linear(xq, xl, codes, scales, g, A, B, s, L, nthreads), (xc, xs, gx)
