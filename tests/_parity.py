"""Shared helpers of the GPU parity tests: moving synth arrays to the device and the
tolerances the parity bar fixes.

Tolerances (floating point; integer/byte results are compared bit for bit):
  * GEMM: per element |bf16(Y_gpu) - bf16(Y_ref)| <= max(1e-2 * rms(Y_ref), 1 bf16 ulp of Y_ref).
    1e-2 * rms is the stated bar; a large element's bf16 rounding alone can exceed it
    (half an ulp is 2^-9 |Y|), so one bf16 ulp of the element is also allowed.
  * RMSNorm: per element |y_gpu - y_ref| <= 1 bf16 ulp of y_ref, and
    rms(y_gpu - bf16(y_ref)) / rms(y_ref) <= 1e-3. The bf16 output's own rounding is
    about 1.5e-3 of rms, so the 1e-3 bar is read against the bf16-rounded reference,
    as for the GEMM.
"""
import numpy as np
import torch

import synth


def dev_bf16(bits: np.ndarray, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def dev(a: np.ndarray, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host_bits(t) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_f64(bits: np.ndarray) -> np.ndarray:
    return synth.bf16_to_f32(bits).astype(np.float64)


def bf16_round(v: np.ndarray) -> np.ndarray:
    return synth.bf16_to_f32(synth.bf16_bits(np.asarray(v, dtype=np.float64).astype(np.float32))).astype(np.float64)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def assert_gemm_close(y_gpu_bits: np.ndarray, y_ref: np.ndarray, what: str = ""):
    y = bf16_f64(y_gpu_bits)
    ref_b = bf16_round(y_ref)
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    tol = np.maximum(1e-2 * rms, bf16_ulp(y_ref))
    err = np.abs(y - ref_b)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance; worst at {i}: "
                             f"gpu {y[i]!r} ref {y_ref[i]!r} tol {tol[i]!r} (rms {rms:.4g})")
    return float(err.max() / rms) if rms else 0.0


def assert_rmsnorm_close(y_gpu_bits: np.ndarray, y_ref: np.ndarray, what: str = ""):
    y = bf16_f64(y_gpu_bits)
    err = np.abs(y - y_ref)
    ulp = bf16_ulp(y_ref)
    bad = err > ulp
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond 1 bf16 ulp; worst {err[bad].max()!r}"
    err_b = np.abs(y - bf16_round(y_ref))
    rel = float(np.sqrt(np.mean(err_b ** 2)) / np.sqrt(np.mean(y_ref ** 2)))
    assert rel <= 1e-3, f"{what}: rms error ratio {rel}"
    return rel
