"""The C-ABI library builds, loads and exports every symbol include/nvfp4rl.h declares;
host-side validation rejects bad arguments before touching a GPU (no compute calls here)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4rl.h")


@pytest.fixture(scope="module")
def nv():
    from nvfp4_quantized_rl_gb300 import _build
    _build.build()
    import nvfp4_quantized_rl_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"NVFP4RL_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    for required in ("nvfp4_quantize", "nvfp4_quantize_guided", "nvfp4_quantize_batch", "rmsnorm_aqn",
                     "nvfp4_quantize_record", "nvfp4_quantize_cached", "ais_mixing", "nvfp4_kv_append",
                     "nvfp4_kv_decode_attention",
                     "rmsnorm_aqn_quantize", "nvfp4_lora_linear",
                     "nvfp4_lora_linear_w4a4", "aqn_sigma"):
        assert required in names


def test_library_exports_every_declared_symbol(nv):
    L = ctypes.CDLL(nv.LIB_PATH)
    names = declared_functions()
    assert names
    for name in names:
        assert hasattr(L, name), f"{name} declared in the header but not exported"
    # and the binding declares a ctypes signature for each of them
    assert set(names) == set(nv._signatures())


def test_aqn_sigma_matches_the_oracle(nv):
    for k in range(11):
        assert nv.aqn_sigma(1e-2, 5e-4, k, 10) == pytest.approx(oracle.aqn_sigma(1e-2, 5e-4, k, 10), rel=1e-15)
    assert np.isnan(nv.aqn_sigma(1e-2, 5e-4, 0, 0))


def test_status_strings(nv):
    for s in range(10):
        assert nv.status_string(s) and nv.status_string(s) != "unknown status"


def test_workspace_bytes(nv):
    assert nv.workspace_bytes(nv.OP_QUANTIZE, 0, 0, 0) >= 4
    w16 = nv.workspace_bytes(nv.OP_LINEAR_W4A16, 64, 3584, 3584, 32)
    w4 = nv.workspace_bytes(nv.OP_LINEAR_W4A4, 64, 3584, 3584, 32)
    assert w16 >= 64 * 32 * 2 and w4 >= 64 * 3584 // 2 + 64 * 3584 // 16
    assert nv.workspace_bytes(7, 1, 1, 1) == 0 and nv.workspace_bytes(nv.OP_LINEAR_W4A16, -1, 1, 1) == 0


# Fake, never-dereferenced addresses: validation fails before any device access.
A0, A1, A2, A3, A4 = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000


def _q(nv, x=A0, dtype=0, rows=4, cols=32, codes=A1, scales=A2, g=A3, amax=None, ws=A4, wsb=256):
    return nv.lib().nvfp4_quantize(x, dtype, rows, cols, codes, scales, g, amax, ws, wsb, None)


def test_quantize_validation(nv):
    assert _q(nv, x=None) == 1                 # null input
    assert _q(nv, dtype=3) == 1                # bad dtype
    assert _q(nv, rows=-1) == 1
    assert _q(nv, cols=24) == 3                # not a multiple of 16
    assert _q(nv, x=A0 + 8) == 2               # misaligned
    assert _q(nv, codes=A0) == 7               # output overlaps input
    assert _q(nv, ws=None) == 4                # no workspace and no amax_in
    assert _q(nv, wsb=8) == 4                  # workspace too small
    g = nv.lib().nvfp4_quantize_guided(A0, 0, 4, 32, None, A1, A2, A3, None, A4, 256, None)
    assert g == 1                              # guided without a mask


def test_quantize_record_validation(nv):
    rec = nv.lib().nvfp4_quantize_record
    A5 = A4 + 0x10000
    assert rec(A0, 0, 4, 32, A1, A2, A3, None, None, A4, 256, None) == 1      # no record buffer
    assert rec(A0, 0, 4, 32, A1, A2, A3, A5 + 4, None, A4, 256, None) == 2    # misaligned record
    assert rec(A0, 0, 4, 32, A1, A2, A3, A1, None, A4, 256, None) == 7        # record over the codes
    assert rec(A0, 0, 4, 32, A1, A2, A3, A0 + 16, None, A4, 256, None) == 7   # record over the input
    assert rec(A0, 0, 4, 32, A1, A2, A3, A5, None, None, 0, None) == 4        # no workspace, no amax_in
    assert rec(A0, 0, 4, 24, A1, A2, A3, A5, None, A4, 256, None) == 3
    assert rec(A0, 0, 0, 32, A1, A2, A3, None, None, None, 0, None) == 0      # empty: nothing to do


def test_quantize_cached_validation(nv):
    cac = nv.lib().nvfp4_quantize_cached
    A5 = A4 + 0x10000
    assert cac(A0, 0, 4, 32, None, A2, A3, A1, None) == 1      # no mask
    assert cac(A0, 0, 4, 32, A5, None, A3, A1, None) == 1      # no scales
    assert cac(A0, 0, 4, 32, A5, A2, None, A1, None) == 1      # no g
    assert cac(A0, 5, 4, 32, A5, A2, A3, A1, None) == 1        # bad dtype
    assert cac(A0, 0, 4, 40, A5, A2, A3, A1, None) == 3        # cols not a multiple of 16
    assert cac(A0, 0, 4, 32, A5 + 8, A2, A3, A1, None) == 2    # misaligned mask
    assert cac(A0, 0, 4, 32, A5, A2, A3 + 2, A1, None) == 2    # misaligned g
    assert cac(A0, 0, 4, 32, A5, A2, A3, A5, None) == 7        # codes over the mask
    assert cac(A0, 0, 4, 32, A5, A2, A3, A2, None) == 7        # codes over the scales
    assert cac(A0, 0, 0, 32, None, None, None, None, None) == 0  # empty: nothing to do


def test_ais_validation(nv):
    ais = nv.lib().ais_mixing
    W = 0x90000  # workspace
    wsb = nv.workspace_bytes(nv.OP_AIS, 0, 0, 0)
    assert wsb >= 1024 * 64
    ok = dict(lr=A0, lt=A1, adv=A2, n=64, C=2.0, d=0.05, g=0.5, b=1.0, w=A3, st=A4, ws=W, wsb=wsb)

    def call(**k):
        a = {**ok, **k}
        return ais(a["lr"], a["lt"], a["adv"], a["n"], a["C"], a["d"], a["g"], a["b"], a["w"], a["st"], a["ws"],
                   a["wsb"], None)
    assert call(n=-1) == 1
    assert call(n=0, lr=None) == 0                  # empty batch: nothing to do
    assert call(C=0.0) == 1 and call(d=-1.0) == 1 and call(g=0.0) == 1 and call(b=-0.5) == 1
    assert call(C=float("inf")) == 1 and call(b=float("nan")) == 1
    assert call(adv=None) == 1 and call(st=None) == 1
    assert call(lt=A1 + 4) == 2 and call(w=A3 + 8) == 2 and call(st=A4 + 4) == 2
    assert call(ws=None) == 4 and call(wsb=16) == 4
    assert call(w=A0 + 64) == 7                     # weights over an input
    assert call(st=A3 + 8) == 7                     # statistics over the weights
    assert call(ws=A2) == 7                         # workspace over an input


def test_kv_validation(nv):
    app, att = nv.lib().nvfp4_kv_append, nv.lib().nvfp4_kv_decode_attention
    C0, C1, C2, C3 = 0x100000, 0x200000, 0x300000, 0x400000  # caches of 2 x 8 x 2 rows
    ok = dict(k=A0, v=A1, B=2, H=2, D=128, pos=A2, gk=A3, gv=A3 + 4, kc=C0, ks=C1, vc=C2, vs=C3, L=8)

    def ap(**kw):
        a = {**ok, **kw}
        return app(a["k"], a["v"], a["B"], a["H"], a["D"], a["pos"], a["gk"], a["gv"], a["kc"], a["ks"], a["vc"],
                   a["vs"], a["L"], None)
    assert ap(B=-1) == 1 and ap(H=0) == 1 and ap(L=0) == 1
    assert ap(D=24) == 3
    assert ap(B=0, k=None) == 0
    assert ap(pos=None) == 1 and ap(gv=None) == 1
    assert ap(k=A0 + 8) == 2 and ap(pos=A2 + 2) == 2 and ap(ks=C1 + 4) == 2
    assert ap(vc=C0 + 16) == 7          # two caches overlap
    assert ap(kc=A0) == 7               # a cache over an input
    wsb = nv.workspace_bytes(nv.OP_KV_ATTENTION, 64, 4, 8192)
    assert wsb > 0 and nv.workspace_bytes(nv.OP_KV_ATTENTION, 4096, 4, 64) == 0  # one span: no merge buffer
    ok2 = dict(q=A0, kc=C0, ks=C1, gk=A3, vc=C2, vs=C3, gv=A3 + 4, lens=A2, B=2, Hq=4, H=2, D=128, L=8,
               scale=0.1, out=A4, ws=None, wsb=0)

    def at(**kw):
        a = {**ok2, **kw}
        return att(a["q"], a["kc"], a["ks"], a["gk"], a["vc"], a["vs"], a["gv"], a["lens"], a["B"], a["Hq"], a["H"],
                   a["D"], a["L"], a["scale"], a["out"], a["ws"], a["wsb"], None)
    assert at(D=64) == 3                # head dimension 128 only
    assert at(Hq=5) == 3                # Hq not a multiple of Hkv
    assert at(Hq=34, H=2) == 3          # more than 16 query heads per KV head
    assert at(scale=float("inf")) == 1 and at(lens=None) == 1
    assert at(out=A4 + 8) == 2
    assert at(out=A0 + 64) == 7         # output over the query
    assert at(B=64, H=4, Hq=28, L=8192, out=A4) == 4  # several spans need the merge buffer


def _qb(nv, n=2, xs=(A0, A0 + 0x1000), rows=(4, 8), cols=(32, 64), dtype=0, codes=(A1, A1 + 0x1000),
        scales=(A2, A2 + 0x1000), g=(A3, A3 + 0x100), ws=A4, wsb=256):
    P, I = ctypes.c_void_p * len(xs), ctypes.c_int64 * len(xs)
    return nv.lib().nvfp4_quantize_batch(n, P(*xs), I(*rows), I(*cols), dtype, P(*codes), P(*scales), P(*g), ws,
                                         wsb, None)


def test_quantize_batch_validation(nv):
    assert nv.workspace_bytes(nv.OP_QUANTIZE_BATCH, 300, 0, 0) >= 300 * 4
    assert nv.workspace_bytes(nv.OP_QUANTIZE_BATCH, 5000, 0, 0) == 0  # more than 4096 tensors
    assert _qb(nv, n=-1) == 1
    assert _qb(nv, n=0) == 0                                           # nothing to do
    assert _qb(nv, dtype=2) == 1
    assert _qb(nv, rows=(4, -1)) == 1
    assert _qb(nv, cols=(32, 40)) == 3                                 # not a multiple of 16
    assert _qb(nv, xs=(A0, A0 + 8)) == 2                               # misaligned input
    assert _qb(nv, g=(A3, A3 + 2)) == 2                                # misaligned g
    assert _qb(nv, ws=None) == 4
    assert _qb(nv, wsb=16) == 4
    assert _qb(nv, codes=(A1, A1)) == 7                                # two outputs in one place
    assert _qb(nv, scales=(A2, A0 + 0x1000)) == 7                      # an output over an input
    assert _qb(nv, g=(A3, A4)) == 7                                    # an output over the workspace
    assert _qb(nv, rows=(0, 0)) == 0                                   # all tensors empty: no-op


def _lin(nv, fn="nvfp4_lora_linear", x=A0, M=8, K=512, codes=A1, scales=A2, g=A3, N=256, A=None, B=None, r=0,
         s=2.0, off=None, G=0, y=A4, ws=0x60000, wsb=1 << 30):
    return getattr(nv.lib(), fn)(x, M, K, codes, scales, g, N, A, B, r, s, off, G, y, ws, wsb, None)


def test_linear_validation(nv):
    assert _lin(nv, x=None) == 1
    assert _lin(nv, r=16) == 1                 # r > 0 without A, B
    assert _lin(nv, r=300, A=0x70000, B=0x80000) == 1
    assert _lin(nv, K=500) == 3                # K not a multiple of 256
    assert _lin(nv, N=200) == 3                # N not a multiple of 128
    assert _lin(nv, x=A0 + 4) == 2
    assert _lin(nv, y=A0) == 7                 # y overlaps x
    assert _lin(nv, wsb=16) == 4
    assert _lin(nv, off=0x90000, G=4) == 3     # grouped W4A16 is not provided
    assert _lin(nv, fn="nvfp4_lora_linear_w4a4", off=0x90000, G=0) == 1
    assert _lin(nv, fn="nvfp4_lora_linear_w4a4", off=0x90000, G=4, r=16, A=0x70000, B=0x80000) == 1
    assert _lin(nv, s=float("nan")) == 1
    # LoRA ranks: 0 or a multiple of 16 up to 128 (both tcgen05 kernels); others in [0, 256] are
    # unsupported shapes, above 256 invalid
    for fn in ("nvfp4_lora_linear", "nvfp4_lora_linear_w4a4"):
        for bad_r in (8, 24, 136, 144, 256):
            assert _lin(nv, fn=fn, r=bad_r, A=0x70000, B=0x80000) == 3, (fn, bad_r)
    assert _lin(nv, M=65536) == 3              # above the largest M
    for op in (nv.OP_LINEAR_W4A16, nv.OP_LINEAR_W4A4):
        assert nv.workspace_bytes(op, 64, 256, 512, 8) == 0
        assert nv.workspace_bytes(op, 64, 256, 512, 136) == 0
        for r in (0, 16, 64, 128):
            assert nv.workspace_bytes(op, 200, 256, 512, r) > 0, (op, r)


def _linq(nv, x=A0, xc=0x90000, xs=0xA0000, xg=0xB0000, M=8, K=512, codes=A1, scales=A2, g=A3, N=256, A=None,
          B=None, r=0, s=2.0, off=None, G=0, y=A4, ws=0x60000, wsb=1 << 30):
    return nv.lib().nvfp4_lora_linear_w4a4_quantized(x, xc, xs, xg, M, K, codes, scales, g, N, A, B, r, s, off, G, y,
                                                     ws, wsb, None)


def test_linear_w4a4_quantized_validation(nv):
    assert _linq(nv, xc=None) == 1                  # the activation codes are required
    assert _linq(nv, xg=None) == 1
    assert _linq(nv, x=None, r=16, A=0x70000, B=0x80000) == 1  # the LoRA branch reads x
    assert _linq(nv, xs=0xA0000 + 8) == 2           # misaligned scales
    assert _linq(nv, xg=0xB0000 + 2) == 2           # misaligned g_x
    assert _linq(nv, y=0x90000) == 7                # y over the activation codes
    assert _linq(nv, ws=0xA0000) == 7               # the workspace over the activation scales
    assert _linq(nv, K=500) == 3 and _linq(nv, r=8, A=0x70000, B=0x80000) == 3
    assert _linq(nv, wsb=16) == 4
    # without activation codes to hold, the workspace is smaller than the quantize-on-the-fly call's
    for r in (0, 32):
        q = nv.workspace_bytes(nv.OP_LINEAR_W4A4_QUANTIZED, 4096, 3584, 3584, r)
        assert 0 < q < nv.workspace_bytes(nv.OP_LINEAR_W4A4, 4096, 3584, 3584, r) - 4096 * 3584 // 2


def test_rmsnorm_validation(nv):
    L = nv.lib()
    assert L.rmsnorm_aqn(None, 4, 64, A1, None, 0.0, 1e-6, A2, None) == 1
    assert L.rmsnorm_aqn(A0, 4, 60, A1, None, 0.0, 1e-6, A2, None) == 3
    assert L.rmsnorm_aqn(A0, 4, 64, A1, None, 0.0, -1.0, A2, None) == 1
    assert L.rmsnorm_aqn(A0, 4, 64, A1 + 4, None, 0.0, 1e-6, A2, None) == 2
    assert L.rmsnorm_aqn(A0, 4, 64, A1, None, 0.0, 1e-6, A0, None) == 7


def test_rmsnorm_quantize_validation(nv):
    L = nv.lib()
    def call(x=A0, M=4, H=64, w=A1, eps=None, y=A2, c=A3, sc=A4, g=0x60000, ws=0x70000, wsb=256):
        return L.rmsnorm_aqn_quantize(x, M, H, w, eps, 0.0, 1e-6, y, c, sc, g, ws, wsb, None)
    assert nv.workspace_bytes(nv.OP_RMSNORM_QUANTIZE, 0, 0, 0) >= 8
    assert call(x=None) == 1
    assert call(H=40) == 3                       # not a multiple of 16
    assert call(H=16384) == 3                    # above the largest row
    assert call(y=A2 + 8) == 2                   # misaligned
    assert call(ws=None) == 4
    assert call(wsb=4) == 4
    assert call(y=A0) == 7                       # y over x
    assert call(c=A2) == 7                       # codes over y
    assert call(g=0x70000) == 7                  # g over the workspace


def test_binding_refuses_cpu_tensors(nv):
    import torch
    with pytest.raises(ValueError):
        nv.nvfp4_quantize(torch.zeros(4, 32))
