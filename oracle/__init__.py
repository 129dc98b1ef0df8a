"""CPU oracle for the small-M MoE decode/verify step (test infrastructure only).

This package is the plain, slow definition the CUDA library is checked against.
Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import it; the product path never does. It shares no code with the CUDA
library: ``oracle.cpp`` is compiled on its own with g++ and loaded through ctypes.

Every function here only marshals numpy arrays into the C functions of
``oracle.cpp``; the arithmetic lives there, with its citations.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FMT_BF16, FMT_MXFP8, FMT_NVFP4, FMT_MXFP4 = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile oracle.cpp into liboracle.so (g++, -ffp-contract=off, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


class Layer(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("I", ctypes.c_int32), ("I_sh", ctypes.c_int32),
                ("w_fmt", ctypes.c_int32), ("sh_fmt", ctypes.c_int32),
                ("has_shared", ctypes.c_int32), ("has_bias", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("emit_next", ctypes.c_int32),
                ("rsf", ctypes.c_double), ("eps", ctypes.c_double),
                ("gs_a1", ctypes.c_float), ("gs_a2", ctypes.c_float),
                ("gs_a1_sh", ctypes.c_float), ("gs_a2_sh", ctypes.c_float),
                ("swiglu_limit", ctypes.c_double)]


class Proj(ctypes.Structure):
    _fields_ = [("vals", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("gs", ctypes.c_float)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            L.or_e4m3_decode.restype = ctypes.c_double
            L.or_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.or_e2m1_decode.restype = ctypes.c_double
            L.or_e2m1_decode.argtypes = [ctypes.c_uint8]
            L.or_e8m0_decode.restype = ctypes.c_double
            L.or_e8m0_decode.argtypes = [ctypes.c_uint8]
            L.or_e4m3_encode.restype = ctypes.c_uint8
            L.or_e4m3_encode.argtypes = [ctypes.c_float]
            L.or_e2m1_encode.restype = ctypes.c_uint8
            L.or_e2m1_encode.argtypes = [ctypes.c_float]
            L.or_double_to_bf16.restype = ctypes.c_uint16
            L.or_double_to_bf16.argtypes = [ctypes.c_double]
            L.or_quant.restype = None
            L.or_quant.argtypes = [ctypes.c_int, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_float, P, P]
            L.or_dequant.restype = None
            L.or_dequant.argtypes = [ctypes.c_int, P, P, ctypes.c_double, ctypes.c_int64, ctypes.c_int64, P]
            L.or_router.restype = None
            L.or_router.argtypes = [ctypes.POINTER(Layer), ctypes.c_int, P, P, P, P, P, P, P, P, P]
            L.or_route.restype = None
            L.or_route.argtypes = [ctypes.POINTER(Layer), ctypes.c_int, P, P, P, P, P, P, P]
            L.or_quant_x.restype = None
            L.or_quant_x.argtypes = [ctypes.c_int, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_float, P, P]
            L.or_expert_row.restype = None
            L.or_expert_row.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(Proj),
                                        ctypes.POINTER(Proj), P, ctypes.c_float, ctypes.c_double, P, P, P, P]
            L.or_finalize_row.restype = None
            L.or_finalize_row.argtypes = [ctypes.POINTER(Layer), P, P, P, P, P, P, P]
            L.or_step_rows.restype = ctypes.c_int
            L.or_step_rows.argtypes = [ctypes.POINTER(Layer), ctypes.c_int, P, ctypes.c_int, P, P, P, P, P, P,
                                       P, P, P, P, P, P, P, P, P, P, P, P, P]
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def row_bytes(fmt, K):
    return 2 * K if fmt == FMT_BF16 else (K if fmt == FMT_MXFP8 else K // 2)


def row_scales(fmt, K):
    return K // 32 if fmt in (FMT_MXFP8, FMT_MXFP4) else (K // 16 if fmt == FMT_NVFP4 else 0)


def e4m3_decode(b):
    return lib().or_e4m3_decode(int(b))


def e2m1_decode(b):
    return lib().or_e2m1_decode(int(b))


def e8m0_decode(b):
    return lib().or_e8m0_decode(int(b))


def e4m3_encode(x):
    return lib().or_e4m3_encode(float(x))


def e2m1_encode(x):
    return lib().or_e2m1_encode(float(x))


def double_to_bf16(d):
    return lib().or_double_to_bf16(float(d))


def quant(fmt, v, gs=1.0):
    """Quantise fp32 rows [R, K] -> (codes [R, row_bytes], scales [R, row_scales])."""
    v = _c(v, np.float32)
    R, K = v.shape
    q = np.zeros((R, row_bytes(fmt, K)), np.uint8)
    s = np.zeros((R, max(row_scales(fmt, K), 1)), np.uint8)
    lib().or_quant(fmt, _p(v), R, K, gs, _p(q), _p(s))
    return q, s[:, :row_scales(fmt, K)]


def dequant(fmt, q, s, K, gs=1.0):
    q = _c(q, np.uint8)
    s = _c(s, np.uint8) if s is not None and s.size else None
    R = q.shape[0]
    out = np.zeros((R, K), np.float64)
    lib().or_dequant(fmt, _p(q), _p(s), gs, R, K, _p(out))
    return out


def make_layer(cfg, gs_a=(1.0, 1.0, 1.0, 1.0)):
    return Layer(cfg["H"], cfg["E"], cfg["k"], cfg["I"], cfg["I_sh"], cfg["w_fmt"], cfg["sh_fmt"],
                 int(cfg.get("has_shared", True)), int(cfg["has_bias"]), int(cfg.get("renormalize", True)),
                 int(cfg.get("emit_next", False)), float(cfg["rsf"]), float(cfg["eps"]),
                 float(gs_a[0]), float(gs_a[1]), float(gs_a[2]), float(gs_a[3]),
                 float(cfg.get("swiglu_limit", 0.0)))


def router(layer, x_bf16, wg_bf16, bias=None, logits_in=None):
    """Returns logits f32 [M,E], scores f32 [M,E], topk_idx i32 [M,k], topk_w f64 [M,k], margin [M]."""
    x = _c(x_bf16, np.uint16)
    M = x.shape[0]
    E, k = layer.E, layer.k
    wg = _c(wg_bf16, np.uint16)
    bias = _c(bias, np.float32)
    li = _c(logits_in, np.float32)
    logits = np.zeros((M, E), np.float32)
    scores = np.zeros((M, E), np.float32)
    idx = np.zeros((M, k), np.int32)
    w = np.zeros((M, k), np.float64)
    margin = np.zeros(M, np.float64)
    lib().or_router(ctypes.byref(layer), M, _p(x), _p(wg), _p(bias), _p(li), _p(logits), _p(scores), _p(idx),
                    _p(w), _p(margin))
    return logits, scores, idx, w, margin


def route(layer, topk_idx):
    """Returns counts [E+1], offsets [E+2], perm, inv_perm, tiles [T,3]."""
    t = _c(topk_idx, np.int32)
    M = t.shape[0]
    E, k = layer.E, layer.k
    P = M * k + (M if layer.has_shared else 0)
    counts = np.zeros(E + 1, np.int32)
    offsets = np.zeros(E + 2, np.int32)
    perm = np.zeros(max(P, 1), np.int32)
    inv = np.zeros(max(P, 1), np.int32)
    tiles = np.zeros((P + E + 1, 3), np.int32)
    nt = np.zeros(1, np.int32)
    lib().or_route(ctypes.byref(layer), M, _p(t), _p(counts), _p(offsets), _p(perm), _p(inv), _p(tiles), _p(nt))
    return counts, offsets, perm[:P], inv[:P], tiles[:nt[0]]


def quant_x(fmt, x_bf16, gs=1.0):
    x = _c(x_bf16, np.uint16)
    R, H = x.shape
    q = np.zeros((R, row_bytes(fmt, H)), np.uint8)
    s = np.zeros((R, max(row_scales(fmt, H), 1)), np.uint8)
    lib().or_quant_x(fmt, _p(x), R, H, gs, _p(q), _p(s))
    return q, s[:, :row_scales(fmt, H)]


def _proj(vals, scales, gs):
    return Proj(vals.ctypes.data, None if scales is None or scales.size == 0 else scales.ctypes.data, float(gs))


def expert_row(fmt, H, I, w13, w2, xdq, gs_a2=1.0, limit=0.0):
    """One expert on one dequantised input row.

    w13 = (vals [2I, rb], scales [2I, rs] | None, gs), w2 = (vals [H, rb], scales, gs).
    Returns hq codes, hq scales, h (double, pre-quantisation), y (double [H]).
    """
    v13, s13, g13 = (_c(w13[0], np.uint8), _c(w13[1], np.uint8) if w13[1] is not None else None, w13[2])
    v2, s2, g2 = (_c(w2[0], np.uint8), _c(w2[1], np.uint8) if w2[1] is not None else None, w2[2])
    p13, p2 = _proj(v13, s13, g13), _proj(v2, s2, g2)
    xdq = _c(xdq, np.float64)
    hq = np.zeros(row_bytes(fmt, I), np.uint8)
    hs = np.zeros(max(row_scales(fmt, I), 1), np.uint8)
    h = np.zeros(I, np.float64)
    y = np.zeros(H, np.float64)
    lib().or_expert_row(fmt, H, I, ctypes.byref(p13), ctypes.byref(p2), _p(xdq), gs_a2, limit, _p(hq), _p(hs),
                        _p(h), _p(y))
    return hq, hs[:row_scales(fmt, I)], h, y


def finalize_row(layer, moe, residual_bf16, gamma_bf16, want_q=False):
    moe = _c(moe, np.float64)
    r = _c(residual_bf16, np.uint16)
    g = _c(gamma_bf16, np.uint16)
    H = layer.H
    res_out = np.zeros(H, np.uint16)
    out = np.zeros(H, np.uint16)
    oq = np.zeros(H, np.uint8) if want_q else None
    os_ = np.zeros(H // 32, np.uint8) if want_q else None
    lib().or_finalize_row(ctypes.byref(layer), _p(moe), _p(r), _p(g), _p(res_out), _p(out), _p(oq), _p(os_))
    return out, res_out, oq, os_


def step_rows(layer, rows, x, residual, gamma, wg, bias, w13, w2, sh13=None, sh2=None, logits_in=None,
              want_q=False):
    """Whole step a1..a7 for the listed rows.

    w13[e] / w2[e]: (vals, scales|None, gs) per expert, or None where not supplied.
    Returns dict with topk_idx, topk_w, margin, y_pairs, y_shared, out, res_out, outq, outs.
    """
    H, E, k = layer.H, layer.E, layer.k
    rows = np.ascontiguousarray(rows, np.int32)
    n = len(rows)
    keep = []

    def mk(t):
        if t is None:
            return Proj(None, None, 1.0)
        v = _c(t[0], np.uint8)
        s = _c(t[1], np.uint8) if t[1] is not None else None
        keep.append((v, s))
        return _proj(v, s, t[2])

    W13 = (Proj * E)(*[mk(t) for t in w13])
    W2 = (Proj * E)(*[mk(t) for t in w2])
    S13, S2 = mk(sh13), mk(sh2)
    x = _c(x, np.uint16)
    residual = _c(residual, np.uint16)
    gamma = _c(gamma, np.uint16)
    wg = _c(wg, np.uint16)
    bias = _c(bias, np.float32)
    li = _c(logits_in, np.float32)
    M = x.shape[0]
    idx = np.zeros((n, k), np.int32)
    w = np.zeros((n, k), np.float64)
    margin = np.zeros(n, np.float64)
    yp = np.zeros((n, k, H), np.float64)
    ys = np.zeros((n, H), np.float64)
    out = np.zeros((n, H), np.uint16)
    ro = np.zeros((n, H), np.uint16)
    oq = np.zeros((n, H), np.uint8) if want_q else None
    os_ = np.zeros((n, H // 32), np.uint8) if want_q else None
    rc = lib().or_step_rows(ctypes.byref(layer), M, _p(rows), n, _p(x), _p(residual), _p(gamma), _p(wg),
                            _p(bias), _p(li), W13, W2, ctypes.byref(S13), ctypes.byref(S2), _p(idx), _p(w),
                            _p(margin), _p(yp), _p(ys), _p(out), _p(ro), _p(oq), _p(os_))
    if rc != 0:
        raise KeyError("oracle step needs expert %d, which was not supplied" % (-rc - 1))
    return dict(topk_idx=idx, topk_w=w, margin=margin, y_pairs=yp, y_shared=ys, out=out, res_out=ro,
                outq=oq, outs=os_)
