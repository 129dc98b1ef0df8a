"""ctypes binding of libmoestep.so (include/moestep.h).

Argument marshalling only: every function takes torch tensors (or raw addresses) and a
stream, and calls the C function of the same name. All arithmetic runs in the library's
CUDA kernels; if the library is missing, loading fails with an error (there is no other
path).
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoestep.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_TIMEOUT = range(5)
MOE_FMT_BF16, MOE_FMT_MXFP8, MOE_FMT_NVFP4, MOE_FMT_MXFP4 = 0, 1, 2, 3
MOE_W13, MOE_W2, MOE_SH13, MOE_SH2 = 0, 1, 2, 3
MOE_SCHED_STATIC, MOE_SCHED_HYBRID, MOE_SCHED_DYNAMIC = 0, 1, 2
SCHEDULES = {"static": MOE_SCHED_STATIC, "hybrid": MOE_SCHED_HYBRID, "dynamic": MOE_SCHED_DYNAMIC}
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
                4: "MOE_ERR_TIMEOUT"}

# Every symbol the header declares.
EXPORTS = ("moe_last_error_string", "moe_packed_bytes", "moe_act_bytes", "moe_act_scale_bytes", "moe_hq_bytes",
           "moe_hq_scale_bytes", "moe_workspace_bytes", "moe_workspace_init", "moe_ws_view", "moe_pack_weights",
           "moe_router_topk", "moe_route_tiles", "moe_expert_gate_up", "moe_expert_down", "moe_expert_ffn",
           "moe_finalize_norm",
           "moe_step", "moe_get_status", "moe_router_topk_noalloc")


class MoeError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), msg))
        self.status = status


class LayerDesc(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("I", ctypes.c_int32),
                ("I_shared", ctypes.c_int32), ("w_fmt", ctypes.c_int32), ("shared_fmt", ctypes.c_int32),
                ("has_shared", ctypes.c_int32), ("has_bias", ctypes.c_int32), ("renormalize", ctypes.c_int32),
                ("emit_next_mxfp8", ctypes.c_int32), ("routed_scaling_factor", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("gs_a1", ctypes.c_float), ("gs_a2", ctypes.c_float),
                ("gs_a1_shared", ctypes.c_float), ("gs_a2_shared", ctypes.c_float),
                ("swiglu_limit", ctypes.c_float), ("gemm_schedule", ctypes.c_int32), ("ffn_launches", ctypes.c_int32),
                ("front_launches", ctypes.c_int32)]


class QWeight(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("global_scale", ctypes.c_void_p)]


class StepArgs(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("w_gate", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("w13", QWeight), ("w2", QWeight), ("sh13", QWeight), ("sh2", QWeight),
                ("residual", ctypes.c_void_p), ("gamma", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("outq", ctypes.c_void_p), ("outq_scales", ctypes.c_void_p)]


class WsPtrs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "status", "logits", "scores", "topk_idx", "topk_w", "expert_counts", "perm", "inv_perm", "tiles",
        "num_tiles", "xq", "xq_scales", "xq_shared", "xq_shared_scales", "hq", "hq_scales", "y_pairs")]


_lib = None


def lib():
    """Load libmoestep.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmoestep.so is not built (run __graft_entry__.build() or "
                               "python -m moe_decode_step_router_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        D = ctypes.POINTER(LayerDesc)
        sig = {
            "moe_last_error_string": (ctypes.c_char_p, []),
            "moe_packed_bytes": (SZ, [D, I32]),
            "moe_act_bytes": (SZ, [I32, I32, I32]),
            "moe_act_scale_bytes": (SZ, [I32, I32, I32]),
            "moe_hq_bytes": (SZ, [D, I32]),
            "moe_hq_scale_bytes": (SZ, [D, I32]),
            "moe_workspace_bytes": (SZ, [D]),
            "moe_workspace_init": (I32, [D, P, P]),
            "moe_ws_view": (I32, [D, P, ctypes.POINTER(WsPtrs)]),
            "moe_pack_weights": (I32, [D, I32, P, P, P, P]),
            "moe_router_topk": (I32, [D, P, P, P, P, I32, P, P, P, P, P, P, P, P, P]),
            "moe_route_tiles": (I32, [D, P, I32, P, P, P, P, P, P, P]),
            "moe_expert_gate_up": (I32, [D, ctypes.POINTER(QWeight), ctypes.POINTER(QWeight), P, P, P, P, P, I32,
                                         P, P, P, P]),
            "moe_expert_down": (I32, [D, ctypes.POINTER(QWeight), ctypes.POINTER(QWeight), P, P, I32, P, P, P]),
            "moe_expert_ffn": (I32, [D, ctypes.POINTER(QWeight), ctypes.POINTER(QWeight), ctypes.POINTER(QWeight),
                                     ctypes.POINTER(QWeight), P, P, P, P, P, I32, P, P, P, P, P]),
            "moe_finalize_norm": (I32, [D, P, P, P, I32, P, P, P, P, P, P, P]),
            "moe_step": (I32, [D, ctypes.POINTER(StepArgs), I32, P, P]),
            "moe_get_status": (I32, [P, P, ctypes.POINTER(ctypes.c_int)]),
            "moe_router_topk_noalloc": (I32, [D, P, P, P, P, I32, P, P, P, P, P, P, P, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st):
    if st != MOE_OK:
        raise MoeError(st, lib().moe_last_error_string().decode())


def layer_desc(cfg, gs_a=(1.0, 1.0, 1.0, 1.0)) -> LayerDesc:
    """The layer descriptor of a workload dict; `schedule` ("static", "hybrid", "dynamic"),
    `ffn_launches` and `front_launches` (1 or 2) are the optional execution choices."""
    return LayerDesc(cfg["H"], cfg["E"], cfg["k"], cfg["I"], cfg["I_sh"], cfg["w_fmt"], cfg["sh_fmt"],
                     int(cfg.get("has_shared", True)), int(cfg["has_bias"]), int(cfg.get("renormalize", True)),
                     int(cfg.get("emit_next", False)), float(cfg["rsf"]), float(cfg["eps"]), float(gs_a[0]),
                     float(gs_a[1]), float(gs_a[2]), float(gs_a[3]), float(cfg.get("swiglu_limit", 0.0)),
                     SCHEDULES[cfg.get("schedule", "static")], int(cfg.get("ffn_launches", 1)),
                     int(cfg.get("front_launches", 2)))


def qweight(packed, gs=None) -> QWeight:
    return QWeight(_ptr(packed), _ptr(gs))


# ---------------------------------------------------------------- sizes
def moe_packed_bytes(d, which):
    return lib().moe_packed_bytes(ctypes.byref(d), which)


def moe_act_bytes(fmt, rows, K):
    return lib().moe_act_bytes(fmt, rows, K)


def moe_act_scale_bytes(fmt, rows, K):
    return lib().moe_act_scale_bytes(fmt, rows, K)


def moe_hq_bytes(d, max_rows):
    return lib().moe_hq_bytes(ctypes.byref(d), max_rows)


def moe_hq_scale_bytes(d, max_rows):
    return lib().moe_hq_scale_bytes(ctypes.byref(d), max_rows)


def moe_workspace_bytes(d):
    return lib().moe_workspace_bytes(ctypes.byref(d))


# ---------------------------------------------------------------- calls
def moe_workspace_init(d, ws, stream=None):
    _check(lib().moe_workspace_init(ctypes.byref(d), _ptr(ws), _stream(stream)))


def moe_ws_view(d, ws) -> WsPtrs:
    out = WsPtrs()
    _check(lib().moe_ws_view(ctypes.byref(d), _ptr(ws), ctypes.byref(out)))
    return out


def moe_pack_weights(d, which, codes, scales, dst, stream=None):
    _check(lib().moe_pack_weights(ctypes.byref(d), which, _ptr(codes), _ptr(scales), _ptr(dst), _stream(stream)))


def moe_router_topk(d, x, w_gate, bias, logits_in, M, logits_out, topk_idx, topk_w, xq, xq_scales, xq_sh,
                    xq_sh_scales, ws, stream=None):
    _check(lib().moe_router_topk(ctypes.byref(d), _ptr(x), _ptr(w_gate), _ptr(bias), _ptr(logits_in), M,
                                 _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w), _ptr(xq), _ptr(xq_scales),
                                 _ptr(xq_sh), _ptr(xq_sh_scales), _ptr(ws), _stream(stream)))


def moe_router_topk_noalloc(d, x, w_gate, bias, logits_in, M, logits_out, topk_idx, topk_w, xq, xq_scales, xq_sh,
                            xq_sh_scales, stream=None):
    _check(lib().moe_router_topk_noalloc(ctypes.byref(d), _ptr(x), _ptr(w_gate), _ptr(bias), _ptr(logits_in), M,
                                         _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w), _ptr(xq), _ptr(xq_scales),
                                         _ptr(xq_sh), _ptr(xq_sh_scales), _stream(stream)))


def moe_route_tiles(d, topk_idx, M, tiles, num_tiles, perm, inv_perm, expert_counts, ws, stream=None):
    _check(lib().moe_route_tiles(ctypes.byref(d), _ptr(topk_idx), M, _ptr(tiles), _ptr(num_tiles), _ptr(perm),
                                 _ptr(inv_perm), _ptr(expert_counts), _ptr(ws), _stream(stream)))


def moe_expert_gate_up(d, w13, sh13, xq, xq_scales, xq_sh, xq_sh_scales, perm, M, hq, hq_scales, ws, stream=None):
    _check(lib().moe_expert_gate_up(ctypes.byref(d), ctypes.byref(w13), ctypes.byref(sh13), _ptr(xq),
                                    _ptr(xq_scales), _ptr(xq_sh), _ptr(xq_sh_scales), _ptr(perm), M, _ptr(hq),
                                    _ptr(hq_scales), _ptr(ws), _stream(stream)))


def moe_expert_down(d, w2, sh2, hq, hq_scales, M, y_pairs, ws, stream=None):
    _check(lib().moe_expert_down(ctypes.byref(d), ctypes.byref(w2), ctypes.byref(sh2), _ptr(hq), _ptr(hq_scales),
                                 M, _ptr(y_pairs), _ptr(ws), _stream(stream)))


def moe_expert_ffn(d, w13, sh13, w2, sh2, xq, xq_scales, xq_sh, xq_sh_scales, perm, M, hq, hq_scales, y_pairs, ws,
                   stream=None):
    _check(lib().moe_expert_ffn(ctypes.byref(d), ctypes.byref(w13), ctypes.byref(sh13), ctypes.byref(w2),
                                ctypes.byref(sh2), _ptr(xq), _ptr(xq_scales), _ptr(xq_sh), _ptr(xq_sh_scales),
                                _ptr(perm), M, _ptr(hq), _ptr(hq_scales), _ptr(y_pairs), _ptr(ws), _stream(stream)))


def moe_finalize_norm(d, y_pairs, topk_w, inv_perm, M, residual, gamma, out, outq, outq_scales, ws, stream=None):
    _check(lib().moe_finalize_norm(ctypes.byref(d), _ptr(y_pairs), _ptr(topk_w), _ptr(inv_perm), M,
                                   _ptr(residual), _ptr(gamma), _ptr(out), _ptr(outq), _ptr(outq_scales), _ptr(ws),
                                   _stream(stream)))


def moe_step(d, args: StepArgs, M, ws, stream=None):
    _check(lib().moe_step(ctypes.byref(d), ctypes.byref(args), M, _ptr(ws), _stream(stream)))


def moe_get_status(ws, stream=None) -> int:
    v = ctypes.c_int(0)
    _check(lib().moe_get_status(_ptr(ws), _stream(stream), ctypes.byref(v)))
    return v.value
