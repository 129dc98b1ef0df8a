"""Helpers of the GPU parity tests: decode the library's tiled layouts back to the
canonical ones (numpy), drive the oracle on the same seeded inputs, and apply the
output tolerance of the step."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
from moe_decode_step_router_gb300 import moestep as ms
from moe_decode_step_router_gb300 import synth
from moe_decode_step_router_gb300.runtime import MoELayer

FMT = {0: "bf16", 1: "mxfp8", 2: "nvfp4"}


def cuda_ok():
    return torch.cuda.is_available()


def u16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().astype(np.uint16)


def bf16_to_f64(a16):
    return torch.from_numpy(np.ascontiguousarray(a16).astype(np.int16)).view(torch.bfloat16).double().numpy()


def npy(t):
    return None if t is None else t.detach().cpu().numpy()


def row_bytes(fmt, K):
    return 2 * K if fmt == 0 else (K if fmt == 1 else K // 2)


def row_scales(fmt, K):
    return K // 32 if fmt in (1, 3) else (K // 16 if fmt == 2 else 0)


def untile(buf, fmt, rows, K, Rpad=None):
    """Tiled activation codes -> canonical [rows, row_bytes]."""
    buf = np.asarray(buf, np.uint8).ravel()
    Rpad = Rpad or -(-rows // 16) * 16
    rb = row_bytes(fmt, K)
    KS = rb // 128
    t = buf[:KS * Rpad * 128].reshape(KS, Rpad, 8, 16)
    out = np.zeros((rows, rb), np.uint8)
    for r in range(rows):
        pos = np.arange(8) ^ (r & 7)              # chunk c is stored at position c ^ (r & 7)
        out[r] = t[:, r, pos, :].reshape(-1)
    return out


def untile_scales(buf, fmt, rows, K):
    """Tiled scale atoms -> canonical [rows, row_scales]."""
    buf = np.asarray(buf, np.uint8).ravel()
    rb = row_bytes(fmt, K)
    KS = rb // 128
    A = {1: 1, 2: 4, 3: 2}[fmt]
    at = buf[:KS * A * 512].reshape(KS, A, 512)
    out = np.zeros((rows, row_scales(fmt, K)), np.uint8)
    for r in range(rows):
        off = (r % 32) * 16 + (r // 32) * 4
        out[r] = at[:, :, off:off + 4].reshape(-1)
    return out


def host_weights(inp, E):
    n = lambda t: None if t is None else t.detach().cpu().numpy()
    w13 = [(n(inp["w13"][0][e]), n(inp["w13"][1][e]) if inp["w13"][1] is not None else None,
            float(inp["w13"][2][e])) for e in range(E)]
    w2 = [(n(inp["w2"][0][e]), n(inp["w2"][1][e]) if inp["w2"][1] is not None else None, float(inp["w2"][2][e]))
          for e in range(E)]
    sh13 = sh2 = None
    if "sh13" in inp:
        sh13 = (n(inp["sh13"][0][0]), n(inp["sh13"][1][0]) if inp["sh13"][1] is not None else None,
                float(inp["sh13"][2][0]))
        sh2 = (n(inp["sh2"][0][0]), n(inp["sh2"][1][0]) if inp["sh2"][1] is not None else None,
               float(inp["sh2"][2][0]))
    return w13, w2, sh13, sh2


def expert_weights_for(inp, experts):
    """Host copies of only the listed experts (others None)."""
    E = inp["w13"][0].shape[0]
    w13, w2 = [None] * E, [None] * E
    for e in sorted(set(int(v) for v in experts)):
        w13[e] = (npy(inp["w13"][0][e]), npy(inp["w13"][1][e]) if inp["w13"][1] is not None else None,
                  float(inp["w13"][2][e]))
        w2[e] = (npy(inp["w2"][0][e]), npy(inp["w2"][1][e]) if inp["w2"][1] is not None else None,
                 float(inp["w2"][2][e]))
    return w13, w2


def check_output(got16, ref16, what="out"):
    """Step output bound: rel-L2 <= 5e-3 and |err| <= 1e-2 max|ref| + 2^-7 |ref| per element."""
    g = bf16_to_f64(got16)
    r = bf16_to_f64(ref16)
    err = np.abs(g - r)
    rel_l2 = np.sqrt((err ** 2).sum() / max((r ** 2).sum(), 1e-300))
    bound = 1e-2 * np.abs(r).max() + 2 ** -7 * np.abs(r)
    bad = err > bound
    assert rel_l2 <= 5e-3, "%s: rel-L2 %.3g" % (what, rel_l2)
    assert not bad.any(), "%s: %d elements over the bound, worst %.3g (bound %.3g)" % (
        what, bad.sum(), err[bad].max(), bound[bad][np.argmax(err[bad])])
    return rel_l2


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.sqrt(((a - b) ** 2).sum() / max((b ** 2).sum(), 1e-300)))


def make(cfg, seed=0, M=None, device="cuda"):
    M = cfg["M"] if M is None else M
    inp = synth.make_inputs(cfg, seed, device=device, M=M)
    layer = MoELayer(cfg, inp, device)
    return inp, layer


def oracle_layer(cfg, inp):
    return oracle.make_layer(cfg, inp["gs_a"])


def oracle_step_rows_parallel(L, rows, *args, **kw):
    """oracle.step_rows over `rows`, one row per task on a pool of host threads.

    Rows are independent in the step's definition, and the oracle's C code keeps no
    global state and releases the interpreter lock while it runs, so the rows run in
    parallel; the result is the same dict as one call over all the rows."""
    rows = [int(r) for r in rows]
    with ThreadPoolExecutor(max_workers=max(1, min(len(rows), os.cpu_count() or 1))) as ex:
        parts = list(ex.map(lambda r: oracle.step_rows(L, [r], *args, **kw), rows))
    out = {}
    for key in parts[0]:
        vals = [p[key] for p in parts]
        out[key] = None if vals[0] is None else np.concatenate(vals, axis=0)
    return out


def check_next_mxfp8(out16, oq, os_):
    """The next layer's MXFP8 input is the block quantisation of the step's own bf16 output:
    bit for bit the oracle's quantiser applied to the same values."""
    v = bf16_to_f64(out16).astype(np.float32)
    rq, rs = oracle.quant(oracle.FMT_MXFP8, v)
    assert (np.asarray(oq) == rq).all(), "next-layer MXFP8 codes differ from the quantiser of the output"
    assert (np.asarray(os_) == rs).all(), "next-layer MXFP8 scales differ from the quantiser of the output"
