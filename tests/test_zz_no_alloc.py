"""The allocation-free router entry point against the workspace one.

moe_router_topk_noalloc is for callers that cannot hand the library device memory (a
framework that owns every allocation, or a loop that must not allocate while running):
its scratch is a fixed array inside the library. Called twice in a row, each time on new
inputs, it must give what moe_router_topk gives on the same inputs: the same expert ids,
weights, logits and quantised FC1 inputs (these are the same kernels, so the comparison is
exact, which is within every tolerance the other tests use), up to the largest layer the
descriptor allows.

A library-internal call (not in the public header) also makes the router's copy wait run
out on purpose (its gate-row barrier expects 16 bytes that no copy brings, with a 50 ms
limit): the call must return on its own with every expert id -1 and every weight 0 rather
than a top-k of stale scores, and the next ordinary call must give the results of one on a
fresh library (the timeout record is cleared).
"""
import ctypes
import time

import numpy as np
import pytest
import torch

from moe_decode_step_router_gb300 import moestep as ms
from moe_decode_step_router_gb300 import synth

pytestmark = pytest.mark.gpu

CASES = {
    "nvfp4_e512": synth.config("nvfp4_h4096_e512_k10", M=8),
    # the largest layer: H 8192, 512 experts, 64 rows
    "nvfp4_h8192_e512_m64": synth.config("nvfp4_h4096_e512_k10", M=64, H=8192),
    "mxfp8_bias": synth.config("mxfp8_h7168_e256_k8_8rows", M=13),
    "nvfp4_bf16_shared": synth.config("nvfp4_h6144_e256_k8_16rows", M=16),
}


def _outputs(cfg, M):
    d = "cuda"
    E, k, H = cfg["E"], cfg["k"], cfg["H"]
    fr, fs = cfg["w_fmt"], cfg["sh_fmt"]
    return dict(
        logits=torch.full((M, E), -1.0, dtype=torch.float32, device=d),
        idx=torch.full((M, k), -1, dtype=torch.int32, device=d),
        w=torch.full((M, k), -1.0, dtype=torch.float32, device=d),
        xq=torch.zeros(ms.moe_act_bytes(fr, M, H), dtype=torch.uint8, device=d),
        xs=torch.zeros(max(16, ms.moe_act_scale_bytes(fr, M, H)), dtype=torch.uint8, device=d),
        xq_sh=torch.zeros(ms.moe_act_bytes(fs, M, H), dtype=torch.uint8, device=d),
        xs_sh=torch.zeros(max(16, ms.moe_act_scale_bytes(fs, M, H)), dtype=torch.uint8, device=d))


def _same(a, b):
    for name in ("idx", "w", "logits", "xq", "xs", "xq_sh", "xs_sh"):
        assert torch.equal(a[name], b[name]), name


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_workspace_entry_point_twice(name):
    cfg = CASES[name]
    M = cfg["M"]
    d = ms.layer_desc(cfg, synth.act_global_scales(cfg))
    ws = torch.empty(ms.moe_workspace_bytes(d), dtype=torch.uint8, device="cuda")
    ms.moe_workspace_init(d, ws)
    for seed in (3, 4):  # two calls in a row, on different inputs
        inp = synth.make_inputs(cfg, seed, device="cuda", weights=False)
        ref, got = _outputs(cfg, M), _outputs(cfg, M)
        ms.moe_router_topk(d, inp["x"], inp["wg"], inp["bias"], None, M, ref["logits"], ref["idx"], ref["w"],
                           ref["xq"], ref["xs"], ref["xq_sh"], ref["xs_sh"], ws)
        ms.moe_router_topk_noalloc(d, inp["x"], inp["wg"], inp["bias"], None, M, got["logits"], got["idx"],
                                   got["w"], got["xq"], got["xs"], got["xq_sh"], got["xs_sh"])
        torch.cuda.synchronize()
        assert (ref["idx"] >= 0).all() and (ref["w"] > 0).all()
        _same(ref, got)


def test_noalloc_with_given_logits_twice():
    cfg = CASES["mxfp8_bias"]
    M, E = cfg["M"], cfg["E"]
    d = ms.layer_desc(cfg, synth.act_global_scales(cfg))
    ws = torch.empty(ms.moe_workspace_bytes(d), dtype=torch.uint8, device="cuda")
    ms.moe_workspace_init(d, ws)
    inp = synth.make_inputs(cfg, 5, device="cuda", weights=False)
    for seed in (11, 12):
        li = torch.from_numpy(np.random.default_rng(seed).standard_normal((M, E)).astype(np.float32) * 2).cuda()
        ref, got = _outputs(cfg, M), _outputs(cfg, M)
        ms.moe_router_topk(d, inp["x"], inp["wg"], inp["bias"], li, M, ref["logits"], ref["idx"], ref["w"],
                           ref["xq"], ref["xs"], ref["xq_sh"], ref["xs_sh"], ws)
        ms.moe_router_topk_noalloc(d, inp["x"], inp["wg"], inp["bias"], li, M, got["logits"], got["idx"], got["w"],
                                   got["xq"], got["xs"], got["xq_sh"], got["xs_sh"])
        torch.cuda.synchronize()
        _same(ref, got)


def _router_unreachable_wait():
    f = ms.lib().moe_internal_router_noalloc_unreachable_wait
    P = ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(ms.LayerDesc), P, P, P, ctypes.c_int, P, P, P, P, P, P, P, ctypes.c_uint64, P]
    return f


@pytest.mark.parametrize("name", ["nvfp4_e512", "mxfp8_bias"])
def test_noalloc_router_wait_runs_out_then_recovers(name):
    cfg = CASES[name]
    M = cfg["M"]
    d = ms.layer_desc(cfg, synth.act_global_scales(cfg))
    inp = synth.make_inputs(cfg, 6, device="cuda", weights=False)
    ref = _outputs(cfg, M)
    ms.moe_router_topk_noalloc(d, inp["x"], inp["wg"], inp["bias"], None, M, ref["logits"], ref["idx"], ref["w"],
                               ref["xq"], ref["xs"], ref["xq_sh"], ref["xs_sh"])
    torch.cuda.synchronize()
    assert (ref["idx"] >= 0).all() and (ref["w"] > 0).all()
    got = _outputs(cfg, M)
    got["idx"].fill_(3)  # what a caller's buffers hold from an earlier step
    got["w"].fill_(0.5)
    t0 = time.perf_counter()
    st = _router_unreachable_wait()(ctypes.byref(d), ms._ptr(inp["x"]), ms._ptr(inp["wg"]), ms._ptr(inp["bias"]), M,
                                    ms._ptr(got["logits"]), ms._ptr(got["idx"]), ms._ptr(got["w"]), ms._ptr(got["xq"]),
                                    ms._ptr(got["xs"]), ms._ptr(got["xq_sh"]), ms._ptr(got["xs_sh"]), 50_000_000,
                                    ms._stream(None))
    assert st == ms.MOE_OK, ms.lib().moe_last_error_string().decode()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert 0.04 < dt < 1.5, "the call took %.3f s" % dt
    assert (got["idx"] == -1).all() and (got["w"] == 0).all()
    assert (got["logits"] == -1.0).all()  # the router wrote nothing
    for q in ("xq", "xs", "xq_sh", "xs_sh"):  # the FC1 inputs do not depend on the router
        assert torch.equal(got[q], ref[q]), q
    assert torch.ones(4, device="cuda").sum().item() == 4.0  # the context is still usable
    for _ in range(2):
        again = _outputs(cfg, M)
        ms.moe_router_topk_noalloc(d, inp["x"], inp["wg"], inp["bias"], None, M, again["logits"], again["idx"],
                                   again["w"], again["xq"], again["xs"], again["xq_sh"], again["xs_sh"])
        torch.cuda.synchronize()
        _same(ref, again)
