"""The bounded waits of the expert GEMM, made to run out on purpose, on the GPU.

A library-internal call (not in the public header) runs the one-launch FFN with every down
item waiting for a counter value its FC1 units never reach, and every wait limited to
50 ms. The launch must return on its own, record MOE_ERR_TIMEOUT in the workspace status
word, leave the context usable, and after moe_workspace_init the next step must match the
oracle and the step before the timeout bit for bit. No wait is removed and nothing faults:
the kernel gives up, drains its copies and MMAs, frees its tensor memory and returns.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
from moe_decode_step_router_gb300 import moestep as ms
from moe_decode_step_router_gb300 import synth

from gpu_util import check_output, host_weights, make, oracle_layer, u16

pytestmark = pytest.mark.gpu


def _internal():
    f = ms.lib().moe_internal_ffn_unreachable_wait
    P, QW = ctypes.c_void_p, ctypes.POINTER(ms.QWeight)
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(ms.LayerDesc), QW, QW, QW, QW, P, P, P, P, P, ctypes.c_int, P, P, P, P,
                  ctypes.c_uint64, P]
    return f


@pytest.mark.parametrize("name,M", [("tiny_mxfp8", 4), ("nvfp4_h4096_e512_k10", 3)])
def test_gemm_wait_runs_out_and_the_workspace_recovers(name, M):
    cfg = synth.config(name, M=M) if name == "tiny_mxfp8" else synth.config(name, M=M, H=1024, E=32, k=4, I=512,
                                                                               I_sh=256)
    inp, layer = make(cfg, seed=3, M=M)
    H = cfg["H"]
    out0 = torch.zeros(M, H, dtype=torch.bfloat16, device="cuda")
    res0 = inp["residual"].clone()
    layer.step(inp["x"], res0, out0)
    torch.cuda.synchronize()
    assert layer.status() == 0
    # the routing and FC1 inputs of that step are in the workspace: run the FFN with an
    # unreachable counter target and 50 ms waits
    v, q = layer.view, layer.qw
    perm = layer.ws_tensor("perm", torch.int32, (M * cfg["k"] + M,))
    stream = torch.cuda.current_stream()
    t0 = time.perf_counter()
    st = _internal()(ctypes.byref(layer.d), ctypes.byref(q["w13"]), ctypes.byref(q["sh13"]), ctypes.byref(q["w2"]),
                     ctypes.byref(q["sh2"]), v.xq, v.xq_scales, v.xq_shared, v.xq_shared_scales, perm.data_ptr(), M,
                     v.hq, v.hq_scales, v.y_pairs, layer.ws.data_ptr(), 50_000_000, stream.cuda_stream)
    assert st == ms.MOE_OK, ms.lib().moe_last_error_string().decode()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert layer.status() == ms.MOE_ERR_TIMEOUT
    assert 0.04 < dt < 1.5, "the launch took %.3f s" % dt
    # the context is still usable
    assert torch.ones(4, device="cuda").sum().item() == 4.0
    ms.moe_workspace_init(layer.d, layer.ws)
    assert layer.status() == 0
    out1 = torch.zeros_like(out0)
    res1 = inp["residual"].clone()
    layer.step(inp["x"], res1, out1)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(out1, out0) and torch.equal(res1, res0)
    L = oracle_layer(cfg, inp)
    w13, w2, sh13, sh2 = host_weights(inp, cfg["E"])
    ref = oracle.step_rows(L, np.arange(M), u16(inp["x"]), u16(inp["residual"]), u16(inp["gamma"]), u16(inp["wg"]),
                           None if inp["bias"] is None else inp["bias"].cpu().numpy(), w13, w2, sh13, sh2)
    ok = ref["margin"] >= 1e-5
    check_output(u16(out1)[ok], ref["out"][ok], "out after the timeout")
