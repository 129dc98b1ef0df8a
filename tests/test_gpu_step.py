"""End-to-end moe_step (four PDL-chained launches; five with two FFN launches) against the
oracle, in eager mode and under CUDA-graph replay; bitwise determinism over repeated
replays; row-map invariance; and the full-size workloads, every row of each checked
against the oracle (rows run on parallel host threads)."""
import numpy as np
import pytest
import torch

import oracle
from moe_decode_step_router_gb300 import synth

from gpu_util import (check_next_mxfp8, check_output, expert_weights_for, host_weights, make, npy, oracle_layer,
                      oracle_step_rows_parallel, u16)

pytestmark = pytest.mark.gpu

SMALL = {
    "mx_mx": synth.config("tiny_mxfp8", E=16, k=2, I=256, I_sh=256, emit_next=True),
    "mx_bias": synth.config("tiny_mxfp8", H=2048, E=64, k=8, I=512, I_sh=512, has_bias=True, rsf=2.5),
    "nv_bf16": synth.config("nvfp4_h6144_e256_k8_16rows", H=1024, E=16, k=4, I=256, I_sh=256),
    "nv_mx": synth.config("nvfp4_h4096_e512_k10", H=1024, E=32, k=4, I=512, I_sh=256, emit_next=True),
    "mx4_mx": synth.config("mxfp4_h7168_e256_k8", H=1024, E=16, k=4, I=256, I_sh=256),
}


def _outputs(cfg, M, dev="cuda"):
    H = cfg["H"]
    out = torch.zeros(M, H, dtype=torch.bfloat16, device=dev)
    M8 = -(-M // 8) * 8
    oq = torch.zeros(M8, H, dtype=torch.uint8, device=dev) if cfg.get("emit_next") else None
    os_ = torch.zeros(M8, H // 32, dtype=torch.uint8, device=dev) if cfg.get("emit_next") else None
    return out, oq, os_


def _run(layer, inp, M):
    out, oq, os_ = _outputs(layer.cfg, M)
    res = inp["residual"].clone()
    layer.step(inp["x"], res, out, oq, os_)
    torch.cuda.synchronize()
    assert layer.status() == 0
    return out, res, oq, os_


def _oracle_rows(cfg, inp, rows):
    L = oracle_layer(cfg, inp)
    x16, wg16 = u16(inp["x"]), u16(inp["wg"])
    bias = npy(inp["bias"])
    _, _, idx, _, _ = oracle.router(L, x16[rows], wg16, bias=bias)
    w13, w2 = expert_weights_for(inp, idx.ravel())
    _, _, sh13, sh2 = host_weights(dict(inp, w13=inp["w13"], w2=inp["w2"]), 0)
    return oracle_step_rows_parallel(L, rows, x16, u16(inp["residual"]), u16(inp["gamma"]), wg16, bias, w13, w2,
                                     sh13, sh2, want_q=bool(cfg.get("emit_next")))


def _check_rows(layer, inp, rows, out, res, oq, os_, ref):
    M = out.shape[0]
    idx = layer.ws_tensor("topk_idx", torch.int32, (M, layer.cfg["k"]))
    gidx = npy(idx)[rows]
    ok = (ref["margin"] >= 1e-5)
    assert (gidx[ok] == ref["topk_idx"][ok]).all(), "routing differs on rows with a clear margin"
    keep = ok | (gidx == ref["topk_idx"]).all(1)
    if keep.any():
        check_output(u16(out)[rows][keep], ref["out"][keep], "out")
        check_output(u16(res)[rows][keep], ref["res_out"][keep], "residual")
    if oq is not None:
        # every row, excused or not: the quantiser of the GPU's own output, bit for bit
        check_next_mxfp8(u16(out)[rows], npy(oq)[rows], npy(os_)[rows])


@pytest.mark.parametrize("sched", ["static", "dynamic"])
@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("M", [1, 8, 23, 64])
def test_step_matches_oracle(name, M, sched):
    # the GEMMs' work schedule (equal static ranges, items taken from a counter, or both)
    # changes only how units are cut between CTAs, never the result beyond fp32 summation
    # order
    cfg = dict(SMALL[name], schedule=sched)
    inp, layer = make(cfg, seed=10 + M, M=M)
    out, res, oq, os_ = _run(layer, inp, M)
    rows = list(range(M))
    ref = _oracle_rows(cfg, inp, rows)
    _check_rows(layer, inp, rows, out, res, oq, os_, ref)
    if oq is not None:  # padding rows of the 8-row tiles are zero
        assert (npy(oq)[M:] == 0).all() and (npy(os_)[M:] == 0).all()


@pytest.mark.parametrize("sched", ["static", "dynamic", "hybrid"])
def test_graph_replay_equals_eager_and_is_deterministic(sched):
    # when items come from a counter the CTA that computes one changes from run to run;
    # the bytes must not
    cfg = dict(SMALL["nv_mx"], schedule=sched)
    M = 19
    inp, layer = make(cfg, seed=5, M=M)
    out_e, res_e, oq_e, os_e = _run(layer, inp, M)
    out, oq, os_ = _outputs(cfg, M)
    res = inp["residual"].clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer.step(inp["x"], res, out, oq, os_)
    first = None
    for i in range(50):
        res.copy_(inp["residual"])
        g.replay()
        torch.cuda.synchronize()
        cur = (u16(out).tobytes(), u16(res).tobytes(), npy(oq).tobytes())
        if first is None:
            first = cur
            assert cur[0] == u16(out_e).tobytes() and cur[1] == u16(res_e).tobytes()
        assert cur == first, "replay %d differs" % i
    assert layer.status() == 0


def test_row_map_invariance():
    cfg = SMALL["mx_bias"]
    M = 24
    inp, layer = make(cfg, seed=9, M=M)
    out1, res1, _, _ = _run(layer, inp, M)
    p = torch.randperm(M, generator=torch.Generator().manual_seed(1))
    inp2 = dict(inp, x=inp["x"][p].contiguous(), residual=inp["residual"][p].contiguous())
    out2, res2, _, _ = _run(layer, inp2, M)
    assert torch.equal(out1[p], out2) and torch.equal(res1[p], res2)


# (workload, rows, GEMM schedule); "static" is the default. Every row of each is compared
# with the oracle: at these sizes the kernels take their multi-tile, stream-K and
# hot-expert paths.
FULL = [("tiny_mxfp8", None, "static"), ("mxfp8_h7168_e256_k8_8rows", None, "static"),
        ("nvfp4_h6144_e256_k8_16rows", None, "static"), ("mxfp8_skew_48rows", None, "static"),
        ("nvfp4_h4096_e512_k10", 1, "static"), ("nvfp4_h4096_e512_k10", 8, "static"),
        ("nvfp4_h4096_e512_k10", 16, "static"), ("nvfp4_h4096_e512_k10", 64, "static"),
        ("mxfp8_h7168_e256_k8_8rows", None, "hybrid"),
        ("nvfp4_h6144_e256_k8_16rows", None, "dynamic"), ("nvfp4_h4096_e512_k10", 1, "dynamic"),
        ("nvfp4_h4096_e512_k10", 32, "hybrid"), ("mxfp8_h7168_e256_k8_8rows", None, "dynamic"),
        ("mxfp4_h7168_e256_k8", None, "static"), ("mxfp4_h7168_e256_k8", 64, "static")]


@pytest.mark.parametrize("name,M,sched", FULL, ids=["%s-%s-%s" % f for f in FULL])
def test_full_size_every_row(name, M, sched):
    cfg = synth.config(name, schedule=sched) if M is None else synth.config(name, M=M, schedule=sched)
    M = cfg["M"]
    inp, layer = make(cfg, seed=0, M=M)
    out, res, oq, os_ = _run(layer, inp, M)
    rows = list(range(M))
    ref = _oracle_rows(cfg, inp, rows)
    _check_rows(layer, inp, rows, out, res, oq, os_, ref)
    # rows excused by a routing margin below 1e-5 are rare
    assert (ref["margin"] >= 1e-5).mean() >= 0.9
    assert torch.isfinite(out.float()).all()
    if cfg.get("skew"):
        counts = npy(layer.ws_tensor("expert_counts", torch.int32, (cfg["E"] + 1,)))
        assert (counts[:cfg["E"]] > 8).any()
        idle = (counts[:cfg["E"]] == 0).mean()
        assert 0.25 < idle < 0.55


@pytest.mark.parametrize("sched", ["hybrid", "dynamic"])
def test_full_size_counter_schedules_are_deterministic(sched):
    # these schedules hand units to whichever CTA is free first
    cfg = synth.config("mxfp8_h7168_e256_k8_8rows", schedule=sched)
    M = cfg["M"]
    inp, layer = make(cfg, seed=1, M=M)
    runs = []
    for _ in range(3):
        out, res, _, _ = _run(layer, inp, M)
        runs.append((u16(out).tobytes(), u16(res).tobytes()))
    assert runs[0] == runs[1] == runs[2]


# Clamped SwiGLU ("SGLang-NVIDIA-Mega" README, shared_ll row): the limit is chosen below
# the typical |gate| so that most gate and up values of every format are cut.
@pytest.mark.parametrize("name", ["mx_mx", "nv_bf16", "nv_mx"])
@pytest.mark.parametrize("M", [8, 37])
def test_clamped_swiglu_step_matches_oracle(name, M):
    cfg = dict(SMALL[name], swiglu_limit=0.25)
    inp, layer = make(cfg, seed=40 + M, M=M)
    out, res, oq, os_ = _run(layer, inp, M)
    rows = list(range(M))
    ref = _oracle_rows(cfg, inp, rows)
    _check_rows(layer, inp, rows, out, res, oq, os_, ref)
    # the limit does change the step
    plain = _oracle_rows(dict(cfg, swiglu_limit=0.0), inp, rows)
    assert np.abs(plain["out"].astype(np.int64) - ref["out"].astype(np.int64)).max() > 0


def test_clamped_swiglu_full_size_sampled_rows():
    cfg = synth.config("mxfp8_h7168_e256_k8_8rows", swiglu_limit=1.0)
    M = cfg["M"]
    inp, layer = make(cfg, seed=2, M=M)
    out, res, oq, os_ = _run(layer, inp, M)
    rows = [0, M - 1]
    ref = _oracle_rows(cfg, inp, rows)
    _check_rows(layer, inp, rows, out, res, oq, os_, ref)


# moe_step runs gate_up and down as one launch (down items wait in the kernel for their
# group's gate_up units); a layer with ffn_launches = 2 runs the two separate launches.
# Both cut the same units at the same steps, so the bytes must agree exactly.
@pytest.mark.parametrize("name,M", [(n, m) for n in SMALL for m in (1, 23)] + [("full", 8)])
def test_one_launch_ffn_equals_two_launches(name, M):
    cfg = synth.config("mxfp8_h7168_e256_k8_8rows") if name == "full" else SMALL[name]
    inp, layer = make(cfg, seed=21 + M, M=M)
    layer.d.ffn_launches = 2
    two = _run(layer, inp, M)
    layer.d.ffn_launches = 1
    one = _run(layer, inp, M)
    assert torch.equal(one[0], two[0]) and torch.equal(one[1], two[1])
    if one[2] is not None:
        assert torch.equal(one[2], two[2]) and torch.equal(one[3], two[3])


# A layer with front_launches = 1 runs the router, the top-k, the routing and the FC1 input
# quantisation as one launch (the last router CTA of an 8-row block takes its rows' top-k,
# the last block routes); the default runs the router launch and the top-k / routing
# launch. Same arithmetic in the same order: the same bytes, at every row count (one row
# block, several, and the 512-expert layer's 128 router CTAs per block).
@pytest.mark.parametrize("name,M", [(n, m) for n in SMALL for m in (1, 23, 64)] + [("full", 8), ("full512", 16)])
def test_one_launch_front_equals_two_launches(name, M):
    cfg = (synth.config("mxfp8_h7168_e256_k8_8rows") if name == "full" else
           synth.config("nvfp4_h4096_e512_k10", M=M) if name == "full512" else SMALL[name])
    inp, layer = make(cfg, seed=31 + M, M=M)
    layer.d.front_launches = 2
    two = _run(layer, inp, M)
    idx2 = layer.ws_tensor("topk_idx", torch.int32, (M, cfg["k"])).clone()
    layer.d.front_launches = 1
    one = _run(layer, inp, M)
    idx1 = layer.ws_tensor("topk_idx", torch.int32, (M, cfg["k"]))
    assert torch.equal(idx1, idx2)
    assert torch.equal(one[0], two[0]) and torch.equal(one[1], two[1])
    if one[2] is not None:
        assert torch.equal(one[2], two[2]) and torch.equal(one[3], two[3])
