"""GPU parity of each stage of the step against the oracle, through the C ABI.

Routing, route tiles and the FC1 input quantisation are compared bit for bit on the same
fp32 logits; the expert GEMMs and the finalize within the step's tolerance. Shapes span
several 128-row blocks, ragged row counts (1..64) and every format pairing the workloads
use (MXFP8 + MXFP8, NVFP4 + BF16 shared, NVFP4 + MXFP8 shared).
"""
import numpy as np
import pytest
import torch

import oracle
from moe_decode_step_router_gb300 import moestep as ms
from moe_decode_step_router_gb300 import synth

from gpu_util import (bf16_to_f64, check_next_mxfp8, check_output, expert_weights_for, host_weights, make, npy,
                      oracle_layer, rel_l2, row_bytes, row_scales, u16, untile, untile_scales)

pytestmark = pytest.mark.gpu

SMALL = {
    "mx_mx": synth.config("tiny_mxfp8", E=16, k=2, I=256, I_sh=256),
    "mx_mx_bias": synth.config("tiny_mxfp8", E=32, k=8, I=512, I_sh=256, H=2048, has_bias=True, rsf=2.5),
    "nv_bf16": synth.config("nvfp4_h6144_e256_k8_16rows", H=1024, E=16, k=4, I=256, I_sh=256),
    "nv_mx": synth.config("nvfp4_h4096_e512_k10", H=1024, E=32, k=4, I=512, I_sh=256),
    "mx4_mx": synth.config("mxfp4_h7168_e256_k8", H=1024, E=16, k=4, I=256, I_sh=256),
    "mx4_mx4_bias": synth.config("mxfp4_h7168_e256_k8", H=2048, E=32, k=8, I=512, I_sh=512, sh_fmt=3,
                                 has_bias=True, rsf=2.5),
}


def _alloc(layer, M, dev="cuda"):
    d, cfg = layer.d, layer.cfg
    E, k, H = cfg["E"], cfg["k"], cfg["H"]
    t = {}
    t["logits"] = torch.zeros(M, E, dtype=torch.float32, device=dev)
    t["idx"] = torch.zeros(M, k, dtype=torch.int32, device=dev)
    t["w"] = torch.zeros(M, k, dtype=torch.float32, device=dev)
    t["xq"] = torch.zeros(ms.moe_act_bytes(cfg["w_fmt"], M, H), dtype=torch.uint8, device=dev)
    t["xs"] = torch.zeros(max(ms.moe_act_scale_bytes(cfg["w_fmt"], M, H), 16), dtype=torch.uint8, device=dev)
    t["xq_sh"] = torch.zeros(ms.moe_act_bytes(cfg["sh_fmt"], M, H), dtype=torch.uint8, device=dev)
    t["xs_sh"] = torch.zeros(max(ms.moe_act_scale_bytes(cfg["sh_fmt"], M, H), 16), dtype=torch.uint8, device=dev)
    P = M * k + M
    t["counts"] = torch.zeros(E + 1, dtype=torch.int32, device=dev)
    t["perm"] = torch.zeros(P, dtype=torch.int32, device=dev)
    t["inv"] = torch.zeros(P, dtype=torch.int32, device=dev)
    t["tiles"] = torch.zeros(P + E + 1, 3, dtype=torch.int32, device=dev)
    t["nt"] = torch.zeros(1, dtype=torch.int32, device=dev)
    t["hq"] = torch.zeros(ms.moe_hq_bytes(d, M), dtype=torch.uint8, device=dev)
    t["hs"] = torch.zeros(ms.moe_hq_scale_bytes(d, M), dtype=torch.uint8, device=dev)
    t["y"] = torch.zeros(P, H, dtype=torch.float32, device=dev)
    t["out"] = torch.zeros(M, H, dtype=torch.bfloat16, device=dev)
    return t


ATOMS = {0: 0, 1: 1, 2: 4, 3: 2}  # scale atoms per 128-byte K step (BF16, MXFP8, NVFP4, MXFP4)


def _logits(M, E, seed):
    g = np.random.default_rng(seed)
    return (g.standard_normal((M, E)) * 2.0).astype(np.float32)


def _hq_routed_bytes(cfg, M):
    P = M * cfg["k"]
    G = min(P, cfg["E"])
    return -(-((P + 15 * G) * row_bytes(cfg["w_fmt"], cfg["I"])) // 256) * 256


def _hs_routed_bytes(cfg, M):
    P = M * cfg["k"]
    G = min(P, cfg["E"])
    f = cfg["w_fmt"]
    KS = row_bytes(f, cfg["I"]) // 128
    return -(-(G * KS * ATOMS[f] * 512) // 256) * 256


def _gpu_hidden(cfg, M, counts, hq, hs):
    """Per routed expert: (codes, scales) of its group block; and the shared block."""
    f, I = cfg["w_fmt"], cfg["I"]
    rb = row_bytes(f, I)
    KS = rb // 128
    A = ATOMS[f]
    out = {}
    row_off = gi = 0
    for e in range(cfg["E"]):
        c = int(counts[e])
        if c == 0:
            continue
        Rp = -(-c // 16) * 16
        blk = hq[row_off * rb:(row_off + Rp) * rb]
        sblk = hs[gi * KS * A * 512:(gi + 1) * KS * A * 512]
        out[e] = (untile(blk, f, c, I, Rp), untile_scales(sblk, f, c, I))
        row_off += Rp
        gi += 1
    fs, Is = cfg["sh_fmt"], cfg["I_sh"]
    hb, sb = _hq_routed_bytes(cfg, M), _hs_routed_bytes(cfg, M)
    sh_codes = untile(hq[hb:], fs, M, Is)
    sh_sc = untile_scales(hs[sb:], fs, M, Is) if fs != 0 else None
    return out, (sh_codes, sh_sc)


def _cmp_hidden(fmt, got, ref, I, gs):
    """Requantised FC2 inputs: nearly all codes equal; dequantised values close."""
    gq, gsc = got
    rq, rsc = ref
    if fmt == 0:
        g = bf16_to_f64(gq.view(np.uint16))
        r = bf16_to_f64(rq.view(np.uint16))
        assert rel_l2(g, r) < 2e-3
        return
    same = (gq == rq).mean()
    assert same > 0.98, "only %.4f of hidden codes agree" % same
    g = oracle.dequant(fmt, gq, gsc, I, gs)
    r = oracle.dequant(fmt, rq, rsc, I, gs)
    assert rel_l2(g, r) < (2e-2 if fmt in (2, 3) else 5e-3)


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("M", [1, 5, 16, 37, 64])
def test_stages_against_oracle(name, M):
    cfg = SMALL[name]
    inp, layer = make(cfg, seed=M, M=M)
    d = layer.d
    E, k, H, I = cfg["E"], cfg["k"], cfg["H"], cfg["I"]
    L = oracle_layer(cfg, inp)
    t = _alloc(layer, M)
    li = _logits(M, E, 100 + M)
    li_d = torch.from_numpy(li).cuda()
    x16, wg16 = u16(inp["x"]), u16(inp["wg"])
    bias = npy(inp["bias"])
    # ---- a1..a3 with given logits: routing and quantisation bit-exact
    ms.moe_router_topk(d, inp["x"], inp["wg"], inp["bias"], li_d, M, t["logits"], t["idx"], t["w"], t["xq"], t["xs"],
                       t["xq_sh"], t["xs_sh"], layer.ws)
    torch.cuda.synchronize()
    _, _, oidx, ow, _ = oracle.router(L, x16, wg16, bias=bias, logits_in=li)
    assert (npy(t["idx"]) == oidx).all()
    # weights: fp32 sum and division on the GPU (a few ulps) vs the oracle's double
    assert np.allclose(npy(t["w"]), ow, rtol=2 ** -20, atol=0)
    fr, fs = cfg["w_fmt"], cfg["sh_fmt"]
    gs_a1, gs_a2, gs_a1s, gs_a2s = inp["gs_a"]
    oq, osc = oracle.quant_x(fr, x16, gs_a1)
    assert (untile(npy(t["xq"]), fr, M, H) == oq).all()
    assert (untile_scales(npy(t["xs"]), fr, M, H) == osc).all()
    xq_sh, xs_sh = (t["xq"], t["xs"]) if fs == fr else (t["xq_sh"], t["xs_sh"])
    oq_s, osc_s = oracle.quant_x(fs, x16, gs_a1s)
    assert (untile(npy(xq_sh), fs, M, H) == oq_s).all()
    if fs != 0:
        assert (untile_scales(npy(xs_sh), fs, M, H) == osc_s).all()
    # ---- a4 route: bit-exact
    ms.moe_route_tiles(d, t["idx"], M, t["tiles"], t["nt"], t["perm"], t["inv"], t["counts"], layer.ws)
    torch.cuda.synchronize()
    counts, offsets, perm, inv, tiles = oracle.route(L, oidx)
    assert (npy(t["counts"]) == counts).all()
    assert (npy(t["perm"]) == perm).all() and (npy(t["inv"]) == inv).all()
    nt = int(npy(t["nt"])[0])
    assert nt == len(tiles) and (npy(t["tiles"])[:nt] == tiles).all()
    # ---- a5 gate_up
    ms.moe_expert_gate_up(d, layer.qw["w13"], layer.qw["sh13"], t["xq"], t["xs"], xq_sh, xs_sh, t["perm"], M,
                          t["hq"], t["hs"], layer.ws)
    torch.cuda.synchronize()
    assert layer.status() == 0
    w13, w2, sh13, sh2 = host_weights(inp, E)
    xdq = oracle.dequant(fr, oq, osc, H, gs_a1)
    xdq_s = oracle.dequant(fs, oq_s, osc_s if fs else None, H, gs_a1s)
    got_h, got_sh = _gpu_hidden(cfg, M, counts, npy(t["hq"]), npy(t["hs"]))
    ref_y = {}
    for e, (gq, gsc) in got_h.items():
        rows = [perm[offsets[e] + r] for r in range(counts[e])]
        rq, rs, ys = [], [], []
        for p in rows:
            hq, hs, _, y = oracle.expert_row(fr, H, I, w13[e], w2[e], xdq[p // k], gs_a2)
            rq.append(hq)
            rs.append(hs)
            ref_y[p] = y
        _cmp_hidden(fr, (gq, gsc), (np.stack(rq), np.stack(rs) if fr else None), I, gs_a2)
    shq, shs = [], []
    for m in range(M):
        hq, hs, _, y = oracle.expert_row(fs, H, cfg["I_sh"], sh13, sh2, xdq_s[m], gs_a2s)
        shq.append(hq)
        shs.append(hs)
        ref_y[M * k + m] = y
    _cmp_hidden(fs, got_sh, (np.stack(shq), np.stack(shs) if fs else None), cfg["I_sh"], gs_a2s)
    # ---- a6 down
    ms.moe_expert_down(d, layer.qw["w2"], layer.qw["sh2"], t["hq"], t["hs"], M, t["y"], layer.ws)
    torch.cuda.synchronize()
    assert layer.status() == 0
    y = npy(t["y"])
    for p, yr in ref_y.items():
        assert rel_l2(y[inv[p]], yr) < (3e-2 if fr in (2, 3) else 1e-2), (p, rel_l2(y[inv[p]], yr))
    # ---- a5 + a6 in one launch: the same bytes as the two calls
    hq1, hs1, y1 = torch.zeros_like(t["hq"]), torch.zeros_like(t["hs"]), torch.zeros_like(t["y"])
    ms.moe_expert_ffn(d, layer.qw["w13"], layer.qw["sh13"], layer.qw["w2"], layer.qw["sh2"], t["xq"], t["xs"], xq_sh,
                      xs_sh, t["perm"], M, hq1, hs1, y1, layer.ws)
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(hq1, t["hq"]) and torch.equal(hs1, t["hs"]) and torch.equal(y1, t["y"])
    # ---- a7 finalize (with the next layer's MXFP8 input), and the whole step against the
    # oracle's own step
    res = inp["residual"].clone()
    M8 = -(-M // 8) * 8
    oq = torch.full((M8, H), 0xAB, dtype=torch.uint8, device="cuda")
    osc = torch.full((M8, H // 32), 0xAB, dtype=torch.uint8, device="cuda")
    ms.moe_finalize_norm(d, t["y"], t["w"], t["inv"], M, res, inp["gamma"], t["out"], oq, osc, layer.ws)
    torch.cuda.synchronize()
    ref = oracle.step_rows(L, np.arange(M), x16, u16(inp["residual"]), u16(inp["gamma"]), wg16, bias, w13, w2, sh13,
                           sh2, logits_in=li)
    check_output(u16(t["out"]), ref["out"], "out")
    check_output(u16(res), ref["res_out"], "residual")
    check_next_mxfp8(u16(t["out"]), npy(oq)[:M], npy(osc)[:M])
    assert (npy(oq)[M:] == 0).all() and (npy(osc)[M:] == 0).all(), "padding rows of the 8-row tiles"
    # without the optional output the other outputs are the same bytes
    res2, out2 = inp["residual"].clone(), torch.zeros_like(t["out"])
    ms.moe_finalize_norm(d, t["y"], t["w"], t["inv"], M, res2, inp["gamma"], out2, None, None, layer.ws)
    torch.cuda.synchronize()
    assert torch.equal(out2, t["out"]) and torch.equal(res2, res)


# The GEMV runs in CTAs of 4 experts x 8 rows over the whole of H. (H, E, M): one row block
# (1, 5, 8 rows), several with a ragged last one (16, 33, 48 rows), E not a multiple of 4
# (60, 62), the 256-expert layers' shapes, and 64 rows of the 512-expert layer up to H 8192.
ROUTER_CASES = [(4096, 64, 33), (4096, 64, 1), (4096, 60, 5), (4096, 64, 8), (4096, 62, 16), (7168, 256, 8),
                (6144, 256, 16), (7168, 256, 48), (4096, 512, 64), (8192, 512, 64)]


@pytest.mark.parametrize("H,E,M", ROUTER_CASES)
def test_router_gemv_logits_and_routing(H, E, M):
    cfg = synth.config("tiny_mxfp8", E=E, k=6, H=H, has_bias=True, rsf=2.5)
    inp, layer = make(cfg, seed=3 + M, M=M)
    t = _alloc(layer, M)
    ms.moe_router_topk(layer.d, inp["x"], inp["wg"], inp["bias"], None, M, t["logits"], t["idx"], t["w"], t["xq"],
                       t["xs"], t["xq_sh"], t["xs_sh"], layer.ws)
    torch.cuda.synchronize()
    L = oracle_layer(cfg, inp)
    x16, wg16 = u16(inp["x"]), u16(inp["wg"])
    ol, os_, oidx, ow, margin = oracle.router(L, x16, wg16, bias=npy(inp["bias"]))
    # fp32 accumulation bound: H * 2^-24 * sum |x w| per logit
    absdot = np.abs(bf16_to_f64(x16)) @ np.abs(bf16_to_f64(wg16)).T
    err = np.abs(npy(t["logits"]).astype(np.float64) - ol)
    assert (err <= cfg["H"] * 2 ** -24 * absdot + 1e-30).all()
    ok_rows = margin >= 1e-5
    assert ok_rows.mean() > 0.5
    assert (npy(t["idx"])[ok_rows] == oidx[ok_rows]).all()
    assert np.allclose(npy(t["w"])[ok_rows], ow[ok_rows], rtol=2 ** -20, atol=0)
    # the summation order is fixed: a second call gives the same logits, bit for bit
    first = npy(t["logits"]).copy()
    ms.moe_router_topk(layer.d, inp["x"], inp["wg"], inp["bias"], None, M, t["logits"], t["idx"], t["w"], t["xq"],
                       t["xs"], t["xq_sh"], t["xs_sh"], layer.ws)
    torch.cuda.synchronize()
    assert (npy(t["logits"]) == first).all()


@pytest.mark.parametrize("M,skew", [(1, False), (8, False), (48, True), (64, True)])
def test_route_multi_tile_bitexact(M, skew):
    cfg = synth.config("mxfp8_skew_48rows", H=1024, E=256, k=8, I=256, I_sh=256)
    inp, layer = make(cfg, seed=1, M=M)
    g = np.random.default_rng(M)
    p = (np.arange(1, 257) ** -1.2) if skew else np.ones(256)
    idx = np.stack([g.choice(256, 8, replace=False, p=p / p.sum()) for _ in range(M)]).astype(np.int32)
    t = _alloc(layer, M)
    ms.moe_route_tiles(layer.d, torch.from_numpy(idx).cuda(), M, t["tiles"], t["nt"], t["perm"], t["inv"],
                       t["counts"], layer.ws)
    torch.cuda.synchronize()
    counts, offsets, perm, inv, tiles = oracle.route(oracle_layer(cfg, inp), idx)
    assert (npy(t["counts"]) == counts).all() and (npy(t["perm"]) == perm).all()
    assert (npy(t["inv"]) == inv).all()
    nt = int(npy(t["nt"])[0])
    assert nt == len(tiles) and (npy(t["tiles"])[:nt] == tiles).all()
    if skew:
        assert (tiles[:, 2] == 8).any() and (counts[:256] > 8).any()


def test_route_rejects_out_of_range_expert_ids():
    cfg = synth.config("tiny_mxfp8")
    inp, layer = make(cfg, seed=0, M=4)
    t = _alloc(layer, 4)
    idx = torch.tensor([[0, 1], [2, 16], [3, 4], [5, 6]], dtype=torch.int32, device="cuda")
    t["nt"].fill_(-1)
    ms.moe_route_tiles(layer.d, idx, 4, t["tiles"], t["nt"], t["perm"], t["inv"], t["counts"], layer.ws)
    assert layer.status() == ms.MOE_ERR_INVALID_ARG
    assert int(npy(t["nt"])[0]) == 0
    ms.moe_workspace_init(layer.d, layer.ws)
    assert layer.status() == 0


# Ties of the selection key ("ties going to the lower index"). The GPU top-k keeps each
# lane's candidates in registers (expert e in lane e % 32) and breaks a tie between lanes
# by a second reduction, a tie inside a lane by its ascending scan; every case below is
# decided by the index rule alone, and the oracle decides it by a full sort.
def _tie_logits(M, E, k, rng):
    lg = (rng.standard_normal((M, E)) - 3.0).astype(np.float32)
    v = np.float32(5.0)
    # 0: ten equal keys over several lanes, and three in one lane (2, 34, 66), straddling the k-th slot
    lg[0, [2, 34, 66, 98, 7, 39, 11, 200, 13, 250]] = v
    # 1: every key equal: the k lowest indices
    lg[1, :] = np.float32(0.0)
    # 2: different logits whose fp32 sigmoid is the same (1.0): ties by index, then the rest
    lg[2, [40, 8, 100]] = [30.0, 25.0, 20.0]
    # 3: six distinct leaders, then three equal keys in one lane (6, 38, 70) for the last two slots
    lg[3, :6] = [9.0, 8.5, 8.0, 7.5, 7.0, 6.5]
    lg[3, [70, 38, 6]] = np.float32(2.0)
    # 4: scores of exactly zero (sigmoid underflow) fill the slots after three positive ones
    lg[4, :] = np.float32(-200.0)
    lg[4, [150, 3, 77]] = np.float32(1.0)
    # 5..: random rows with every value repeated at another expert
    for m in range(5, M):
        src = rng.permutation(E)[: E // 2]
        dst = rng.permutation(E)[: E // 2]
        lg[m, dst] = lg[m, src]
        lg[m, rng.permutation(E)[:k]] = np.float32(4.0)
    return lg


def _one_lane_logits(M, E, k, rng):
    """Rows whose top keys sit in one or two lanes of the top-k warp (experts e with the same
    e % 32), so one lane wins round after round: its next-best key is promoted, then its keys
    are scanned again after the one just taken, many times over. Some rows repeat a key inside
    the lane (exact ties in the lane's own order) or tie a lane key with another lane's."""
    lg = rng.standard_normal((M, E)).astype(np.float32)
    per_lane = E // 32
    for m in range(M):
        lanes = [m % 32] if k <= per_lane else [m % 32, (m + 7) % 32]
        ids = [ln + 32 * i for ln in lanes for i in range(per_lane)][:k + 2]
        vals = np.float32(6.0) + rng.permutation(len(ids)).astype(np.float32) * np.float32(0.25)
        if m % 3 == 1:
            vals[::3] = np.float32(7.0)  # equal keys within the lane, several of them
        lg[m, ids] = vals
        if m % 3 == 2:
            lg[m, (m + 1) % 32] = lg[m, ids[0]]  # a key of another lane equal to one of these
    return lg


@pytest.mark.parametrize("E,k", [(512, 16), (512, 10), (256, 16), (256, 8)])
def test_topk_when_one_lane_holds_the_top_keys(E, k):
    M = 24
    cfg = synth.config("tiny_mxfp8", E=E, k=k, has_bias=False, rsf=1.0)
    inp, layer = make(cfg, seed=5, M=M)
    li = _one_lane_logits(M, E, k, np.random.default_rng(E * 31 + k))
    t = _alloc(layer, M)
    ms.moe_router_topk(layer.d, inp["x"], inp["wg"], None, torch.from_numpy(li).cuda(), M, t["logits"], t["idx"],
                       t["w"], t["xq"], t["xs"], t["xq_sh"], t["xs_sh"], layer.ws)
    torch.cuda.synchronize()
    L = oracle_layer(cfg, inp)
    _, _, oidx, ow, _ = oracle.router(L, u16(inp["x"]), u16(inp["wg"]), logits_in=li)
    gidx = npy(t["idx"])
    assert (gidx == oidx).all(), "rows %s differ" % np.nonzero((gidx != oidx).any(1))[0]
    assert np.allclose(npy(t["w"]), ow, rtol=2 ** -20, atol=0)
    # the rows are what they claim to be: most of each row's top-k share one lane
    share = [np.bincount(oidx[m] % 32).max() for m in range(M)]
    assert min(share) >= min(k, E // 32) - 2


@pytest.mark.parametrize("E,k,bias", [(256, 8, False), (256, 8, True), (512, 10, True), (512, 10, False)])
def test_topk_ties_go_to_the_lower_index(E, k, bias):
    M = 12
    cfg = synth.config("tiny_mxfp8", E=E, k=k, has_bias=bias, rsf=2.5)
    inp, layer = make(cfg, seed=2, M=M)
    rng = np.random.default_rng(E + k)
    li = _tie_logits(M, E, k, rng)
    b = None
    if bias:
        # equal biases keep the ties above; on row 4 two experts get equal keys from
        # different scores: s = 0.5 (logit 0) + 0.25 and s' + (0.75 - s'), exact in fp32
        b = np.full(E, np.float32(0.125), np.float32)
        L0 = oracle_layer(dict(cfg, has_bias=False), inp)
        li[4, 9] = np.float32(0.0)
        li[4, 21] = np.float32(1.7)
        _, sc, _, _, _ = oracle.router(L0, u16(inp["x"]), u16(inp["wg"]), logits_in=li)
        b[9] = np.float32(0.25)
        b[21] = np.float32(np.float32(0.75) - sc[4, 21])
        assert np.float32(sc[4, 9] + b[9]) == np.float32(sc[4, 21] + b[21]) == np.float32(0.75)
        assert sc[4, 9] != sc[4, 21]
        inp["bias"] = torch.from_numpy(b).cuda()
    t = _alloc(layer, M)
    ms.moe_router_topk(layer.d, inp["x"], inp["wg"], inp["bias"] if bias else None, torch.from_numpy(li).cuda(), M,
                       t["logits"], t["idx"], t["w"], t["xq"], t["xs"], t["xq_sh"], t["xs_sh"], layer.ws)
    torch.cuda.synchronize()
    L = oracle_layer(cfg, inp)
    _, _, oidx, ow, _ = oracle.router(L, u16(inp["x"]), u16(inp["wg"]), bias=b, logits_in=li)
    gidx = npy(t["idx"])
    assert (gidx == oidx).all(), "rows %s differ" % np.nonzero((gidx != oidx).any(1))[0]
    assert np.allclose(npy(t["w"]), ow, rtol=2 ** -20, atol=0)
    # the cases are what they claim to be
    if not bias:  # (with the bias, experts 9 and 21 lead row 1)
        assert list(oidx[1]) == list(range(k))
    assert oidx[0][:min(k, 10)].tolist() == sorted([2, 34, 66, 98, 7, 39, 11, 200, 13, 250])[:min(k, 10)]
    assert oidx[2][:3].tolist() == [8, 40, 100]
    if bias:
        assert 9 in oidx[4] and 21 in oidx[4] and list(oidx[4]).index(9) < list(oidx[4]).index(21)
