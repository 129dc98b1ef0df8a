"""Pins of the oracle's expert FFN (a5, a6), finalize (a7) and whole-row step.

Expert: closed forms with constant operands, one-hot FC2 rows (linearity), and a
brute-force numpy computation that decodes the codes with PyTorch's float8 view and
a format table, then multiplies in float64.
Finalize: constant rows, scale invariance of RMSNorm, and the bf16 rounding of the
residual checked with PyTorch's cast.
Step: the whole-row step equals the composition of the stages, and is invariant to
the order of the rows it is given.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import FMT_BF16, FMT_MXFP4, FMT_MXFP8, FMT_NVFP4
from moe_decode_step_router_gb300 import synth

E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])


def _deq_indep(fmt, vals, scales, gs, K):
    """Independent decode: torch float8/bf16 views, the E2M1 table, 2^(s-127)."""
    vals = np.asarray(vals)
    if fmt == FMT_MXFP8:
        v = torch.from_numpy(np.ascontiguousarray(vals)).view(torch.float8_e4m3fn).double().numpy()
        s = np.ldexp(1.0, scales.astype(np.int64) - 127)
        return v * np.repeat(s, 32, axis=-1)
    if fmt in (FMT_NVFP4, FMT_MXFP4):
        lo, hi = vals & 15, vals >> 4
        nib = np.stack([lo, hi], axis=-1).reshape(vals.shape[:-1] + (K,))
        if fmt == FMT_MXFP4:
            return E2M1[nib] * np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=-1)
        s = torch.from_numpy(np.ascontiguousarray(scales)).view(torch.float8_e4m3fn).double().numpy()
        return E2M1[nib] * np.repeat(s, 16, axis=-1) * float(gs)
    return torch.from_numpy(np.ascontiguousarray(vals)).view(torch.bfloat16).double().numpy()


def _mx_const(rows, K, code, sbyte):
    return np.full((rows, K), code, np.uint8), np.full((rows, K // 32), sbyte, np.uint8)


def test_expert_closed_form_mxfp8():
    H, I = 64, 32
    # gate rows = 2^-7 (code 1.0, scale 2^-7), up rows = 2^-6; x = 1 dequantised
    v13 = np.concatenate([np.full((I, H), 0x38, np.uint8), np.full((I, H), 0x38, np.uint8)])
    s13 = np.concatenate([np.full((I, H // 32), 120, np.uint8), np.full((I, H // 32), 121, np.uint8)])
    v2, s2 = _mx_const(H, I, 0x38, 127)
    hq, hs, h, y = oracle.expert_row(FMT_MXFP8, H, I, (v13, s13, 1.0), (v2, s2, 1.0), np.ones(H))
    g, u = H * 2.0 ** -7, H * 2.0 ** -6           # 0.5 and 1.0
    want = g / (1 + math.exp(-g)) * u
    assert np.all(h == want)
    hd = oracle.dequant(FMT_MXFP8, hq[None], hs[None], I)[0]
    assert np.allclose(y, I * hd[0])              # W2 == 1 everywhere: y_n = sum_i hq_i


@pytest.mark.parametrize("gsign,usign", [(1, 1), (-1, 1), (1, -1), (-1, -1)])
def test_expert_clamped_swiglu_closed_form(gsign, usign):
    # Clamped SwiGLU ("SGLang-NVIDIA-Mega" README, shared_ll row): g -> min(g, L),
    # u -> clamp(u, -L, L), then silu(g) u. |g| = 0.5, |u| = 1.0 and L = 0.25: a positive
    # gate is cut to L, a negative one is left alone (upper bound only), u is cut either way.
    H, I, L = 64, 32, 0.25
    gcode, ucode = (0x38 if gsign > 0 else 0xB8), (0x38 if usign > 0 else 0xB8)   # +-1.0 in E4M3
    v13 = np.concatenate([np.full((I, H), gcode, np.uint8), np.full((I, H), ucode, np.uint8)])
    s13 = np.concatenate([np.full((I, H // 32), 120, np.uint8), np.full((I, H // 32), 121, np.uint8)])
    v2, s2 = _mx_const(H, I, 0x38, 127)
    _, _, h, _ = oracle.expert_row(FMT_MXFP8, H, I, (v13, s13, 1.0), (v2, s2, 1.0), np.ones(H), limit=L)
    g = 0.5 * gsign
    g = L if g > L else g
    u = L * usign
    assert np.all(h == g / (1 + math.exp(-g)) * u)
    # a limit above every |g| and |u| changes nothing; a limit <= 0 means unclamped
    _, _, h_off, _ = oracle.expert_row(FMT_MXFP8, H, I, (v13, s13, 1.0), (v2, s2, 1.0), np.ones(H), limit=0.0)
    _, _, h_big, _ = oracle.expert_row(FMT_MXFP8, H, I, (v13, s13, 1.0), (v2, s2, 1.0), np.ones(H), limit=4.0)
    g0, u0 = 0.5 * gsign, 1.0 * usign
    assert np.all(h_off == g0 / (1 + math.exp(-g0)) * u0) and np.all(h_big == h_off)


def test_expert_clamped_swiglu_brute_force():
    H, I = 128, 64
    g = synth._gen(7, "cpu")
    v13, s13, gs13 = [t.numpy() if t is not None else None for t in synth.weight(FMT_MXFP8, 1, 2 * I, H, g, "cpu")]
    v2, s2, gs2 = [t.numpy() if t is not None else None for t in synth.weight(FMT_MXFP8, 1, H, I, g, "cpu")]
    xdq = np.random.default_rng(17).standard_normal(H) * 8.0
    W13 = _deq_indep(FMT_MXFP8, v13[0], s13[0], 1.0, H)
    gg, uu = W13[:I] @ xdq, W13[I:] @ xdq
    L = float(np.median(np.abs(np.concatenate([gg, uu]))))   # about half the values are cut
    _, _, h, _ = oracle.expert_row(FMT_MXFP8, H, I, (v13[0], s13[0], 1.0), (v2[0], s2[0], 1.0), xdq, limit=L)
    gc, uc = np.minimum(gg, L), np.clip(uu, -L, L)
    assert (gg > L).any() and (np.abs(uu) > L).any() and (gg < -L).any()
    assert np.allclose(h, gc / (1 + np.exp(-gc)) * uc, rtol=1e-12, atol=1e-12)


def test_expert_fc2_one_hot_rows():
    rng = np.random.default_rng(12)
    H, I = 64, 64
    v13 = rng.integers(0, 0x7E, (2 * I, H), dtype=np.uint8)
    s13 = rng.integers(118, 124, (2 * I, H // 32), dtype=np.uint8)
    v2 = np.zeros((H, I), np.uint8)
    s2 = np.full((H, I // 32), 127, np.uint8)
    col = rng.integers(0, I, H)
    v2[np.arange(H), col] = 0x38                  # W2[n, col[n]] = 1
    xdq = rng.standard_normal(H)
    hq, hs, h, y = oracle.expert_row(FMT_MXFP8, H, I, (v13, s13, 1.0), (v2, s2, 1.0), xdq)
    hd = oracle.dequant(FMT_MXFP8, hq[None], hs[None], I)[0]
    assert np.all(y == hd[col])


@pytest.mark.parametrize("fmt", [FMT_MXFP8, FMT_NVFP4, FMT_MXFP4, FMT_BF16])
def test_expert_brute_force(fmt):
    H, I = 128, 64
    g = synth._gen(5, "cpu")
    v13, s13, gs13 = [t.numpy() if t is not None else None for t in synth.weight(fmt, 1, 2 * I, H, g, "cpu")]
    v2, s2, gs2 = [t.numpy() if t is not None else None for t in synth.weight(fmt, 1, H, I, g, "cpu")]
    xdq = np.random.default_rng(13).standard_normal(H)
    w13 = (v13[0], None if s13 is None else s13[0], gs13[0])
    w2 = (v2[0], None if s2 is None else s2[0], gs2[0])
    gs_a2 = 2.0 ** -6 if fmt == FMT_NVFP4 else 1.0
    hq, hs, h, y = oracle.expert_row(fmt, H, I, w13, w2, xdq, gs_a2)
    W13 = _deq_indep(fmt, w13[0], w13[1], w13[2], H)
    W2 = _deq_indep(fmt, w2[0], w2[1], w2[2], I)
    gg, uu = W13[:I] @ xdq, W13[I:] @ xdq
    h_ref = gg / (1 + np.exp(-gg)) * uu
    assert np.allclose(h, h_ref, rtol=1e-12, atol=1e-12)
    hd = _deq_indep(fmt, hq, hs if hs.size else None, gs_a2, I)
    assert np.allclose(y, W2 @ hd, rtol=1e-12, atol=1e-12)
    # the requantised h is within the format's rounding bound of h
    err = np.abs(hd - h_ref)
    if fmt == FMT_MXFP8:      # 3 mantissa bits: half an ulp is 2^-4 relative (normal range)
        blk = np.repeat(np.abs(h_ref).reshape(-1, 32).max(1), 32)
        assert (err <= 2 ** -4 * np.abs(h_ref) + blk * 2 ** -17).all()
    elif fmt == FMT_NVFP4:    # largest E2M1 half-gap is 1 (between 4 and 6) of a block max near 6
        blk = np.repeat(np.abs(h_ref).reshape(-1, 16).max(1), 16)
        assert (err <= blk * (1.0 / 6.0) * (1 + 2 ** -3)).all()
    elif fmt == FMT_MXFP4:    # half-gap 1 at scale 2^e, block max in (3, 6] * 2^e (plus fp32 of h)
        blk = np.repeat(np.abs(h_ref).reshape(-1, 32).max(1), 32)
        assert (err <= blk / 3.0 * (1 + 2 ** -20)).all()
    else:
        assert (err <= 2 ** -8 * np.abs(h_ref)).all()


def _bf16(a):
    t = torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().astype(np.uint16)


def _layer(H):
    return oracle.make_layer(dict(H=H, E=4, k=2, I=32, I_sh=32, w_fmt=FMT_MXFP8, sh_fmt=FMT_MXFP8,
                                  has_bias=False, rsf=1.0, eps=1e-6))


def test_finalize_constant_row():
    H = 256
    L = _layer(H)
    gamma = _bf16(np.linspace(0.5, 1.5, H))
    out, res, _, _ = oracle.finalize_row(L, np.zeros(H), _bf16(np.full(H, -3.0)), gamma)
    ref = torch.from_numpy(gamma.astype(np.int16)).view(torch.bfloat16).double().numpy()
    got = torch.from_numpy(out.astype(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.allclose(got, -ref * 3.0 / math.sqrt(9.0 + 1e-6), rtol=2 ** -8)
    assert (res == _bf16(np.full(H, -3.0))).all()


@pytest.mark.parametrize("H", [256, 1280])
def test_finalize_rmsnorm_exact_mean_square(H):
    """Rows whose mean square is exact, so RMSNorm has a closed form (moe = 0).

    |residual| = 2 everywhere: mean square 4, (4 + 1e-6)^-1/2 = 0.5 (1 - 1.25e-7), and
    out = bf16(r / 2 * gamma) = +-gamma bit for bit (the factor 1 - 1.25e-7 is far below
    half a bf16 ulp). A wrong mean (dividing by H - 1 or H + 1) moves out by 1 / (2H),
    which moves gamma = 1 to another bf16 value at H = 256. 3/8 of the entries +-3 and
    5/8 +-1 also give mean square 4 (9 * 3/8 + 5/8). eps = 12 with |r| = 2 gives
    (4 + 12)^-1/2 = 1/4 exactly: eps inside the square root."""
    rng = np.random.default_rng(H)
    sign = rng.choice([-1.0, 1.0], H)
    grid = np.array([0.5, 0.75, 1.0, 1.25, 1.5, 1.75])  # 1.5 * grid and grid / 4 stay on the bf16 grid
    gam = rng.choice(grid, H)
    gam[:8] = 1.0
    gamma = _bf16(gam)
    b2f = lambda a: torch.from_numpy(a.astype(np.int16)).view(torch.bfloat16).double().numpy()
    L = _layer(H)
    out, res, _, _ = oracle.finalize_row(L, np.zeros(H), _bf16(2.0 * sign), gamma)
    assert (out == _bf16(sign * gam)).all()
    assert (res == _bf16(2.0 * sign)).all()
    mag = np.where(rng.permutation(H) < 3 * H // 8, 3.0, 1.0)
    assert (mag ** 2).mean() == 4.0
    out, _, _, _ = oracle.finalize_row(L, np.zeros(H), _bf16(mag * sign), gamma)
    assert (b2f(out) == mag * sign * 0.5 * gam).all()
    L12 = oracle.make_layer(dict(H=H, E=4, k=2, I=32, I_sh=32, w_fmt=FMT_MXFP8, sh_fmt=FMT_MXFP8, has_bias=False,
                                 rsf=1.0, eps=12.0))
    out, _, _, _ = oracle.finalize_row(L12, np.zeros(H), _bf16(2.0 * sign), gamma)
    assert (b2f(out) == sign * 0.5 * gam).all()


def test_finalize_scale_invariance_and_residual_rounding():
    rng = np.random.default_rng(14)
    H = 512
    L = _layer(H)
    gamma = _bf16(rng.standard_normal(H) * 0.1 + 1)
    res16 = _bf16(rng.standard_normal(H))
    # moe on the bf16 grid, so residual + moe (two 8-bit significands) is exact in fp32
    moe = torch.from_numpy(rng.standard_normal(H).astype(np.float32)).to(torch.bfloat16).double().numpy()
    out1, r1, _, _ = oracle.finalize_row(L, moe, res16, gamma)
    resd = torch.from_numpy(res16.astype(np.int16)).view(torch.bfloat16).double().numpy()
    # the fp32 sum is exact, so torch's fp32 -> bf16 cast rounds once, like the oracle
    s32 = (resd + moe).astype(np.float32)
    assert np.all(s32.astype(np.float64) == resd + moe)
    assert (r1 == _bf16(s32)).all()
    for j in (-4, 3):
        out2, r2, _, _ = oracle.finalize_row(L, moe * 2.0 ** j, _bf16(resd * 2.0 ** j), gamma)
        a = torch.from_numpy(out1.astype(np.int16)).view(torch.bfloat16).double().numpy()
        b = torch.from_numpy(out2.astype(np.int16)).view(torch.bfloat16).double().numpy()
        assert np.abs(a - b).max() <= 2 ** -7 * np.abs(a).max()


def test_finalize_next_layer_quant():
    rng = np.random.default_rng(15)
    H = 256
    L = _layer(H)
    out, _, q, s = oracle.finalize_row(L, rng.standard_normal(H), _bf16(rng.standard_normal(H)),
                                       _bf16(np.ones(H)), want_q=True)
    outf = torch.from_numpy(out.astype(np.int16)).view(torch.bfloat16).float().numpy()
    q2, s2 = oracle.quant(FMT_MXFP8, outf[None])
    assert (q == q2[0]).all() and (s == s2[0]).all()


def _tiny(seed=0, M=5):
    cfg = synth.config("tiny_mxfp8", M=M, H=256, E=8, k=3, I=64, I_sh=64, has_bias=True, rsf=2.5)
    d = synth.make_inputs(cfg, seed)
    L = oracle.make_layer(cfg, d["gs_a"])
    n = lambda t: t.numpy() if t is not None else None
    x = d["x"].view(torch.int16).numpy().astype(np.uint16)
    res = d["residual"].view(torch.int16).numpy().astype(np.uint16)
    gam = d["gamma"].view(torch.int16).numpy().astype(np.uint16)
    wg = d["wg"].view(torch.int16).numpy().astype(np.uint16)
    w13 = [(d["w13"][0][e].numpy(), d["w13"][1][e].numpy(), float(d["w13"][2][e])) for e in range(8)]
    w2 = [(d["w2"][0][e].numpy(), d["w2"][1][e].numpy(), float(d["w2"][2][e])) for e in range(8)]
    sh13 = (d["sh13"][0][0].numpy(), d["sh13"][1][0].numpy(), 1.0)
    sh2 = (d["sh2"][0][0].numpy(), d["sh2"][1][0].numpy(), 1.0)
    return cfg, L, x, res, gam, wg, n(d["bias"]), w13, w2, sh13, sh2


def test_step_equals_stage_composition():
    cfg, L, x, res, gam, wg, bias, w13, w2, sh13, sh2 = _tiny()
    M = x.shape[0]
    st = oracle.step_rows(L, np.arange(M), x, res, gam, wg, bias, w13, w2, sh13, sh2, want_q=True)
    _, _, idx, w, _ = oracle.router(L, x, wg, bias)
    assert (st["topk_idx"] == idx).all()
    xq, xs = oracle.quant_x(FMT_MXFP8, x)
    xdq = oracle.dequant(FMT_MXFP8, xq, xs, cfg["H"])
    for m in range(M):
        moe = np.zeros(cfg["H"])
        for j in range(cfg["k"]):
            _, _, _, y = oracle.expert_row(FMT_MXFP8, cfg["H"], cfg["I"], w13[idx[m, j]], w2[idx[m, j]], xdq[m])
            moe += w[m, j] * y
        _, _, _, ys = oracle.expert_row(FMT_MXFP8, cfg["H"], cfg["I_sh"], sh13, sh2, xdq[m])
        out, ro, q, s = oracle.finalize_row(L, moe + ys, res[m], gam, want_q=True)
        assert (out == st["out"][m]).all() and (ro == st["res_out"][m]).all()
        assert (q == st["outq"][m]).all() and (s == st["outs"][m]).all()


def test_step_row_map_invariance():
    cfg, L, x, res, gam, wg, bias, w13, w2, sh13, sh2 = _tiny(seed=3, M=6)
    a = oracle.step_rows(L, np.arange(6), x, res, gam, wg, bias, w13, w2, sh13, sh2)
    p = np.array([4, 1, 5, 0, 3, 2])
    b = oracle.step_rows(L, np.arange(6), x[p], res[p], gam, wg, bias, w13, w2, sh13, sh2)
    assert (a["out"][p] == b["out"]).all() and (a["res_out"][p] == b["res_out"]).all()
    c = oracle.step_rows(L, p, x, res, gam, wg, bias, w13, w2, sh13, sh2)
    assert (a["out"][p] == c["out"]).all()


def test_step_missing_expert_raises():
    cfg, L, x, res, gam, wg, bias, w13, w2, sh13, sh2 = _tiny()
    with pytest.raises(KeyError):
        oracle.step_rows(L, [0], x, res, gam, wg, bias, [None] * 8, [None] * 8, sh13, sh2)
