"""Seeded synthetic inputs for the MoE step, in canonical layouts.

Both the CUDA path and the CPU oracle are fed from here. The module holds none of
the step's arithmetic: it draws random numbers and stores them in the weight and
activation formats (library casts only), so neither side can borrow the other's
quantisation, routing or GEMM code from it.

Recipes (all seeded):
  x, residual  bf16 N(0, 1)                         gamma  bf16 N(1, 0.1)
  router gate  bf16 N(0, 0.02)                      bias   fp32 N(0, 0.01) where named
  MXFP8 weight per 32-block: exponent e uniform in {-12, -11, -10}; code = E4M3 cast of
               clamp(N(0, 0.02) * 2^-e, +-448); scale byte = 127 + e (decodes ~ N(0, 0.02))
  NVFP4 weight E2M1 codes drawn from a fixed magnitude table (random sign); E4M3 block
               scale bytes uniform in [0x30, 0x40] (0.5 .. 2.0); per-expert fp32 global
               scale 2^-8 * (1 + U(0, 1)/4)
  MXFP4 weight E2M1 codes drawn from the same magnitude table (random sign); E8M0 scale
               bytes uniform in {119, 120} (2^-8, 2^-7): values up to ~0.05, ~N(0, 0.01)
  BF16 weight  bf16 N(0, 0.02)
  NVFP4 static activation scales: FC1 input 2^-8, FC2 input 2^-6 (plain constants).
  Skewed routing: the selection bias adds beta * r_e^-1.2 over a seeded permutation r of
               the ranks 1..E; beta is a stored constant chosen so that about 40% of the
               experts are idle at 48 rows (see oracle/calibrate_skew.py).
"""
from __future__ import annotations

import torch

FMT_BF16, FMT_MXFP8, FMT_NVFP4, FMT_MXFP4 = 0, 1, 2, 3
FMT_NAMES = {FMT_BF16: "bf16", FMT_MXFP8: "mxfp8", FMT_NVFP4: "nvfp4", FMT_MXFP4: "mxfp4"}

# Magnitude index 0..7 of E2M1 (0, .5, 1, 1.5, 2, 3, 4, 6): draw probabilities.
NVFP4_MAG_PROBS = (0.10, 0.18, 0.17, 0.15, 0.13, 0.12, 0.09, 0.06)
GS_A1_NVFP4 = 2.0 ** -8
GS_A2_NVFP4 = 2.0 ** -6
# Selection-bias amplitude of the skewed config (written by oracle/calibrate_skew.py).
SKEW_BETA = 1.0149

_BASE = dict(has_shared=True, renormalize=True, eps=1e-6, emit_next=False, skew=False, has_bias=False,
             rsf=1.0)

CONFIGS = {
    # 1 row, MXFP8, the small case the oracle finishes in seconds.
    "tiny_mxfp8": dict(_BASE, M=1, H=1024, E=16, k=2, I=256, I_sh=256, w_fmt=FMT_MXFP8, sh_fmt=FMT_MXFP8),
    # 8 rows, MXFP8 routed + shared, selection bias, rsf 2.5: the headline workload.
    "mxfp8_h7168_e256_k8_8rows": dict(_BASE, M=8, H=7168, E=256, k=8, I=2048, I_sh=2048, w_fmt=FMT_MXFP8,
                                      sh_fmt=FMT_MXFP8, has_bias=True, rsf=2.5),
    # 16 rows, NVFP4 routed, BF16 shared.
    "nvfp4_h6144_e256_k8_16rows": dict(_BASE, M=16, H=6144, E=256, k=8, I=2048, I_sh=2048, w_fmt=FMT_NVFP4,
                                       sh_fmt=FMT_BF16),
    # 48 rows, MXFP8, Zipf-skewed selection, emits the next layer's MXFP8 input.
    "mxfp8_skew_48rows": dict(_BASE, M=48, H=7168, E=256, k=8, I=2048, I_sh=2048, w_fmt=FMT_MXFP8,
                              sh_fmt=FMT_MXFP8, has_bias=True, rsf=2.5, skew=True, emit_next=True),
    # Packed MXFP4 routed experts (the pages' packed-MXFP4 decode steps of 1-8, 16, 32 and
    # 64 rows give no shapes: the headline's are used) + MXFP8 shared.
    "mxfp4_h7168_e256_k8": dict(_BASE, M=8, H=7168, E=256, k=8, I=2048, I_sh=2048, w_fmt=FMT_MXFP4,
                                sh_fmt=FMT_MXFP8),
    # Row sweep on H 4096, 512 experts, top-10, NVFP4 routed + MXFP8 shared.
    "nvfp4_h4096_e512_k10": dict(_BASE, M=8, H=4096, E=512, k=10, I=1024, I_sh=1024, w_fmt=FMT_NVFP4,
                                 sh_fmt=FMT_MXFP8),
}
SWEEP_ROWS = (1, 2, 4, 8, 16, 32, 48, 64)


def config(name, **over):
    c = dict(CONFIGS[name])
    c.update(over)
    c["name"] = name
    return c


def act_global_scales(cfg):
    """(gs_a1, gs_a2, gs_a1_shared, gs_a2_shared): 1.0 unless the format is NVFP4."""
    a = (GS_A1_NVFP4, GS_A2_NVFP4) if cfg["w_fmt"] == FMT_NVFP4 else (1.0, 1.0)
    s = (GS_A1_NVFP4, GS_A2_NVFP4) if cfg["sh_fmt"] == FMT_NVFP4 else (1.0, 1.0)
    return a + s


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _bf16(shape, mean, std, g, device):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std + mean
    return t.to(torch.bfloat16)


def _row_bytes(fmt, K):
    return 2 * K if fmt == FMT_BF16 else (K if fmt == FMT_MXFP8 else K // 2)


def _row_scales(fmt, K):
    return K // 32 if fmt in (FMT_MXFP8, FMT_MXFP4) else (K // 16 if fmt == FMT_NVFP4 else 0)


def weight(fmt, n_exp, rows, K, g, device, chunk_elems=1 << 28):
    """Random weights [n_exp, rows, K] in `fmt`: (codes uint8, scales uint8 | None, gs fp32 [n_exp])."""
    rb, rs = _row_bytes(fmt, K), _row_scales(fmt, K)
    vals = torch.empty((n_exp, rows, rb), dtype=torch.uint8, device=device)
    scales = torch.empty((n_exp, rows, rs), dtype=torch.uint8, device=device) if rs else None
    gs = torch.ones(n_exp, dtype=torch.float32, device=device)
    per = max(1, chunk_elems // max(1, rows * K))
    for e0 in range(0, n_exp, per):
        e1 = min(n_exp, e0 + per)
        n = e1 - e0
        if fmt == FMT_BF16:
            w = torch.randn((n, rows, K), generator=g, device=device) * 0.02
            vals[e0:e1] = w.to(torch.bfloat16).view(torch.uint8).reshape(n, rows, rb)
        elif fmt == FMT_MXFP8:
            ex = torch.randint(-12, -9, (n, rows, K // 32), generator=g, device=device)
            w = torch.randn((n, rows, K // 32, 32), generator=g, device=device) * 0.02
            w = (w * torch.exp2(-ex.float()).unsqueeze(-1)).clamp_(-448.0, 448.0)
            vals[e0:e1] = w.to(torch.float8_e4m3fn).view(torch.uint8).reshape(n, rows, K)
            scales[e0:e1] = (ex + 127).to(torch.uint8)
        else:
            probs = torch.tensor(NVFP4_MAG_PROBS, device=device)
            mag = torch.multinomial(probs, n * rows * K, replacement=True, generator=g).reshape(n, rows, K)
            sign = torch.randint(0, 2, (n, rows, K), generator=g, device=device)
            nib = (mag + 8 * sign).to(torch.uint8)
            vals[e0:e1] = nib[..., 0::2] | (nib[..., 1::2] << 4)
            if fmt == FMT_MXFP4:
                scales[e0:e1] = torch.randint(119, 121, (n, rows, K // 32), generator=g,
                                              device=device).to(torch.uint8)
            else:
                scales[e0:e1] = torch.randint(0x30, 0x41, (n, rows, K // 16), generator=g,
                                              device=device).to(torch.uint8)
                gs[e0:e1] = (2.0 ** -8) * (1.0 + 0.25 * torch.rand(n, generator=g, device=device))
    return vals, scales, gs


def skew_bias(E, g, device, beta=SKEW_BETA):
    """Zipf(s=1.2) selection-bias term beta * r_e^-1.2 over a seeded permutation of ranks 1..E."""
    ranks = torch.randperm(E, generator=g, device=device).to(torch.float64) + 1.0
    return (beta * ranks.pow(-1.2)).to(torch.float32)


def make_inputs(cfg, seed=0, device="cpu", M=None, weights=True):
    """All inputs of one step of `cfg`, canonical layouts, as torch tensors on `device`."""
    M = cfg["M"] if M is None else M
    H, E, I, Ish = cfg["H"], cfg["E"], cfg["I"], cfg["I_sh"]
    # activations, router gate and bias come from the CPU generator on every machine,
    # so the routing of a seed is the same wherever the weights are drawn
    g = _gen(seed, "cpu")
    d = {}
    d["x"] = _bf16((M, H), 0.0, 1.0, g, "cpu").to(device)
    d["residual"] = _bf16((M, H), 0.0, 1.0, g, "cpu").to(device)
    d["gamma"] = _bf16((H,), 1.0, 0.1, g, "cpu").to(device)
    d["wg"] = _bf16((E, H), 0.0, 0.02, g, "cpu").to(device)
    bias = None
    if cfg["has_bias"]:
        bias = torch.randn(E, generator=g) * 0.01
        if cfg.get("skew"):
            bias = bias + skew_bias(E, _gen(seed + 7919, "cpu"), "cpu")
        bias = bias.to(device)
    d["bias"] = bias
    if weights:
        d["w13"] = weight(cfg["w_fmt"], E, 2 * I, H, _gen(seed + 1, device), device)
        d["w2"] = weight(cfg["w_fmt"], E, H, I, _gen(seed + 2, device), device)
        if cfg["has_shared"]:
            d["sh13"] = weight(cfg["sh_fmt"], 1, 2 * Ish, H, _gen(seed + 3, device), device)
            d["sh2"] = weight(cfg["sh_fmt"], 1, H, Ish, _gen(seed + 4, device), device)
    d["gs_a"] = act_global_scales(cfg)
    return d


def step_inputs(cfg, seed, device="cpu", M=None):
    """Only the per-step activations (x, residual) for another seed (weights unchanged)."""
    M = cfg["M"] if M is None else M
    g = _gen(seed, "cpu")
    x = _bf16((M, cfg["H"]), 0.0, 1.0, g, "cpu").to(device)
    r = _bf16((M, cfg["H"]), 0.0, 1.0, g, "cpu").to(device)
    return x, r


def unique_weight_bytes(cfg, n_active_experts):
    """Bytes a step must stream: selected experts' W13+W2 codes, block scales and global
    scales, the shared expert's, and the router gate."""
    H, I, Ish, E = cfg["H"], cfg["I"], cfg["I_sh"], cfg["E"]

    def proj(fmt, rows, K):
        return rows * (_row_bytes(fmt, K) + _row_scales(fmt, K)) + (4 if fmt == FMT_NVFP4 else 0)

    per_exp = proj(cfg["w_fmt"], 2 * I, H) + proj(cfg["w_fmt"], H, I)
    sh = (proj(cfg["sh_fmt"], 2 * Ish, H) + proj(cfg["sh_fmt"], H, Ish)) if cfg["has_shared"] else 0
    return n_active_experts * per_exp + sh + E * H * 2


def expected_active(cfg, M=None):
    M = cfg["M"] if M is None else M
    E, k = cfg["E"], cfg["k"]
    return E * (1.0 - (1.0 - k / E) ** M)


