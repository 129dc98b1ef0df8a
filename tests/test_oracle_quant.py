"""Pins of the oracle's MXFP8 / NVFP4 block quantisation.

Checked against: hand cases, the scale-rule property (the block maximum lands in
(224, 448] after scaling), grid round trips, and an independent implementation that
picks the exponent by a power-of-two search and rounds with PyTorch's E4M3 cast or a
brute-force E2M1 nearest-even search.
"""
import math

import numpy as np
import torch

import oracle
from oracle import FMT_MXFP4, FMT_MXFP8, FMT_NVFP4

E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_mxfp8_block_of_ones():
    q, s = oracle.quant(FMT_MXFP8, np.ones((1, 32), np.float32))
    assert s[0, 0] == 119          # 448 * 2^-9 < 1 <= 448 * 2^-8
    assert (q == 0x78).all()       # 1 * 2^8 = 256 = E4M3 0x78


def test_mxfp8_zero_block():
    q, s = oracle.quant(FMT_MXFP8, np.zeros((1, 32), np.float32))
    assert s[0, 0] == 0 and (q == 0).all()


def test_mxfp8_scale_rule_property():
    rng = np.random.default_rng(4)
    for scale in (1e-20, 1e-3, 1.0, 3.0, 1e5, 1e30):
        v = (rng.standard_normal((64, 32)) * scale).astype(np.float32)
        q, s = oracle.quant(FMT_MXFP8, v)
        for r in range(64):
            e = int(s[r, 0]) - 127
            amax = float(np.abs(v[r]).max())
            t = amax * 2.0 ** -e
            assert 224.0 < t <= 448.0, (scale, r, t)


def _mxfp8_independent(v):
    """Exponent by a power-of-two search; elements by PyTorch's RNE E4M3 cast."""
    R, K = v.shape
    q = np.zeros((R, K), np.uint8)
    s = np.zeros((R, K // 32), np.uint8)
    for r in range(R):
        for b in range(K // 32):
            blk = v[r, 32 * b:32 * b + 32]
            amax = float(np.abs(blk).max())
            e = -127
            while amax > 448.0 * 2.0 ** e:
                e += 1
            s[r, b] = e + 127
            t = torch.from_numpy((blk * np.float32(2.0 ** -e)).astype(np.float32))
            q[r, 32 * b:32 * b + 32] = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return q, s


def test_mxfp8_matches_independent():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((16, 256)) * rng.choice([1e-2, 1.0, 50.0], size=(16, 1))).astype(np.float32)
    v[3, 5] = 0.0
    v[4, :32] = 0.0
    q, s = oracle.quant(FMT_MXFP8, v)
    q2, s2 = _mxfp8_independent(v)
    assert (q == q2).all() and (s == s2).all()


def test_mxfp8_grid_roundtrip():
    rng = np.random.default_rng(6)
    codes = rng.integers(0, 0x7E, size=(8, 64), dtype=np.uint8) | (rng.integers(0, 2, (8, 64)) * 0x80).astype(np.uint8)
    codes[:, 0] = 0x7E                      # 448 in each first block -> the rule returns the same exponent
    codes[:, 32] = 0xF8                     # -256 in each second block (in (224, 448])
    scales = rng.integers(100, 140, size=(8, 2), dtype=np.uint8)
    v = oracle.dequant(FMT_MXFP8, codes, scales, 64).astype(np.float32)
    q, s = oracle.quant(FMT_MXFP8, v)
    assert (s == scales).all() and (q == codes).all()


def test_mxfp8_dequant_values():
    q = np.array([[0x38] * 32 + [0xB8] * 32], np.uint8)
    s = np.array([[127, 130]], np.uint8)
    d = oracle.dequant(FMT_MXFP8, q, s, 64)
    assert (d[0, :32] == 1.0).all() and (d[0, 32:] == -8.0).all()


def test_nvfp4_hand_case():
    gs = 2.0 ** -8
    v = np.full((1, 16), 6.0 * gs, np.float32)       # amax/(6 gs) = 1 -> scale 1.0 (0x38)
    v[0, 1] = -3.0 * gs
    q, s = oracle.quant(FMT_NVFP4, v, gs)
    assert s[0, 0] == 0x38
    assert q[0, 0] == (0x7 | (0xD << 4))             # 6 in the low nibble, -3 in the high one
    assert (q[0, 1:] == 0x77).all()


def _e2m1_brute(x):
    a = min(abs(x), 6.0)
    best = None
    for code, g in enumerate(E2M1_GRID):
        d = abs(a - g)
        if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
            best = (d, code)
    return best[1] | (8 if math.copysign(1.0, x) < 0 else 0)


def test_nvfp4_matches_independent():
    rng = np.random.default_rng(7)
    gs = np.float32(0.0071)
    v = (rng.standard_normal((6, 64)) * rng.choice([0.01, 1.0, 20.0], size=(6, 1))).astype(np.float32)
    v[2, :16] = 0.0
    q, s = oracle.quant(FMT_NVFP4, v, float(gs))
    for r in range(6):
        for b in range(4):
            blk = v[r, 16 * b:16 * b + 16]
            amax = np.float32(np.abs(blk).max())
            sf = np.float32(amax / np.float32(np.float32(6.0) * gs))
            sc = int(torch.tensor([min(sf, 448.0)]).to(torch.float8_e4m3fn).view(torch.uint8)[0])  # satfinite
            assert s[r, b] == sc
            dsc = float(torch.tensor([sc], dtype=torch.uint8).view(torch.float8_e4m3fn).float()[0])
            denom = np.float32(np.float32(dsc) * gs)
            for i in range(16):
                want = 0 if dsc == 0 else _e2m1_brute(float(np.float32(blk[i] / denom)))
                byte = q[r, 8 * b + i // 2]
                got = (byte >> 4) if i & 1 else (byte & 15)
                assert got == want, (r, b, i)


def test_nvfp4_dequant_values():
    q = np.array([[0x21] * 8], np.uint8)             # even elements 0.5, odd elements 1.0
    s = np.array([[0x40]], np.uint8)                 # 2.0
    d = oracle.dequant(FMT_NVFP4, q, s, 16, gs=0.25)
    assert (d[0, 0::2] == 0.25).all() and (d[0, 1::2] == 0.5).all()


def test_quant_x_bf16_input_is_exact_fp32():
    rng = np.random.default_rng(8)
    xf = torch.from_numpy(rng.standard_normal((3, 128)).astype(np.float32)).to(torch.bfloat16)
    x16 = xf.view(torch.int16).numpy().astype(np.uint16)
    q1, s1 = oracle.quant_x(FMT_MXFP8, x16)
    q2, s2 = oracle.quant(FMT_MXFP8, xf.float().numpy())
    assert (q1 == q2).all() and (s1 == s2).all()


# ---- MXFP4 (OCP MX: packed E2M1 + E8M0 per 32; scale rule of A3 with E2M1's maximum 6)
def test_mxfp4_block_of_ones():
    q, s = oracle.quant(FMT_MXFP4, np.ones((1, 32), np.float32))
    assert s[0, 0] == 125          # 6 * 2^-3 < 1 <= 6 * 2^-2
    assert (q == 0x66).all()       # 1 * 2^2 = 4 = E2M1 0b0110 in both nibbles


def test_mxfp4_scale_rule_property():
    rng = np.random.default_rng(5)
    for scale in (1e-20, 1e-3, 1.0, 3.0, 1e5, 1e30):
        v = (rng.standard_normal((64, 32)) * scale).astype(np.float32)
        q, s = oracle.quant(FMT_MXFP4, v)
        for r in range(64):
            t = float(np.abs(v[r]).max()) * 2.0 ** -(int(s[r, 0]) - 127)
            assert 3.0 < t <= 6.0, (scale, r, t)


def test_mxfp4_matches_independent():
    rng = np.random.default_rng(8)
    v = (rng.standard_normal((6, 64)) * rng.choice([0.01, 1.0, 20.0], size=(6, 1))).astype(np.float32)
    v[3, 32:] = 0.0
    q, s = oracle.quant(FMT_MXFP4, v)
    for r in range(6):
        for b in range(2):
            blk = v[r, 32 * b:32 * b + 32]
            amax = float(np.abs(blk).max())
            e = -127
            while amax > 0 and e < 127 and amax > 6.0 * 2.0 ** e:   # power-of-two search
                e += 1
            assert s[r, b] == e + 127
            for i in range(32):
                want = _e2m1_brute(float(np.float32(blk[i]) * np.float32(2.0 ** -e)))
                byte = q[r, 16 * b + i // 2]
                got = (byte >> 4) if i & 1 else (byte & 15)
                assert got == want, (r, b, i)


def test_mxfp4_grid_roundtrip():
    # values on the E2M1 grid times a power of two come back exactly
    rng = np.random.default_rng(9)
    grid = np.array(E2M1_GRID[1:] + [-g for g in E2M1_GRID[1:]], np.float64)
    for e in (-20, -3, 0, 5):
        v = rng.choice(grid, size=(4, 32)) * 2.0 ** e
        v[:, 0] = 6.0 * 2.0 ** e                      # the block maximum fixes the scale at e
        q, s = oracle.quant(FMT_MXFP4, v.astype(np.float32))
        assert (s == e + 127).all()
        assert np.array_equal(oracle.dequant(FMT_MXFP4, q, s, 32), v)


def test_mxfp4_dequant_values():
    q = np.array([[0x21] * 16], np.uint8)             # even elements 0.5, odd elements 1.0
    s = np.array([[129]], np.uint8)                   # 2^2
    d = oracle.dequant(FMT_MXFP4, q, s, 32)
    assert (d[0, 0::2] == 2.0).all() and (d[0, 1::2] == 4.0).all()
