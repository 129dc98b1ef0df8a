"""Pins of the oracle's number formats against the format definitions and library casts.

The oracle's encoders and decoders are checked against (1) hand-derived code points of
the OCP MX formats (tests/golden/format_points.txt), (2) PyTorch's float8_e4m3fn and
bfloat16 casts (a separate, library implementation of round-to-nearest-even), and
(3) a brute-force nearest-even search over every grid point.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "format_points.txt")
E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _gold():
    rows = []
    for line in open(GOLD):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        rows.append(line.split())
    return rows


def _same(a, b):
    if math.isnan(b):
        return math.isnan(a)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


@pytest.mark.parametrize("row", _gold(), ids=lambda r: "-".join(r))
def test_golden_points(row):
    kind, a, b = row
    if kind == "e4m3":
        assert _same(oracle.e4m3_decode(int(a, 16)), float(b))
    elif kind == "e2m1":
        assert _same(oracle.e2m1_decode(int(a, 16)), float(b))
    elif kind == "e8m0":
        assert _same(oracle.e8m0_decode(int(a, 16)), float(b))
    elif kind == "e4m3_enc":
        assert oracle.e4m3_encode(float(a)) == int(b, 16)
    elif kind == "e2m1_enc":
        assert oracle.e2m1_encode(float(a)) == int(b, 16)
    else:
        raise AssertionError(kind)


def test_e4m3_decode_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        assert _same(oracle.e4m3_decode(c), float(ref[c])), c


def test_e4m3_encode_roundtrips_every_finite_code():
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if math.isnan(v):
            assert oracle.e4m3_encode(float("nan")) == 0x7F
            continue
        assert oracle.e4m3_encode(v) == c, hex(c)


def test_e4m3_encode_matches_torch_rne_random():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 200.0)])
    v = np.clip(v, -448, 448).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(x)) for x in v], np.uint8)
    assert (got == ref).all()


def test_e4m3_encode_midpoints_round_to_even():
    vals = sorted({oracle.e4m3_decode(c) for c in range(0, 0x7F)})
    for lo, hi in zip(vals[:-1], vals[1:]):
        mid = (lo + hi) / 2
        clo, chi = oracle.e4m3_encode(lo), oracle.e4m3_encode(hi)
        want = clo if clo % 2 == 0 else chi
        assert oracle.e4m3_encode(np.float32(mid)) == want
        assert oracle.e4m3_encode(-np.float32(mid)) == want | 0x80


def _e2m1_brute(x):
    """Nearest grid point, ties to the even code, saturating at 6."""
    a = min(abs(x), 6.0)
    best = None
    for code, g in enumerate(E2M1_GRID):
        d = abs(a - g)
        if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
            best = (d, code)
    return best[1] | (8 if math.copysign(1.0, x) < 0 else 0)


def test_e2m1_decode_table():
    for c in range(16):
        want = E2M1_GRID[c & 7] * (-1 if c & 8 else 1)
        assert oracle.e2m1_decode(c) == want


def test_e2m1_encode_brute_force():
    rng = np.random.default_rng(2)
    v = np.concatenate([rng.standard_normal(20000) * 3, np.arange(-700, 701) / 100.0]).astype(np.float32)
    for x in v:
        assert oracle.e2m1_encode(float(x)) == _e2m1_brute(float(x)), x


def test_e8m0_decode_all():
    for b in range(255):
        assert oracle.e8m0_decode(b) == math.ldexp(1.0, b - 127)
    assert math.isnan(oracle.e8m0_decode(255))


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(50000) * s for s in (1e-30, 1e-3, 1.0, 1e4, 1e30)]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.double_to_bf16(float(x)) for x in v], np.uint16)
    assert (got == ref).all()
