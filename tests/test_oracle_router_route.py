"""Pins of the oracle's router (a1, a2) and route (a4) steps.

Router: exact logits on shapes where the double sum of bf16 products is exact
(compared with math.fsum), sigmoid special values, brute-force top-k by a full sort,
the tie rule, weight invariants and the bias-selects-only reading.
Route: a hand-worked example, multi-tile hot experts, and invariants checked on
random routings.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import FMT_MXFP8


def _layer(E=16, k=2, H=64, has_bias=False, rsf=1.0, renorm=True, shared=True):
    cfg = dict(H=H, E=E, k=k, I=32, I_sh=32, w_fmt=FMT_MXFP8, sh_fmt=FMT_MXFP8, has_shared=shared,
               has_bias=has_bias, renormalize=renorm, rsf=rsf, eps=1e-6)
    return oracle.make_layer(cfg)


def _bf16(a):
    t = torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().astype(np.uint16), t.double().numpy()


def test_logits_exact_sum():
    rng = np.random.default_rng(10)
    L = _layer(E=8, H=64)
    x16, xd = _bf16(rng.standard_normal((3, 64)))
    w16, wd = _bf16(rng.standard_normal((8, 64)) * 0.02)
    logits, scores, idx, w, margin = oracle.router(L, x16, w16)
    for m in range(3):
        for e in range(8):
            exact = math.fsum(float(a) * float(b) for a, b in zip(xd[m], wd[e]))
            assert logits[m, e] == np.float32(exact)


def test_sigmoid_special_values():
    L = _layer(E=4, k=2)
    li = np.array([[0.0, 30.0, -30.0, 1.0]], np.float32)
    x16 = np.zeros((1, 64), np.uint16)
    _, scores, idx, _, _ = oracle.router(L, x16, np.zeros((4, 64), np.uint16), logits_in=li)
    assert scores[0, 0] == 0.5
    assert scores[0, 1] == 1.0                       # fp32 rounding of 1 - 9e-14
    assert 0 < scores[0, 2] < 1e-12
    assert scores[0, 3] == np.float32(1.0 / (1.0 + math.exp(-1.0)))
    assert list(idx[0]) == [1, 3]


def _brute_topk(scores, bias, k):
    key = scores if bias is None else (scores + bias).astype(np.float32)
    out = []
    for m in range(scores.shape[0]):
        order = sorted(range(scores.shape[1]), key=lambda e: (-float(key[m, e]), e))
        out.append(order[:k])
    return np.array(out, np.int32)


@pytest.mark.parametrize("has_bias", [False, True])
def test_topk_brute_force(has_bias):
    rng = np.random.default_rng(11)
    E, k = 16, 4
    L = _layer(E=E, k=k, has_bias=has_bias, rsf=2.5)
    x16, _ = _bf16(rng.standard_normal((20, 64)))
    w16, _ = _bf16(rng.standard_normal((E, 64)) * 0.3)
    bias = (rng.standard_normal(E) * 0.05).astype(np.float32) if has_bias else None
    logits, scores, idx, w, margin = oracle.router(L, x16, w16, bias=bias)
    assert (idx == _brute_topk(scores, bias, k)).all()
    # weights: renormalised raw scores (the bias selects only), summing to rsf
    for m in range(20):
        s = scores[m, idx[m]].astype(np.float64)
        assert np.allclose(w[m], s / s.sum() * 2.5, rtol=0, atol=1e-15)
        assert abs(w[m].sum() - 2.5) < 1e-12
        assert len(set(idx[m])) == k
        key = scores[m] + (bias if has_bias else 0)
        assert all(key[idx[m][j]] >= key[idx[m][j + 1]] for j in range(k - 1))


def test_topk_ties_lower_index_wins():
    L = _layer(E=6, k=3)
    li = np.array([[1.0, 2.0, 2.0, 0.5, 2.0, 2.0]], np.float32)
    _, _, idx, _, margin = oracle.router(L, np.zeros((1, 64), np.uint16), np.zeros((6, 64), np.uint16),
                                         logits_in=li)
    assert list(idx[0]) == [1, 2, 4]
    assert margin[0] == 0.0


def test_no_renormalize():
    L = _layer(E=8, k=2, renorm=False, rsf=1.5)
    li = np.array([[0.0, 1.0, -1.0, 2.0, 0.0, 0.0, 0.0, 0.0]], np.float32)
    _, scores, idx, w, _ = oracle.router(L, np.zeros((1, 64), np.uint16), np.zeros((8, 64), np.uint16),
                                         logits_in=li)
    assert list(idx[0]) == [3, 1]
    assert np.allclose(w[0], scores[0, [3, 1]].astype(np.float64) * 1.5, rtol=0, atol=1e-15)


def test_route_hand_example():
    L = _layer(E=4, k=2)
    topk = np.array([[1, 0], [1, 2], [3, 1]], np.int32)
    counts, offsets, perm, inv, tiles = oracle.route(L, topk)
    assert list(counts) == [1, 3, 1, 1, 3]
    assert list(offsets) == [0, 1, 4, 5, 6, 9]
    # pair id = m*k + j: expert 0 <- (0,1)=1; expert 1 <- (0,0)=0,(1,0)=2,(2,1)=5; 2 <- 3; 3 <- 4; shared 6,7,8
    assert list(perm) == [1, 0, 2, 5, 3, 4, 6, 7, 8]
    assert list(inv) == [1, 0, 2, 4, 5, 3, 6, 7, 8]
    assert tiles.tolist() == [[0, 0, 1], [1, 1, 3], [2, 4, 1], [3, 5, 1], [4, 6, 3]]


def test_route_multi_tile_hot_expert():
    L = _layer(E=4, k=1, shared=False)
    topk = np.zeros((20, 1), np.int32)
    topk[19, 0] = 3
    counts, offsets, perm, inv, tiles = oracle.route(L, topk)
    assert list(counts) == [19, 0, 0, 1, 0]
    assert tiles.tolist() == [[0, 0, 8], [0, 8, 8], [0, 16, 3], [3, 19, 1]]


@pytest.mark.parametrize("seed", range(5))
def test_route_invariants(seed):
    rng = np.random.default_rng(seed)
    E, k, M = 32, 4, int(rng.integers(1, 65))
    L = _layer(E=E, k=k)
    hot = rng.random(E) ** 4
    topk = np.array([rng.choice(E, size=k, replace=False, p=hot / hot.sum()) for _ in range(M)], np.int32)
    counts, offsets, perm, inv, tiles = oracle.route(L, topk)
    P = M * k + M
    assert sorted(perm.tolist()) == list(range(P))
    assert (perm[inv] == np.arange(P)).all() and (inv[perm] == np.arange(P)).all()
    assert tiles[:, 2].sum() == P
    assert ((tiles[:, 2] >= 1) & (tiles[:, 2] <= 8)).all()
    for e in range(E + 1):
        assert (tiles[:, 0] == e).sum() == -(-counts[e] // 8)
    # brute force: pairs sorted by (expert, pair id)
    ex = [int(topk.flat[p]) if p < M * k else E for p in range(P)]
    assert perm.tolist() == sorted(range(P), key=lambda p: (ex[p], p))
    for t in tiles:
        assert all(ex[perm[t[1] + r]] == t[0] for r in range(t[2]))
