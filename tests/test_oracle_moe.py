"""Pins for the oracle's routing, permutation and layer code (CPU only).

Pinned against hand-worked cases with closed-form values, numpy.lexsort and
stable argsort as independent sort routines, pure-Python triple loops, a
PyTorch fp64 SwiGLU written from torch's own silu, and the special cases the
method reduces to (one expert, identical experts, integer tables).
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import apl, moe

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _route_cases():
    for line in open(os.path.join(GOLD, "route_hand.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, lg, k, rn, idx, w = [s.strip() for s in line.split("|")]
        yield (name, np.array([float(v) for v in lg.split()], dtype=np.float32), int(k),
               int(rn), [int(v) for v in idx.split()], [eval(e, {"math": math}) for e in w.split(";")])


@pytest.mark.parametrize("case", list(_route_cases()), ids=lambda c: c[0])
def test_route_hand_cases(case):
    _, lg, k, rn, idx, w = case
    gi, gw = moe.route(lg[None, :], k, rn)
    assert gi[0].tolist() == idx
    assert np.allclose(gw[0], w, rtol=1e-14, atol=0)


def test_route_matches_lexsort_and_softmax():
    rng = np.random.default_rng(5)
    L = rng.standard_normal((40, 12)).astype(np.float32)
    L[3, 4] = L[3, 7]                 # exact ties
    L[9, :] = 0.5
    for k in (1, 3, 12):
        for rn in (0, 1):
            idx, w = moe.route(L, k, rn)
            for t in range(L.shape[0]):
                order = np.lexsort((np.arange(12), -L[t].astype(np.float64)))
                assert idx[t].tolist() == order[:k].tolist()
            p = torch.softmax(torch.from_numpy(L.astype(np.float64)), dim=1).numpy()
            want = np.take_along_axis(p, idx, axis=1)
            if rn:
                want = want / want.sum(axis=1, keepdims=True)
            assert np.allclose(w, want, rtol=1e-13, atol=1e-15)
    _, w = moe.route(L, 12, 0)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=1e-14)
    _, w = moe.route(L, 1, 1)
    assert np.all(w == 1.0)


def test_route_rejects_nan():
    L = np.zeros((2, 4), dtype=np.float32)
    L[1, 2] = np.nan
    with pytest.raises(ValueError):
        moe.route(L, 2, 0)


def test_permute_is_stable_counting_sort():
    rng = np.random.default_rng(6)
    E, T, k = 7, 33, 3
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
    counts, offsets, perm, inv = moe.permute(idx, E)
    flat = idx.reshape(-1)
    want_perm = np.argsort(flat, kind="stable")          # pair id t*k+j in (e, t) order
    assert np.array_equal(perm, want_perm)
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(perm[inv], np.arange(T * k))


def _brute_layer(x, logits, k, renorm, Wgu, Wdn):
    """Triple loops in plain Python floats: no numpy arithmetic on the path."""
    T, H = len(x), len(x[0])
    E = len(Wgu)
    I = len(Wgu[0]) // 2
    out = [[0.0] * H for _ in range(T)]
    for t in range(T):
        z = [float(v) for v in logits[t]]
        order = sorted(range(E), key=lambda e: (-z[e], e))[:k]
        m = max(z)
        s = sum(math.exp(v - m) for v in z)
        ws = [math.exp(z[e] - m) / s for e in order]
        if renorm:
            tot = sum(ws)
            ws = [v / tot for v in ws]
        for e, we in zip(order, ws):
            h = []
            for i in range(I):
                g = sum(Wgu[e][i][c] * float(x[t][c]) for c in range(H))
                u = sum(Wgu[e][I + i][c] * float(x[t][c]) for c in range(H))
                h.append(g / (1.0 + math.exp(-g)) * u)
            for r in range(H):
                out[t][r] += we * sum(Wdn[e][r][i] * h[i] for i in range(I))
    return np.array(out)


def _tiny_blocks(rng, E, H, I, bits):
    blocks = []
    for e in range(E):
        pair = []
        for R, K, q in ((2 * I, H, bits[e][0]), (H, I, bits[e][1])):
            P = rng.integers(0, 256, size=(R, K), dtype=np.uint8)
            par = np.sort(rng.normal(0, 0.02 * 8, size=(R, 256)), axis=1).astype(np.float16)
            pair.append(moe.Block(P, par, q))
        blocks.append(tuple(pair))
    return blocks


@pytest.mark.parametrize("renorm", [0, 1])
def test_layer_brute_force_tiny(renorm):
    rng = np.random.default_rng(7)
    E, H, I, T, k = 4, 32, 32, 3, 2
    bits = [(3, 8), (5, 4), (8, 6), (7, 3)]
    blocks = _tiny_blocks(rng, E, H, I, bits)
    x = rng.standard_normal((T, H)).astype(np.float16)
    L = rng.standard_normal((T, E)).astype(np.float32)
    got = moe.layer(x, L, k, renorm, lambda e: blocks[e])
    Wgu = [b[0].weights().tolist() for b in blocks]
    Wdn = [b[1].weights().tolist() for b in blocks]
    want = _brute_layer(x.astype(np.float64).tolist(), L, k, renorm, Wgu, Wdn)
    assert np.allclose(got["out"], want, rtol=1e-12, atol=1e-14)
    # sampled output columns agree with the full computation
    cols = [0, 5, 31]
    part = moe.layer(x, L, k, renorm, lambda e: blocks[e], out_rows=cols)
    assert np.allclose(part["out"], got["out"][:, cols], rtol=1e-14, atol=0)
    # and sampled tokens
    part = moe.layer(x, L, k, renorm, lambda e: blocks[e], out_rows=cols, out_tokens=[2, 0])
    assert np.allclose(part["out"], got["out"][[2, 0]][:, cols], rtol=1e-14, atol=0)


def test_layer_hand_case():
    H = I = 32
    par = np.tile(((np.arange(256) - 128) / 32.0).astype(np.float16), (2 * I, 1))
    P_gu = np.full((2 * I, H), 128, dtype=np.uint8)
    P_gu[0, 0] = 192
    P_gu[I, 0] = 160
    P_dn = np.full((H, I), 128, dtype=np.uint8)
    P_dn[:, 0] = 128 + np.arange(H)
    zero_gu = np.full((2 * I, H), 128, dtype=np.uint8)
    zero_dn = np.full((H, I), 128, dtype=np.uint8)
    blocks = [(moe.Block(P_gu, par, 8), moe.Block(P_dn, par[:H], 8)),
              (moe.Block(zero_gu, par, 8), moe.Block(zero_dn, par[:H], 8))]
    x = np.zeros((1, H), dtype=np.float16)
    x[0, 0] = 1
    L = np.array([[0.5, -0.5]], dtype=np.float32)
    got = moe.layer(x, L, 1, 1, lambda e: blocks[e])["out"][0]
    expr = [l.split("|")[1].strip() for l in open(os.path.join(GOLD, "layer_hand.txt"))
            if l.startswith("expr")][0]
    want = np.array([eval(expr, {"math": math, "r": r}) for r in range(H)])
    assert np.allclose(got, want, rtol=1e-14, atol=1e-15)


def test_single_expert_is_dense_swiglu_in_torch():
    rng = np.random.default_rng(8)
    H, I, T = 64, 96, 5
    (gu, dn), = _tiny_blocks(rng, 1, H, I, [(6, 7)])
    x = rng.standard_normal((T, H)).astype(np.float16)
    L = rng.standard_normal((T, 1)).astype(np.float32)
    got = moe.layer(x, L, 1, 1, lambda e: (gu, dn))["out"]
    X = torch.from_numpy(x.astype(np.float64))
    Wg = torch.from_numpy(gu.weights()[:I])
    Wu = torch.from_numpy(gu.weights()[I:])
    Wd = torch.from_numpy(dn.weights())
    want = torch.nn.functional.linear(
        torch.nn.functional.silu(torch.nn.functional.linear(X, Wg)) * torch.nn.functional.linear(X, Wu), Wd)
    assert np.allclose(got, want.numpy(), rtol=1e-12, atol=1e-14)


def test_identical_experts_make_routing_irrelevant():
    rng = np.random.default_rng(9)
    H, I, T, E = 32, 64, 6, 5
    (gu, dn), = _tiny_blocks(rng, 1, H, I, [(4, 5)])
    x = rng.standard_normal((T, H)).astype(np.float16)
    L1 = rng.standard_normal((T, E)).astype(np.float32)
    L2 = rng.standard_normal((T, E)).astype(np.float32)
    a = moe.layer(x, L1, 3, 1, lambda e: (gu, dn))["out"]
    b = moe.layer(x, L2, 2, 1, lambda e: (gu, dn))["out"]
    c = moe.layer(x, L1[:, :1], 1, 1, lambda e: (gu, dn))["out"]
    assert np.allclose(a, b, rtol=1e-12, atol=1e-14)
    assert np.allclose(a, c, rtol=1e-12, atol=1e-14)


def test_integer_tables_give_integer_outputs():
    # LUT_b[v] = v - 2^(b-1) (integers), x small integers: every sum is an integer.
    rng = np.random.default_rng(10)
    H, I = 32, 32
    blocks = []
    for e in range(2):
        pair = []
        for R, K in ((2 * I, H), (H, I)):
            P = rng.integers(0, 256, size=(R, K), dtype=np.uint8)
            par = np.tile((np.arange(256) - 128).astype(np.float16), (R, 1))
            pair.append(moe.Block(P, par, 8))
        blocks.append(tuple(pair))
    x = rng.integers(-2, 3, size=(3, H)).astype(np.float16)
    L = rng.standard_normal((3, 2)).astype(np.float32)
    res = moe.layer(x, L, 2, 1, lambda e: blocks[e])
    for e in range(2):
        pairs = res["perm"][res["offsets"][e]:res["offsets"][e + 1]]
        X = x.astype(np.float64)[pairs // 2]
        Wgu = blocks[e][0].weights()
        G, U = X @ Wgu[:I].T, X @ Wgu[I:].T
        assert np.array_equal(G, np.round(G)) and np.array_equal(U, np.round(U))


def test_residual_added_once():
    rng = np.random.default_rng(11)
    E, H, I, T = 3, 32, 32, 4
    blocks = _tiny_blocks(rng, E, H, I, [(8, 8)] * E)
    x = rng.standard_normal((T, H)).astype(np.float16)
    L = rng.standard_normal((T, E)).astype(np.float32)
    a = moe.layer(x, L, 2, 0, lambda e: blocks[e])["out"]
    b = moe.layer(x, L, 2, 0, lambda e: blocks[e], residual=x)["out"]
    assert np.allclose(b - a, x.astype(np.float64), rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- routing statistics

def _stats_gold():
    d = {}
    for line in open(os.path.join(GOLD, "stats_hand.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, vals = (x.strip() for x in line.split("|"))
        d[key] = np.array([float(v) for v in vals.split()])
    return d


def test_routing_mass_hand_case():
    g = _stats_gold()
    L = np.stack([g["logits_t0"], g["logits_t1"]]).astype(np.float32)
    idx, w = moe.route(L, 2, 1)
    assert np.array_equal(moe.routing_mass(idx, w, 4), g["M"])
    m1 = moe.stats_update(np.full(4, 0.25), idx, w, 4, 0.25)
    assert np.array_equal(m1, g["m1"])
    assert np.array_equal(moe.stats_update(m1, idx, w, 4, 0.25), g["m2"])


def test_routing_mass_sums_to_one_with_renorm_and_to_the_kept_mass_without():
    rng = np.random.default_rng(5)
    L = rng.standard_normal((37, 9)).astype(np.float32)
    idx, w = moe.route(L, 3, 1)
    assert abs(moe.routing_mass(idx, w, 9).sum() - 1.0) < 1e-12
    idx0, w0 = moe.route(L, 3, 0)
    # the mass kept by the top 3 of a softmax, averaged over tokens (scipy's softmax)
    from scipy.special import softmax
    p = np.sort(softmax(L.astype(np.float64), axis=1), axis=1)[:, ::-1]
    assert abs(moe.routing_mass(idx0, w0, 9).sum() - p[:, :3].sum(axis=1).mean()) < 1e-12


def test_routing_mass_with_all_experts_is_the_mean_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(6)
    L = rng.standard_normal((11, 6)).astype(np.float32)
    idx, w = moe.route(L, 6, 0)
    want = softmax(L.astype(np.float64), axis=1).mean(axis=0)
    assert np.allclose(moe.routing_mass(idx, w, 6), want, rtol=0, atol=1e-14)


def test_repeated_batch_follows_the_geometric_closed_form():
    rng = np.random.default_rng(7)
    L = rng.standard_normal((8, 5)).astype(np.float32)
    idx, w = moe.route(L, 2, 1)
    M = moe.routing_mass(idx, w, 5)
    m0 = rng.random(5)
    a, m = 0.1, m0.copy()
    for n in range(1, 30):
        m = moe.stats_update(m, idx, w, 5, a)
        closed = (1 - a) ** n * m0 + (1 - (1 - a) ** n) * M
        assert np.allclose(m, closed, rtol=0, atol=1e-14)
