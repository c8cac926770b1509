"""Pins for the oracle's APL format code (CPU only).

Each test ties oracle.apl to something other than itself: hand-derived plane
words, the nesting invariant checked by plain integer shifts, bit counts
taken with numpy.unpackbits, closed forms of the child tables, and a
pure-Python brute force of dequantisation.
"""
import os

import numpy as np
import pytest

from oracle import apl

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _hand_rows():
    k = np.arange(32)
    return np.stack([k, 255 - k, np.where(k % 2 == 0, 128, 1)]).astype(np.uint8)


def test_pack_matches_hand_derived_words():
    want = {}
    for line in open(os.path.join(GOLD, "apl_pack_hand.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f = line.split()
        want[int(f[0])] = [int(h, 16) for h in f[1:]]
    planes = apl.pack(_hand_rows(), 8)
    assert planes.shape == (8, 3, 1)
    for r, words in want.items():
        assert [int(planes[p, r, 0]) for p in range(8)] == words, r


def test_pack_rejects_ragged_k():
    with pytest.raises(ValueError):
        apl.pack(np.zeros((2, 48), dtype=np.uint8), 8)


@pytest.mark.parametrize("n", [8, 6, 3])
def test_nesting_invariant_all_values(n):
    # Every parent value in every position; top-b planes give P >> (n - b).
    vals = np.arange(1 << n)
    P = np.stack([np.roll(np.resize(vals, 256), s) for s in range(5)]).astype(np.uint8)
    planes = apl.pack(P, n)
    for b in range(1, n + 1):
        got = apl.unpack(planes, b, n)
        assert np.array_equal(got, P.astype(np.int64) >> (n - b)), b


def test_round_trip_random():
    rng = np.random.default_rng(1)
    P = rng.integers(0, 256, size=(7, 96), dtype=np.uint8)
    assert np.array_equal(apl.unpack(apl.pack(P, 8), 8, 8), P.astype(np.int64))


def test_plane_popcount_equals_bit_count():
    rng = np.random.default_rng(2)
    P = rng.integers(0, 256, size=(5, 128), dtype=np.uint8)
    planes = apl.pack(P, 8)
    bits = np.unpackbits(P[..., None], axis=-1)       # [R][K][8], MSB first
    for p in range(8):
        pc = sum(bin(int(w)).count("1") for w in planes[p].ravel())
        assert pc == int(bits[..., p].sum())


def test_child_lut_linear_parent_closed_form():
    # Parent LUT[v] = v (exact in fp16): the mean of the 2^(8-b) entries with top
    # bits j is j*2^(8-b) + (2^(8-b) - 1)/2, exact in fp16 for these sizes.
    par = np.tile(np.arange(256, dtype=np.float16), (2, 1))
    for b in range(1, 9):
        g = 1 << (8 - b)
        want = np.arange(1 << b) * g + (g - 1) / 2.0
        got = apl.child_lut(par, b, 8)
        assert got.dtype == np.float16
        assert np.array_equal(got.astype(np.float64), np.tile(want, (2, 1))), b


def test_child_lut_is_pairwise_mean_and_sorted():
    rng = np.random.default_rng(3)
    par = np.sort(rng.normal(0, 0.02, size=(4, 256)), axis=1).astype(np.float16)
    p64 = par.astype(np.float64)
    for b in range(3, 8):
        g = 1 << (8 - b)
        # independent fp64 computation: reshape-and-mean
        exact = p64.reshape(4, 1 << b, g).mean(axis=2)
        got = apl.child_lut(par, b, 8).astype(np.float64)
        # within half an fp16 ulp of the exact mean (RNE), and monotone
        ulp = np.spacing(np.abs(exact).astype(np.float16)).astype(np.float64)
        assert np.all(np.abs(got - exact) <= ulp / 2 + 1e-12)
        assert np.all(np.diff(got, axis=1) >= 0)
    assert np.array_equal(apl.child_lut(par, 8, 8), par)


def test_dequant_brute_force():
    rng = np.random.default_rng(4)
    P = rng.integers(0, 256, size=(3, 32), dtype=np.uint8)
    par = rng.normal(0, 0.02, size=(3, 256)).astype(np.float16)
    for b in (3, 5, 8):
        lut = apl.child_lut(par, b, 8)
        W = apl.dequant(P, lut, b, 8)
        for r in range(3):
            for k in range(32):
                v = int(P[r, k]) // (2 ** (8 - b))
                assert W[r, k] == float(lut[r, v])


def test_tile_planes_places_every_bit_at_its_closed_form_index():
    """The page order of the planes: element k of row r of plane p (bit k%32 of
    word w = k//32) sits in page word p*R*W + ((r/32)*(W/2) + w/2)*64 + (r%32)*2
    + w%2, at bit 8*(j//8) + (j%8)//2 + 4*(j%2) with j = k%32 (even elements of
    a byte in its low half, odd ones in its high half), checked bit by bit
    against an explicit loop over that formula."""
    n, R, W = 3, 64, 6
    planes = ((np.arange(n * R * W, dtype=np.uint64) * 2654435761) % (1 << 32)).astype(np.uint32)
    planes = planes.reshape(n, R, W)
    got = apl.tile_planes(planes)
    want = np.zeros(n * R * W, dtype=np.uint32)
    for p in range(n):
        for r in range(R):
            for w in range(W):
                idx = p * R * W + ((r // 32) * (W // 2) + w // 2) * 64 + (r % 32) * 2 + w % 2
                for j in range(32):
                    bit = (int(planes[p, r, w]) >> j) & 1
                    want[idx] |= np.uint32(bit << (8 * (j // 8) + (j % 8) // 2 + 4 * (j % 2)))
    assert np.array_equal(got, want)
    # the same number of set bits in every word: bits are moved, never made
    pc = lambda a: np.array([bin(int(v)).count("1") for v in a.reshape(-1)])
    assert sorted(pc(got).tolist()) == sorted(pc(planes).tolist())
    # a warp reading word pair u of 32 consecutive rows reads 64 contiguous words
    u, g = 1, 1
    block = got[(g * (W // 2) + u) * 64:(g * (W // 2) + u + 1) * 64].reshape(32, 2)
    src = planes[0, 32 * g:32 * g + 32, 2 * u:2 * u + 2]
    # element 0 (bit 0) stays at bit 0 and element 1 moves to bit 4
    assert np.array_equal(block & 1, src & 1)
    assert np.array_equal((block >> 4) & 1, (src >> 1) & 1)


def test_bit_position_is_a_permutation_keeping_even_elements_low():
    pos = [apl.bit_position(e) for e in range(32)]
    assert sorted(pos) == list(range(32))
    for e in range(32):
        assert pos[e] // 8 == e // 8                   # stays in its byte
        assert (pos[e] % 8 < 4) == (e % 2 == 0)         # even elements in the low half
    assert pos[:8] == [0, 4, 1, 5, 2, 6, 3, 7]
