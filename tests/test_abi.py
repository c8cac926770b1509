"""The C-ABI library on the CPU: it loads, exports every function the header
declares, and its host-side packer matches the oracle bit for bit."""
import os
import re

import numpy as np
import pytest

import any_precision_weight_gb300 as pw
from oracle import apl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "pw.h")).read()
    return sorted(set(re.findall(r"^(?:int|size_t|const char\*)\s+(pw_\w+)\s*\(", src, re.M)))


def test_header_and_binding_agree():
    assert _declared() == pw.exported_symbols()


def test_library_exports_every_declared_symbol():
    L = pw.lib()
    for name in _declared():
        assert hasattr(L, name), name


def test_lut_sizes_closed_form():
    # b = 3..8: 8 + 16 + 32 + 64 + 128 + 256 = 504 fp16 entries per row
    assert pw.pw_lut_bytes(2, 3, 8) == 2 * 504 * 2
    assert pw.pw_lut_offset(2, 3, 3) == 0
    assert pw.pw_lut_offset(2, 3, 5) == 2 * (8 + 16) * 2
    assert pw.pw_plane_bytes(64, 256) == 64 * 256 // 8


@pytest.mark.parametrize("R,K,n", [(3, 32, 8), (17, 96, 8), (64, 256, 8), (5, 64, 6), (4, 32, 3)])
def test_pack_matches_oracle_bit_exact(R, K, n):
    rng = np.random.default_rng(R * 1000 + K + n)
    P = rng.integers(0, 1 << n, size=(R, K), dtype=np.uint8)
    par = np.sort(rng.normal(0, 0.02, size=(R, 1 << n)), axis=1).astype(np.float16)
    b_min = min(3, n)
    planes, luts = pw.pw_pack(P, par, n, b_min)
    assert np.array_equal(planes, apl.pack(P, n))
    for b in range(b_min, n + 1):
        off = pw.pw_lut_offset(R, b_min, b) // 2
        got = luts[off:off + R * (1 << b)].reshape(R, 1 << b)
        assert np.array_equal(got, apl.child_lut(par, b, n).view(np.uint16)), b


def test_pack_large_rows_threaded():
    # above the size where the packer splits rows across CPU threads
    rng = np.random.default_rng(12)
    P = rng.integers(0, 256, size=(1100, 1024), dtype=np.uint8)
    par = np.sort(rng.normal(0, 0.02, size=(1100, 256)), axis=1).astype(np.float16)
    planes, luts = pw.pw_pack(P, par, 8, 3)
    assert np.array_equal(planes, apl.pack(P, 8))
    off = pw.pw_lut_offset(1100, 3, 5) // 2
    assert np.array_equal(luts[off:off + 1100 * 32].reshape(1100, 32),
                          apl.child_lut(par, 5, 8).view(np.uint16))


def test_pack_child_table_rounding_edges():
    # pairs whose fp64 mean falls exactly between two fp16 values (ties to even),
    # subnormals, signed zeros, mixed signs, the largest finite values
    pairs = [(0x3C00, 0x3C01), (0x3C01, 0x3C02), (0x0001, 0x0002), (0x0002, 0x0003),
             (0x8000, 0x0000), (0xBC00, 0x3C00), (0x7BFF, 0x7BFE), (0x03FF, 0x0400),
             (0x8001, 0x8002), (0x5640, 0x5641)]
    par = np.zeros((1, 256), dtype=np.uint16)
    for i, (a, b) in enumerate(pairs):
        par[0, 2 * i], par[0, 2 * i + 1] = a, b
    par = par.view(np.float16)
    P = np.zeros((1, 32), dtype=np.uint8)
    _, luts = pw.pw_pack(P, par, 8, 7)
    assert np.array_equal(luts[:128], apl.child_lut(par, 7, 8).view(np.uint16)[0])


def test_pack_rejects_bad_input():
    par = np.zeros((2, 256), dtype=np.float16)
    with pytest.raises(pw.PWError) as e:
        pw.pw_pack(np.zeros((2, 48), dtype=np.uint8), par, 8, 3)
    assert e.value.code == pw.PW_EINVAL
    with pytest.raises(pw.PWError) as e:
        pw.pw_pack(np.full((2, 32), 200, dtype=np.uint8), np.zeros((2, 64), np.float16), 6, 3)
    assert e.value.code == pw.PW_EINVAL


def test_workspace_bytes_cover_sections():
    nb = pw.lib().pw_workspace_bytes(4, 60, 4, 2048, 1408)
    assert nb >= 16 * 1408 * 2 + 16 * 2048 * 4      # h (fp16) and y (fp32) of every pair
    assert pw.lib().pw_workspace_bytes(-1, 60, 4, 2048, 1408) == 0


@pytest.mark.parametrize("R,K,n", [(32, 64, 1), (64, 256, 8), (256, 1408, 6)])
def test_tile_planes_matches_oracle_bit_exact(R, K, n):
    rng = np.random.default_rng(R + K + n)
    planes = rng.integers(0, 1 << 32, size=(n, R, K // 32), dtype=np.uint64).astype(np.uint32)
    assert np.array_equal(pw.pw_tile_planes(planes), apl.tile_planes(planes))


def test_tile_planes_rejects_bad_shapes():
    with pytest.raises(pw.PWError):
        pw.pw_tile_planes(np.zeros((1, 48, 2), dtype=np.uint32))      # R % 32
    with pytest.raises(pw.PWError):
        pw.pw_tile_planes(np.zeros((1, 32, 3), dtype=np.uint32))      # K % 64


def test_tile_planes_threaded_path_matches_oracle():
    """A block large enough for the multi-threaded reordering (2^20 words and more)."""
    rng = np.random.default_rng(5)
    planes = rng.integers(0, 1 << 32, size=(8, 1024, 2048 // 32), dtype=np.uint64).astype(np.uint32)
    assert np.array_equal(pw.pw_tile_planes(planes), apl.tile_planes(planes))
