"""APL bit-plane format, restated plainly (oracle; test infrastructure only).

Source: PagedWeight technical summary, Core components section 1 "Paged
Weight Representation": weights are held in APL's layered bit-plane format
with associated lookup tables, one unit per (layer, expert, gate_up|down)
linear block.  The pages print no bit order or packing; this build fixes:

* a parent index P[r][k] in [0, 2^n) per weight (n = 8 in every workload);
* plane p (p = 0 is the most significant) holds bit (n - 1 - p) of P;
* planes are stored plane-major per block, ``planes[p][r][w]`` uint32,
  with bit j of word w holding element k = 32 w + j (least significant bit
  = lowest k);
* a b-bit weight uses the top b planes: its index is P >> (n - b);
* each row and bitwidth b has its own 2^b-entry fp16 table LUT_b[r].

Child tables (reading of "associated lookup tables"): LUT_n is the parent
table, and for b < n, LUT_b[r][j] is the mean of the 2^(n-b) parent entries
whose index has top b bits equal to j, computed in fp64 and rounded once to
fp16 (round to nearest even).
"""
import numpy as np


def plane_of_bit(p: int, n: int) -> int:
    """Bit position of P that plane p holds (plane 0 = most significant)."""
    return n - 1 - p


def pack(P: np.ndarray, n: int) -> np.ndarray:
    """Parent indices [R][K] -> planes uint32 [n][R][K/32].

    Element by element: plane p, row r, word w, bit j is bit (n-1-p) of
    P[r][32w + j].  K must be a multiple of 32.
    """
    P = np.asarray(P).astype(np.int64)
    R, K = P.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    if P.min() < 0 or P.max() >= (1 << n):
        raise ValueError("index out of range")
    out = np.zeros((n, R, K // 32), dtype=np.uint64)
    for p in range(n):
        bits = (P >> plane_of_bit(p, n)) & 1                  # [R][K]
        bits = bits.reshape(R, K // 32, 32).astype(np.uint64)
        weights = np.uint64(1) << np.arange(32, dtype=np.uint64)   # bit j <-> k = 32w + j
        out[p] = (bits * weights[None, None, :]).sum(axis=2)
    return out.astype(np.uint32)


def unpack(planes: np.ndarray, b: int, n: int) -> np.ndarray:
    """Top b planes [n or more][R][K/32] -> b-bit indices int64 [R][K].

    index = sum over p < b of bit_p << (b - 1 - p); equals P >> (n - b).
    """
    planes = np.asarray(planes, dtype=np.uint64)
    _, R, W = planes.shape
    idx = np.zeros((R, W * 32), dtype=np.int64)
    j = np.arange(32, dtype=np.uint64)
    for p in range(b):
        bits = ((planes[p][:, :, None] >> j[None, None, :]) & np.uint64(1)).astype(np.int64)
        idx |= bits.reshape(R, W * 32) << (b - 1 - p)
    return idx


def bit_position(e: int) -> int:
    """Where element e (0..31) of a plane word sits inside the device page's word:
    within each byte (8 elements), the even elements take bits 0..3 and the odd
    ones bits 4..7, in element order: 8*(e//8) + (e%8)//2 + 4*(e%2)."""
    return 8 * (e // 8) + (e % 8) // 2 + 4 * (e % 2)


def tile_planes(planes: np.ndarray) -> np.ndarray:
    """Planes [n][R][W] -> the device page order, flat uint32.

    Each plane is cut into groups of 32 rows and pairs of words along K; a
    page lists, for each group (in row order) and each word pair (in K order),
    the 32 rows' two words side by side: [n][R/32][W/2][32][2].  Inside every
    word the bits are re-placed by ``bit_position`` (even elements of each
    byte in its low half, odd elements in its high half).  R must be a
    multiple of 32 and W even.
    """
    planes = np.asarray(planes, dtype=np.uint32)
    n, R, W = planes.shape
    if R % 32 or W % 2:
        raise ValueError("R must be a multiple of 32 and W even")
    words = planes.reshape(n, R // 32, 32, W // 2, 2).transpose(0, 1, 3, 2, 4).reshape(-1)
    out = np.zeros_like(words)
    for e in range(32):
        out |= ((words >> np.uint32(e)) & np.uint32(1)) << np.uint32(bit_position(e))
    return out


def child_lut(parent_lut: np.ndarray, b: int, n: int) -> np.ndarray:
    """LUT_b [R][2^b] fp16 from the parent table [R][2^n] fp16 (see module doc)."""
    par = np.asarray(parent_lut, dtype=np.float16).astype(np.float64)
    R, V = par.shape
    if V != (1 << n):
        raise ValueError("parent table must have 2^n entries")
    group = 1 << (n - b)
    child = np.empty((R, 1 << b), dtype=np.float64)
    for j in range(1 << b):
        child[:, j] = par[:, j * group:(j + 1) * group].sum(axis=1) / group
    return child.astype(np.float16)


def child_luts(parent_lut: np.ndarray, b_min: int, n: int) -> dict:
    """{b: LUT_b} for b in [b_min, n]."""
    return {b: child_lut(parent_lut, b, n) for b in range(b_min, n + 1)}


def dequant(P: np.ndarray, lut_b: np.ndarray, b: int, n: int) -> np.ndarray:
    """W_b[r][k] = LUT_b[r][P[r][k] >> (n - b)] in fp64, shape [R][K]."""
    idx = np.asarray(P).astype(np.int64) >> (n - b)
    lut = np.asarray(lut_b, dtype=np.float16).astype(np.float64)
    return np.take_along_axis(lut, idx, axis=1)
