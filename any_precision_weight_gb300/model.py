"""Loading quantised MoE blocks into a PagedMoE page table.

Marshalling only: the packing is pw_pack (C++), the registration is
pw_block_register; this module moves arrays into pinned host memory and
hands the pointers over.
"""
from __future__ import annotations

import numpy as np

from . import KIND_DOWN, KIND_GATE_UP, PagedMoE, pw_lut_bytes, pw_pack, pw_tile_planes


class HostStore:
    """Pinned host backing store carved out of a few large pinned chunks.

    One pinned allocation per block rounds every block up to a power of two
    (about 1.5x the bytes for these shapes) and leaves thousands of small
    pinned regions; chunks of ``chunk_bytes`` hold many blocks each, every
    slice starting on a 256-byte boundary.
    """

    def __init__(self, chunk_bytes: int = 1 << 30):
        self.chunk_bytes = chunk_bytes
        self._chunks = []
        self._cur = None
        self._off = 0

    def alloc(self, nbytes: int):
        """A pinned uint8 CPU tensor of nbytes (a view into a chunk)."""
        import torch
        n = (nbytes + 255) // 256 * 256
        if self._cur is None or self._off + n > self._cur.numel():
            self._cur = torch.empty(max(self.chunk_bytes, n), dtype=torch.uint8, pin_memory=True)
            self._chunks.append(self._cur)
            self._off = 0
        t = self._cur[self._off:self._off + nbytes]
        self._off += n
        return t

    def nbytes(self) -> int:
        return sum(c.numel() for c in self._chunks)


def pack_pinned(P: np.ndarray, parent_lut: np.ndarray, n_bits: int = 8, b_min: int = 3,
                store: HostStore | None = None):
    """pw_pack into pinned torch CPU tensors (planes as int32 in the device page
    layout of pw_tile_planes, tables as int16), from ``store`` if given, else one
    pinned allocation each."""
    import torch
    R, K = P.shape
    pb = n_bits * R * (K // 32) * 4
    lb = pw_lut_bytes(R, b_min, n_bits)
    if store is None:
        planes = torch.empty((n_bits, R, K // 32), dtype=torch.int32, pin_memory=True)
        luts = torch.empty(lb // 2, dtype=torch.int16, pin_memory=True)
    else:
        planes = store.alloc(pb).view(torch.int32).view(n_bits, R, K // 32)
        luts = store.alloc(lb).view(torch.int16)
    flat, _ = pw_pack(P, parent_lut, n_bits, b_min, luts_out=luts.numpy().view(np.uint16))
    pw_tile_planes(flat, out=planes.numpy().view(np.uint32).reshape(-1))
    return planes, luts


def load_expert_layer(moe: PagedMoE, layer: int, blocks, bits, n_bits: int = 8, b_min: int = 3,
                      alloc_planes=None, stream=None, store: HostStore | None = None,
                      per_plane: bool = False):
    """Registers every block of one layer.

    blocks(e, kind) -> (P uint8 [R][K], parent_lut fp16 [R][2^n]);
    bits[e][kind] -> committed bitwidth; alloc_planes(e, kind) -> device pages
    to allocate (default: all n planes); store -> where the pinned host copies
    live (default: one pinned allocation per array).
    """
    for e in range(moe.E):
        for kind in (KIND_GATE_UP, KIND_DOWN):
            P, par = blocks(e, kind)
            planes, luts = pack_pinned(P, par, n_bits, b_min, store=store)
            na = None if alloc_planes is None else alloc_planes(e, kind)
            moe.register(layer, e, kind, planes, luts, int(bits[e][kind]), n_bits=n_bits,
                         b_min=b_min, alloc_planes=na, stream=stream, per_plane=per_plane)
