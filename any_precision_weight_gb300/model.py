"""Loading quantised MoE blocks into a PagedMoE page table.

Marshalling only: the packing is pw_pack (C++), the registration is
pw_block_register; this module moves arrays into pinned host memory and
hands the pointers over.
"""
from __future__ import annotations

import numpy as np

from . import KIND_DOWN, KIND_GATE_UP, PagedMoE, pw_lut_bytes, pw_pack


def pack_pinned(P: np.ndarray, parent_lut: np.ndarray, n_bits: int = 8, b_min: int = 3):
    """pw_pack into pinned torch CPU tensors (planes as int32, tables as int16)."""
    import torch
    R, K = P.shape
    planes = torch.empty((n_bits, R, K // 32), dtype=torch.int32, pin_memory=True)
    luts = torch.empty(pw_lut_bytes(R, b_min, n_bits) // 2, dtype=torch.int16, pin_memory=True)
    pw_pack(P, parent_lut, n_bits, b_min, planes_out=planes.numpy().view(np.uint32),
            luts_out=luts.numpy().view(np.uint16))
    return planes, luts


def load_expert_layer(moe: PagedMoE, layer: int, blocks, bits, n_bits: int = 8, b_min: int = 3,
                      alloc_planes=None, stream=None):
    """Registers every block of one layer.

    blocks(e, kind) -> (P uint8 [R][K], parent_lut fp16 [R][2^n]);
    bits[e][kind] -> committed bitwidth; alloc_planes(e, kind) -> device pages
    to allocate (default: all n planes).
    """
    for e in range(moe.E):
        for kind in (KIND_GATE_UP, KIND_DOWN):
            P, par = blocks(e, kind)
            planes, luts = pack_pinned(P, par, n_bits, b_min)
            na = None if alloc_planes is None else alloc_planes(e, kind)
            moe.register(layer, e, kind, planes, luts, int(bits[e][kind]), n_bits=n_bits,
                         b_min=b_min, alloc_planes=na, stream=stream)
