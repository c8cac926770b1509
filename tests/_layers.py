"""Test helpers: one synthetic layer set up twice, on the GPU through the
library (pw_pack + pw_block_register) and as oracle blocks, from the same
seeded inputs."""
from __future__ import annotations

import numpy as np

import synth
from oracle import moe as omoe

REL_L2 = 1e-3     # float tolerance of the fused layer vs the fp64 oracle
MAX_ABS = 2e-2
GUARD = 256       # canary bytes on both sides of every device buffer of the test layers
LIVE = []         # layers built by the running test; their guards are checked after it


class SynthBlocks:
    """blocks(e, kind) -> (P, parent_lut) for one layer of a synth config."""

    def __init__(self, cfg, layer):
        self.cfg, self.layer = cfg, layer

    def __call__(self, e, kind):
        return (synth.parent_indices(self.cfg, self.layer, e, kind),
                synth.parent_lut(self.cfg, self.layer, e, kind))


def gpu_layer(cfg, n_layers=1, bits=None, blocks=None, alloc_planes=None, layers=None, per_plane=False,
              b_min=3):
    """A PagedMoE with the given layers registered.  bits[l] -> [E][2]; b_min:
    the lowest bitwidth whose tables are stored."""
    import any_precision_weight_gb300 as pw
    from any_precision_weight_gb300.model import load_expert_layer
    m = pw.PagedMoE(n_layers, cfg.E, cfg.H, cfg.I, guard=GUARD)
    LIVE.append(m)
    for l in (range(n_layers) if layers is None else layers):
        b = synth.block_bits(cfg, l) if bits is None else bits[l]
        src = SynthBlocks(cfg, l) if blocks is None else blocks[l]
        load_expert_layer(m, l, src, b, alloc_planes=alloc_planes, per_plane=per_plane, b_min=b_min)
    return m


def oracle_blocks(src, bits):
    """e -> (gate_up Block, down Block) for the oracle, built on demand."""
    cache = {}

    def get(e):
        if e not in cache:
            gu = omoe.Block(*src(e, 0), bits[e][0])
            dn = omoe.Block(*src(e, 1), bits[e][1])
            cache[e] = (gu, dn)
        return cache[e]
    return get


def assert_close(got, want, rel=REL_L2, mx=MAX_ABS):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape
    err = got - want
    rl2 = np.linalg.norm(err) / max(np.linalg.norm(want), 1e-30)
    ma = np.abs(err).max() if err.size else 0.0
    assert rl2 <= rel and ma <= mx, f"rel L2 {rl2:.3e} (<= {rel}), max abs {ma:.3e} (<= {mx})"
    return rl2, ma


def to_np(t):
    return t.detach().cpu().numpy()
