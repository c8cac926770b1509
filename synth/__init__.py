"""Seeded synthetic inputs for the fused APL MoE layer.

This module is shared by the tests, the benchmark and the oracle's tests, and
it holds none of the method's arithmetic: it draws random numbers with the
shapes, value distributions and routing skew of the workloads named on the
PagedWeight pages (Qwen1.5-MoE-A2.7B, Mixtral-8x7B shapes; "Empirical
validation" in the core contributions list), and nothing else.  It never
packs bit-planes, builds child lookup tables, dequantises, routes, permutes
or combines; the product and the oracle each do that with their own code.

Every draw comes from ``numpy.random.default_rng`` (PCG64) seeded by a
``SeedSequence`` over (config seed, stream tag, layer, expert, kind), so that
one block can be regenerated alone and in any order.

Recipe (per config):

* tokens x: fp16(N(0, 1)), shape [T][H];
* parent indices P: uniform on {0..2^n - 1}, n = 8, shape [R][K], uint8;
* parent LUT: per output row, 2^n draws of N(0, 0.02) sorted ascending and
  rounded to fp16, shape [R][2^n];
* router logits: fp32, N(0, 1), plus a per-expert bias (Zipf for the
  Qwen-shaped layer, log-Dirichlet for Mixtral prefill) added in fp64 and
  rounded once to fp32;
* committed bits per block: uniform over the config's set; for the
  Qwen-shaped layer the "hot" experts (routing mass >= 1/E) draw from
  {6, 7, 8};
* 24-layer stack: bits from a greedy fit of a synthetic damage score to 40%
  of the fp16 weight bytes (the input recipe, standing in for the planner's
  output; the hot path only consumes the bits).
"""
from __future__ import annotations

import heapq
from dataclasses import dataclass, field

import numpy as np

N_BITS = 8          # parent bitwidth of every block
B_MIN = 3           # smallest committed bitwidth the configs use
KIND_GATE_UP = 0
KIND_DOWN = 1

_TAG_X, _TAG_LOGITS, _TAG_IDX, _TAG_LUT, _TAG_BITS, _TAG_BIAS, _TAG_SENS, _TAG_RELOAD = range(8)


@dataclass(frozen=True)
class LayerConfig:
    """Shape and draw recipe of one synthetic MoE layer (or a stack of them)."""
    name: str
    T: int                 # tokens in the batch
    H: int                 # hidden size (K of gate_up, R of down)
    E: int                 # experts
    I: int                 # expert intermediate size
    top_k: int
    renorm: int            # 1: routing weights renormalised over the top-k
    bits: tuple            # committed bitwidths drawn uniformly from this set
    bias: str = "none"     # "none" | "zipf" | "dirichlet"
    hot_bits: tuple = ()   # set for hot experts (zipf only)
    seed: int = 0
    n_layers: int = 1
    stack_fit: bool = False   # bits from the greedy fit to a byte target

    def rows(self, kind: int) -> int:
        return 2 * self.I if kind == KIND_GATE_UP else self.H

    def cols(self, kind: int) -> int:
        return self.H if kind == KIND_GATE_UP else self.I

    def with_(self, **kw) -> "LayerConfig":
        d = dict(self.__dict__)
        d.update(kw)
        return LayerConfig(**d)


CONFIGS = {
    # 1. tiny correctness layer
    "tiny": LayerConfig("tiny", T=16, H=256, E=8, I=512, top_k=2, renorm=1,
                        bits=(3, 4, 5, 6, 7, 8), seed=20261),
    # 2. Qwen1.5-MoE-A2.7B-shaped decode layer, batch 4
    "qwen_decode": LayerConfig("qwen_decode", T=4, H=2048, E=60, I=1408, top_k=4, renorm=0,
                               bits=(3, 4, 5, 6, 7, 8), bias="zipf", hot_bits=(6, 7, 8),
                               seed=20262),
    # 3. Mixtral-8x7B-shaped decode layer, batch 1 and batch 4
    "mixtral_decode_t1": LayerConfig("mixtral_decode_t1", T=1, H=4096, E=8, I=14336, top_k=2,
                                     renorm=1, bits=(3, 4, 5, 6, 8), seed=20263),
    "mixtral_decode_t4": LayerConfig("mixtral_decode_t4", T=4, H=4096, E=8, I=14336, top_k=2,
                                     renorm=1, bits=(3, 4, 5, 6, 8), seed=20263),
    # 4. Mixtral-8x7B-shaped prefill, 2048 tokens, Dirichlet(1) expert mix
    "mixtral_prefill": LayerConfig("mixtral_prefill", T=2048, H=4096, E=8, I=14336, top_k=2,
                                   renorm=1, bits=(3, 4, 5, 6, 7, 8), bias="dirichlet",
                                   seed=20264),
    # 5. 24-layer Qwen-shaped stack, decode batch 4, bits fitted to 40% of fp16 bytes
    "qwen_stack": LayerConfig("qwen_stack", T=4, H=2048, E=60, I=1408, top_k=4, renorm=0,
                              bits=(3, 4, 5, 6, 7, 8), bias="zipf", hot_bits=(6, 7, 8),
                              seed=20265, n_layers=24, stack_fit=True),
}


def _rng(cfg: LayerConfig, *tag) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([cfg.seed, *tag]))


# ----------------------------------------------------------------------------- tokens, logits

def tokens(cfg: LayerConfig, step: int = 0, T: int | None = None) -> np.ndarray:
    """fp16 tokens [T][H], N(0, 1)."""
    T = cfg.T if T is None else T
    return _rng(cfg, _TAG_X, step).standard_normal((T, cfg.H)).astype(np.float16)


def expert_mass(cfg: LayerConfig, layer: int = 0) -> np.ndarray:
    """Per-expert routing prior p_e (sums to 1) that skews the logits.

    zipf: p_r proportional to r^-1.1 over ranks r = 1..E, ranks assigned to
    experts by a seeded permutation.  dirichlet: one Dirichlet(1) draw.
    none: uniform.
    """
    E = cfg.E
    if cfg.bias == "zipf":
        r = np.arange(1, E + 1, dtype=np.float64)
        pr = r ** -1.1
        pr /= pr.sum()
        perm = _rng(cfg, _TAG_BIAS, layer).permutation(E)
        p = np.empty(E)
        p[perm] = pr          # expert perm[i] has rank i + 1
        return p
    if cfg.bias == "dirichlet":
        return _rng(cfg, _TAG_BIAS, layer).dirichlet(np.ones(E))
    return np.full(E, 1.0 / E)


def hot_experts(cfg: LayerConfig, layer: int = 0) -> np.ndarray:
    """Boolean [E]: experts whose prior mass is at least 1/E."""
    return expert_mass(cfg, layer) >= 1.0 / cfg.E


def logits(cfg: LayerConfig, layer: int = 0, step: int = 0, T: int | None = None) -> np.ndarray:
    """fp32 router logits [T][E]: N(0, 1) plus ln p_e, summed in fp64, rounded once."""
    T = cfg.T if T is None else T
    z = _rng(cfg, _TAG_LOGITS, layer, step).standard_normal((T, cfg.E))
    if cfg.bias != "none":
        z = z + np.log(expert_mass(cfg, layer))[None, :]
    return z.astype(np.float32)


# ----------------------------------------------------------------------------- weights

def parent_indices(cfg: LayerConfig, layer: int, expert: int, kind: int) -> np.ndarray:
    """uint8 parent indices [R][K], uniform on {0..255}."""
    R, K = cfg.rows(kind), cfg.cols(kind)
    return _rng(cfg, _TAG_IDX, layer, expert, kind).integers(0, 1 << N_BITS, size=(R, K),
                                                             dtype=np.uint8)


def parent_lut(cfg: LayerConfig, layer: int, expert: int, kind: int) -> np.ndarray:
    """fp16 parent lookup table [R][2^n]: per row, sorted N(0, 0.02) centroids."""
    R = cfg.rows(kind)
    c = _rng(cfg, _TAG_LUT, layer, expert, kind).normal(0.0, 0.02, size=(R, 1 << N_BITS))
    c.sort(axis=1)
    return c.astype(np.float16)


def block_bits(cfg: LayerConfig, layer: int = 0) -> np.ndarray:
    """int32 [E][2] committed bits per (expert, kind)."""
    if cfg.stack_fit:
        return stack_bits(cfg)[layer]
    rng = _rng(cfg, _TAG_BITS, layer)
    out = rng.choice(np.asarray(cfg.bits), size=(cfg.E, 2)).astype(np.int32)
    if cfg.hot_bits:
        hot = hot_experts(cfg, layer)
        hb = rng.choice(np.asarray(cfg.hot_bits), size=(cfg.E, 2)).astype(np.int32)
        out[hot] = hb[hot]
    return out


# ----------------------------------------------------------------------------- 24-layer stack

def resident_bytes(R: int, K: int, q: int, b_min: int = B_MIN) -> int:
    """Device bytes of one block at q bits: q planes plus the LUTs for b_min..q."""
    return R * K * q // 8 + R * 2 * sum(1 << c for c in range(b_min, q + 1))


@dataclass
class _Blk:
    layer: int
    expert: int
    kind: int
    R: int
    K: int
    s: float
    m: float
    floor: int
    q: int = N_BITS


def stack_bits(cfg: LayerConfig, target_frac: float = 0.40) -> np.ndarray:
    """int32 [L][E][2] bits for the stack: greedy lowest damage per byte saved.

    Input recipe only.  Start at q = 8 everywhere.  Lowering block i from b
    to b - 1 costs damage m_i * s_i * R * K * (4^-(b-1) - 4^-b) with s_i a
    seeded LogNormal(0, 1) stand-in sensitivity and m_i = 1 + E * p_e a
    routing-mass multiplier; it saves R*K/8 plane bytes and the 2^b-entry LUT.
    Hot experts stop at 6 bits, the rest at 3.  Reductions are taken in order
    of least damage per byte (ties: lower block id) until the resident bytes
    reach ``target_frac`` of the fp16 bytes.
    """
    L, E = cfg.n_layers, cfg.E
    blocks = []
    for l in range(L):
        p = expert_mass(cfg, l)
        hot = p >= 1.0 / E
        sens = _rng(cfg, _TAG_SENS, l).lognormal(0.0, 1.0, size=(E, 2))
        for e in range(E):
            for kind in (KIND_GATE_UP, KIND_DOWN):
                blocks.append(_Blk(l, e, kind, cfg.rows(kind), cfg.cols(kind),
                                   float(sens[e, kind]), 1.0 + E * float(p[e]),
                                   6 if hot[e] else B_MIN))
    fp16_total = sum(b.R * b.K * 2 for b in blocks)
    target = target_frac * fp16_total
    total = sum(resident_bytes(b.R, b.K, b.q) for b in blocks)

    def cand(i):
        b = blocks[i]
        if b.q <= b.floor:
            return None
        dmg = b.m * b.s * b.R * b.K * (4.0 ** -(b.q - 1) - 4.0 ** -b.q)
        saved = b.R * b.K / 8 + b.R * 2 * (1 << b.q)
        return (dmg / saved, i)

    heap = [c for c in (cand(i) for i in range(len(blocks))) if c is not None]
    heapq.heapify(heap)
    while total > target and heap:
        _, i = heapq.heappop(heap)
        b = blocks[i]
        total -= resident_bytes(b.R, b.K, b.q) - resident_bytes(b.R, b.K, b.q - 1)
        b.q -= 1
        c = cand(i)
        if c is not None:
            heapq.heappush(heap, c)
    out = np.zeros((L, E, 2), dtype=np.int32)
    for b in blocks:
        out[b.layer, b.expert, b.kind] = b.q
    return out


def reload_plan(cfg: LayerConfig, bits: np.ndarray, frac: float = 0.25) -> list:
    """Blocks re-committed mid-run: a seeded ``frac`` of blocks with q < 8,
    each raised to min(8, q + 2).  Returns [(layer, expert, kind, q_old, q_new)]."""
    cand = [(l, e, k) for l in range(bits.shape[0]) for e in range(bits.shape[1])
            for k in range(2) if bits[l, e, k] < N_BITS]
    rng = _rng(cfg, _TAG_RELOAD)
    n = int(round(frac * len(cand)))
    pick = sorted(rng.choice(len(cand), size=n, replace=False).tolist())
    out = []
    for i in pick:
        l, e, k = cand[i]
        q = int(bits[l, e, k])
        out.append((l, e, k, q, min(N_BITS, q + 2)))
    return out
