"""The fused MoE expert layer, restated plainly in fp64 (oracle; test
infrastructure only).

Sources: PagedWeight technical summary, Problem statement (an MoE activates a
subset of experts per token) and Core components sections 1 and 3 ("Paged
Weight Representation": per-(layer, expert, gate_up|down) linear blocks at a
committed bitwidth q_i; "Fused Mixed-Precision Kernel": one fused operation
reading APL planes and tables with a different bitwidth per block).  The
pages leave the layer arithmetic to the MoE convention; this build reads it
as:

1. route: per token, order experts by (logit descending, expert index
   ascending) and keep the first k; p = softmax over all E logits (fp64,
   max-subtracted); w[t][j] = p[idx[t][j]], divided by its sum over j when
   ``renorm`` is set;
2. permute: stable counting sort of the pairs (t, j) by expert, then by t;
   offsets = exclusive prefix sum of the per-expert counts;
3. expert MLP per pair: rows [0, I) of the gate_up block are the gate, rows
   [I, 2I) the up projection; h = silu(gate . x) * (up . x) with
   silu(z) = z / (1 + e^-z); y = W_down . h;
4. combine: out[t] = residual[t] (if given) + sum_j w[t][j] * y(t, j).

Routing statistics (the planner's routing-mass input) are the plain
per-expert sum of routing weights divided by the batch size, folded into an
exponential moving average.

Every step is fp64 from the fp16 / fp32 inputs; the GPU's fp16 intermediates
are not modelled.
"""
import numpy as np

from . import apl


# ----------------------------------------------------------------------------- routing

def route(logits: np.ndarray, k: int, renorm: int):
    """Top-k experts per token and their routing weights.

    Returns idx int64 [T][k] (descending logit, ties to the lower expert
    index) and w fp64 [T][k].
    """
    L = np.asarray(logits, dtype=np.float32)
    T, E = L.shape
    if not (1 <= k <= E):
        raise ValueError("top_k out of range")
    if np.isnan(L).any():
        raise ValueError("NaN logit")
    idx = np.zeros((T, k), dtype=np.int64)
    w = np.zeros((T, k), dtype=np.float64)
    for t in range(T):
        row = [float(v) for v in L[t]]            # the given fp32 values, exactly
        order = sorted(range(E), key=lambda e: (-row[e], e))
        top = order[:k]
        z = np.asarray(row, dtype=np.float64)
        ez = np.exp(z - z.max())
        p = ez / ez.sum()
        wt = p[top]
        if renorm:
            wt = wt / wt.sum()
        idx[t] = top
        w[t] = wt
    return idx, w


def routing_mass(idx: np.ndarray, w: np.ndarray, E: int):
    """Per-expert routing mass of one batch: M[e] = (1/T) * sum of w[t][j] over
    the pairs with idx[t][j] == e (the routing-mass signal of the runtime
    planner, "Quality-Aware Runtime Planner").  fp64 [E]."""
    idx = np.asarray(idx)
    w = np.asarray(w, dtype=np.float64)
    T, k = idx.shape
    M = np.zeros(E, dtype=np.float64)
    for t in range(T):
        for j in range(k):
            M[idx[t, j]] += w[t, j]
    return M / T if T else M


def stats_update(m: np.ndarray, idx: np.ndarray, w: np.ndarray, E: int, alpha: float):
    """One step of the routing-mass moving average: (1 - alpha) * m + alpha * M."""
    return (1.0 - alpha) * np.asarray(m, dtype=np.float64) + alpha * routing_mass(idx, w, E)


def permute(idx: np.ndarray, E: int):
    """Stable counting sort of pairs by expert.

    Pair id = t * k + j.  Returns counts [E], offsets [E+1], perm [T*k]
    (pair ids in expert-major, token-ascending order) and inv [T*k]
    (position of each pair id in perm).
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            counts[idx[t, j]] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:E].copy()
    perm = np.zeros(T * k, dtype=np.int64)
    for t in range(T):                       # t ascending keeps each expert's run stable
        for j in range(k):
            e = idx[t, j]
            perm[fill[e]] = t * k + j
            fill[e] += 1
    inv = np.zeros(T * k, dtype=np.int64)
    inv[perm] = np.arange(T * k)
    return counts, offsets, perm, inv


# ----------------------------------------------------------------------------- expert MLP

def silu(z):
    with np.errstate(over="ignore"):      # e^-z -> inf gives silu -> -0, as it should
        return z / (1.0 + np.exp(-z))


def expert_h(W_gu: np.ndarray, X: np.ndarray) -> np.ndarray:
    """h [n][I] = silu(gate . x) * (up . x) for token rows X [n][H]."""
    I = W_gu.shape[0] // 2
    X = np.asarray(X, dtype=np.float64)
    g = X @ W_gu[:I].T
    u = X @ W_gu[I:].T
    return silu(g) * u


def expert_y(W_dn: np.ndarray, Hrows: np.ndarray) -> np.ndarray:
    """y [n][H] = W_down . h for rows Hrows [n][I]."""
    return np.asarray(Hrows, dtype=np.float64) @ W_dn.T


# ----------------------------------------------------------------------------- layer

class Block:
    """One linear block as the oracle sees it: parent indices, its own child
    table at the committed bitwidth q, and n."""

    def __init__(self, P, parent_lut, q, n=8):
        self.P = np.asarray(P)
        self.q = int(q)
        self.n = int(n)
        self.lut = apl.child_lut(parent_lut, self.q, self.n)

    def weights(self, rows=None) -> np.ndarray:
        P = self.P if rows is None else self.P[rows]
        lut = self.lut if rows is None else self.lut[rows]
        return apl.dequant(P, lut, self.q, self.n)


def layer(x, logits, k, renorm, blocks, residual=None, out_rows=None, out_tokens=None):
    """The whole layer.

    ``blocks(e)`` returns (gate_up Block, down Block) for expert e.
    ``out_rows``: optional list of hidden indices; when given, only those
    output columns are computed (h is still computed in full, as it must be).
    ``out_tokens``: optional list of tokens; when given, routing and the
    permutation still cover every token, but the expert MLPs and the combine
    run only for the pairs of these tokens, and ``out`` has their rows.
    Returns a dict with idx, w, counts, offsets, perm, inv, h (per pair, in
    perm order; zero for pairs not computed), y (same, restricted to
    out_rows) and out [len(out_tokens) or T][len(out_rows) or H].
    """
    x = np.asarray(x, dtype=np.float16).astype(np.float64)
    T, H = x.shape
    E = np.asarray(logits).shape[1]
    idx, w = route(logits, k, renorm)
    counts, offsets, perm, inv = permute(idx, E)
    cols = np.arange(H) if out_rows is None else np.asarray(out_rows)
    toks_out = np.arange(T) if out_tokens is None else np.asarray(out_tokens)
    wanted = np.zeros(T, dtype=bool)
    wanted[toks_out] = True
    h_all = None
    y_all = np.zeros((T * k, len(cols)), dtype=np.float64)
    for e in range(E):
        pos = np.arange(offsets[e], offsets[e + 1])
        pos = pos[wanted[perm[pos] // k]]
        if len(pos) == 0:
            continue
        toks = perm[pos] // k
        gu, dn = blocks(e)
        h = expert_h(gu.weights(), x[toks])
        if h_all is None:
            h_all = np.zeros((T * k, h.shape[1]), dtype=np.float64)
        h_all[pos] = h
        y_all[pos] = expert_y(dn.weights(cols), h)
    out = np.zeros((len(toks_out), len(cols)), dtype=np.float64)
    if residual is not None:
        out += np.asarray(residual, dtype=np.float16).astype(np.float64)[toks_out][:, cols]
    for i, t in enumerate(toks_out):
        for j in range(k):
            out[i] += w[t, j] * y_all[inv[t * k + j]]
    return dict(idx=idx, w=w, counts=counts, offsets=offsets, perm=perm, inv=inv,
                h=h_all, y=y_all, out=out)
