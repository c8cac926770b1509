"""Parity of the fused layer on the GPU (through the C ABI) against the oracle.

Bit-exact: routing indices, offsets, permutation; integer-table layers.
Float outputs: rel L2 <= 1e-3 and max abs <= 2e-2 against fp64.
"""
import numpy as np
import pytest

import synth
from oracle import moe as omoe

from _layers import SynthBlocks, assert_close, gpu_layer, oracle_blocks, to_np

pytestmark = pytest.mark.gpu


def _run(m, cfg, x, L, layer=0, k=None, renorm=None, residual=None):
    import torch
    k = cfg.top_k if k is None else k
    renorm = cfg.renorm if renorm is None else renorm
    xd = torch.from_numpy(x).cuda()
    Ld = torch.from_numpy(L).cuda()
    rd = None if residual is None else torch.from_numpy(residual).cuda()
    out, ri, rw, ro, rp = m.pw_moe_forward(layer, xd, Ld, k, renorm, residual=rd, routing=True)
    torch.cuda.synchronize()
    return to_np(out), to_np(ri), to_np(rw), to_np(ro), to_np(rp)


def _check_routing(ref, ri, rw, ro, rp):
    assert np.array_equal(ri, ref["idx"])
    assert np.allclose(rw, ref["w"], rtol=2e-6, atol=1e-7)
    assert np.array_equal(ro, ref["offsets"])
    assert np.array_equal(rp, ref["perm"])


def test_tiny_layer_full():
    cfg = synth.CONFIGS["tiny"]
    m = gpu_layer(cfg)
    x, L = synth.tokens(cfg), synth.logits(cfg)
    out, ri, rw, ro, rp = _run(m, cfg, x, L)
    ref = omoe.layer(x, L, cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), synth.block_bits(cfg)))
    _check_routing(ref, ri, rw, ro, rp)
    assert_close(out, ref["out"])


@pytest.mark.parametrize("q", [3, 4, 5, 6, 7, 8])
def test_tiny_every_bitwidth(q):
    cfg = synth.CONFIGS["tiny"]
    bits = np.full((cfg.E, 2), q, dtype=np.int32)
    m = gpu_layer(cfg, bits={0: bits})
    x, L = synth.tokens(cfg, step=q), synth.logits(cfg, step=q)
    out, *_ = _run(m, cfg, x, L)
    ref = omoe.layer(x, L, cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), bits))
    assert_close(out, ref["out"])


@pytest.mark.parametrize("cfg_name", ["tiny", "pair_build", "prefill_small"])
def test_one_and_two_bit_blocks(cfg_name):
    """Blocks committed at 1 and 2 bits (tables of 2 and 4 entries per row, below
    the 8-entry chunks the kernels otherwise load), mixed with higher bitwidths,
    on both builds of the decode kernel (hidden size 256: without pair tables;
    4096: with them, for q <= 4) and on the tensor-core path (300 tokens)."""
    if cfg_name == "tiny":
        cfg = synth.CONFIGS["tiny"]
    elif cfg_name == "pair_build":
        cfg = synth.CONFIGS["tiny"].with_(H=4096, T=5)
    else:
        cfg = synth.CONFIGS["mixtral_prefill"].with_(T=300, H=256, I=512)
    rng = np.random.default_rng(7)
    bits = rng.integers(1, 9, size=(cfg.E, 2)).astype(np.int32)
    bits[0] = (1, 2)
    bits[1] = (2, 1)
    bits[2] = (3, 4)
    bits[3] = (4, 3)
    m = gpu_layer(cfg, bits={0: bits}, b_min=1)
    x, L = synth.tokens(cfg, step=11), synth.logits(cfg, step=11)
    out, ri, rw, ro, rp = _run(m, cfg, x, L)
    ref = omoe.layer(x, L, cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), bits))
    _check_routing(ref, ri, rw, ro, rp)
    assert_close(out, ref["out"])


@pytest.mark.parametrize("H", [256, 4096])   # the decode kernel's two builds
def test_integer_tables_bit_exact(H):
    """Integer tables whose child table at the committed q is integer, 0/1 tokens
    with 19 ones, top-1 routing: gate sums lie in [38, 57], where e^-g is below
    half an ulp of 1 in fp64 as in fp32, so silu(g) == g on both sides; every
    sum is an exact integer, |h| <= 57 * 19 fits fp16 exactly, and out must
    equal the oracle's fp16 rounding bit for bit."""
    cfg = synth.CONFIGS["tiny"].with_(T=16, top_k=1, renorm=1, H=H)
    rng = np.random.default_rng(99)
    E, H, I = cfg.E, cfg.H, cfg.I
    bits = rng.integers(3, 9, size=(E, 2)).astype(np.int32)
    blk = {}
    for e in range(E):
        for kind in (0, 1):
            R, K = cfg.rows(kind), cfg.cols(kind)
            q = int(bits[e, kind])
            if kind == 0:
                f = np.concatenate([rng.integers(2, 4, size=(I, 1 << q)),       # gate rows: 2 or 3
                                    rng.integers(-1, 2, size=(I, 1 << q))])     # up rows: -1, 0, 1
            else:
                f = rng.integers(-1, 2, size=(R, 1 << q))
            par = np.repeat(f, 1 << (8 - q), axis=1).astype(np.float16)        # child_q == f
            blk[(e, kind)] = (rng.integers(0, 256, size=(R, K), dtype=np.uint8), par)
    src = lambda e, kind: blk[(e, kind)]
    m = gpu_layer(cfg, bits={0: bits}, blocks={0: src})
    x = np.zeros((cfg.T, H), dtype=np.float16)
    for t in range(cfg.T):
        x[t, rng.choice(H, size=19, replace=False)] = 1
    L = synth.logits(cfg)
    out, *_ = _run(m, cfg, x, L)
    ref = omoe.layer(x, L, 1, 1, oracle_blocks(src, bits))
    assert np.array_equal(out.view(np.uint16), ref["out"].astype(np.float16).view(np.uint16))


def test_qwen_decode_layer_full():
    cfg = synth.CONFIGS["qwen_decode"]
    m = gpu_layer(cfg)
    x, L = synth.tokens(cfg), synth.logits(cfg)
    out, ri, rw, ro, rp = _run(m, cfg, x, L)
    ref = omoe.layer(x, L, cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), synth.block_bits(cfg)))
    _check_routing(ref, ri, rw, ro, rp)
    assert_close(out, ref["out"])


def _check_h(m, cfg, ws, ref):
    """h left in the workspace (fp16, permuted pair order) against the oracle's
    fp64 h of every pair, element by element."""
    h = to_np(m.workspace_h(ws, cfg.T, cfg.top_k)).astype(np.float64)
    assert h.shape == ref["h"].shape
    assert_close(h, ref["h"])


@pytest.mark.parametrize("name", ["tiny", "qwen_decode"])
def test_intermediate_h_matches_oracle(name):
    import torch
    cfg = synth.CONFIGS[name]
    m = gpu_layer(cfg)
    x, L = synth.tokens(cfg, step=2), synth.logits(cfg, step=2)
    ws = m.workspace(cfg.T, cfg.top_k)
    m.pw_moe_forward(0, torch.from_numpy(x).cuda(), torch.from_numpy(L).cuda(), cfg.top_k, cfg.renorm, ws=ws)
    torch.cuda.synchronize()
    ref = omoe.layer(x, L, cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), synth.block_bits(cfg)))
    _check_h(m, cfg, ws, ref)


def test_split_k_down_items():
    """An intermediate size much larger than the hidden size (I = 24 H) makes the
    decode kernel split every down item along K (4 parts, added in a fixed
    order): out, h and y against the oracle, and bitwise the same on a rerun."""
    import torch
    cfg = synth.CONFIGS["tiny"].with_(H=256, I=6144, T=5)
    m = gpu_layer(cfg)
    x, L = synth.tokens(cfg, step=8), synth.logits(cfg, step=8)
    ws = m.workspace(cfg.T, cfg.top_k)
    xd, Ld = torch.from_numpy(x).cuda(), torch.from_numpy(L).cuda()
    out = m.pw_moe_forward(0, xd, Ld, cfg.top_k, cfg.renorm, ws=ws).clone()
    torch.cuda.synchronize()
    ref = omoe.layer(x, L, cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), synth.block_bits(cfg)))
    assert_close(to_np(out), ref["out"])
    _check_h(m, cfg, ws, ref)
    y = to_np(m.workspace_y(ws, cfg.T, cfg.top_k)).astype(np.float64)
    assert_close(y, ref["y"])
    again = m.pw_moe_forward(0, xd, Ld, cfg.top_k, cfg.renorm, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), out.view(torch.int16))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mixtral_decode_t1", "mixtral_decode_t4"])
def test_mixtral_decode_full(name):
    """Full-size Mixtral-shaped decode layer: every output column and every
    element of h against the fp64 oracle, routing bit-exact."""
    import torch
    cfg = synth.CONFIGS[name]
    m = gpu_layer(cfg)
    x, L = synth.tokens(cfg), synth.logits(cfg)
    ws = m.workspace(cfg.T, cfg.top_k)
    out, ri, rw, ro, rp = m.pw_moe_forward(0, torch.from_numpy(x).cuda(), torch.from_numpy(L).cuda(),
                                           cfg.top_k, cfg.renorm, ws=ws, routing=True)
    torch.cuda.synchronize()
    ref = omoe.layer(x, L, cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), synth.block_bits(cfg)))
    _check_routing(ref, to_np(ri), to_np(rw), to_np(ro), to_np(rp))
    assert_close(to_np(out), ref["out"])
    _check_h(m, cfg, ws, ref)


def test_prefill_shaped_small():
    # many tokens per expert, ragged counts (Dirichlet mix), small hidden sizes
    cfg = synth.CONFIGS["mixtral_prefill"].with_(T=300, H=256, I=512)
    m = gpu_layer(cfg)
    x, L = synth.tokens(cfg), synth.logits(cfg)
    out, ri, rw, ro, rp = _run(m, cfg, x, L)
    ref = omoe.layer(x, L, cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), synth.block_bits(cfg)))
    _check_routing(ref, ri, rw, ro, rp)
    assert_close(out, ref["out"])


@pytest.mark.slow
def test_mixtral_prefill_sampled():
    """Full-size Mixtral-shaped prefill (2048 tokens) on the tensor-core path:
    routing bit-exact for every token; for 32 sampled tokens (64 routed pairs,
    spread over the experts and over the 128-token tiles), every output column
    and every element of their h rows against the oracle."""
    import torch
    cfg = synth.CONFIGS["mixtral_prefill"]
    m = gpu_layer(cfg)
    x, L = synth.tokens(cfg), synth.logits(cfg)
    ws = m.workspace(cfg.T, cfg.top_k)
    out, ri, rw, ro, rp = m.pw_moe_forward(0, torch.from_numpy(x).cuda(), torch.from_numpy(L).cuda(),
                                           cfg.top_k, cfg.renorm, ws=ws, routing=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(6)
    toks = np.sort(rng.choice(cfg.T, size=32, replace=False))
    ref = omoe.layer(x, L, cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), synth.block_bits(cfg)),
                     out_tokens=toks)
    _check_routing(ref, to_np(ri), to_np(rw), to_np(ro), to_np(rp))
    assert_close(to_np(out)[toks], ref["out"])
    pos = np.sort(ref["inv"].reshape(cfg.T, cfg.top_k)[toks].ravel())   # the sampled tokens' pairs
    h = to_np(m.workspace_h(ws, cfg.T, cfg.top_k)).astype(np.float64)
    assert_close(h[pos], ref["h"][pos])


def test_prefill_gemm_integer_tables_bit_exact():
    """Tensor-core path with integer tables and 0/1 tokens (as in the decode
    test): every product and sum is an exact integer in fp32, so the output must
    equal the oracle's fp16 rounding bit for bit."""
    cfg = synth.CONFIGS["tiny"].with_(T=200, top_k=1, renorm=1)
    rng = np.random.default_rng(98)
    E, H, I = cfg.E, cfg.H, cfg.I
    bits = rng.integers(3, 9, size=(E, 2)).astype(np.int32)
    blk = {}
    for e in range(E):
        for kind in (0, 1):
            R, K = cfg.rows(kind), cfg.cols(kind)
            q = int(bits[e, kind])
            if kind == 0:
                f = np.concatenate([rng.integers(2, 4, size=(I, 1 << q)), rng.integers(-1, 2, size=(I, 1 << q))])
            else:
                f = rng.integers(-1, 2, size=(R, 1 << q))
            par = np.repeat(f, 1 << (8 - q), axis=1).astype(np.float16)
            blk[(e, kind)] = (rng.integers(0, 256, size=(R, K), dtype=np.uint8), par)
    src = lambda e, kind: blk[(e, kind)]
    m = gpu_layer(cfg, bits={0: bits}, blocks={0: src})
    x = np.zeros((cfg.T, H), dtype=np.float16)
    for t in range(cfg.T):
        x[t, rng.choice(H, size=19, replace=False)] = 1
    L = synth.logits(cfg)
    out, *_ = _run(m, cfg, x, L)
    ref = omoe.layer(x, L, 1, 1, oracle_blocks(src, bits))
    assert np.array_equal(out.view(np.uint16), ref["out"].astype(np.float16).view(np.uint16))


def test_residual_topk_extremes_and_determinism():
    import torch
    cfg = synth.CONFIGS["tiny"].with_(T=7)
    m = gpu_layer(cfg)
    src = oracle_blocks(SynthBlocks(cfg, 0), synth.block_bits(cfg))
    x, L = synth.tokens(cfg), synth.logits(cfg)
    res = synth.tokens(cfg, step=3)
    for k, rn in ((1, 1), (1, 0), (cfg.E, 0), (3, 1)):
        out, *_ = _run(m, cfg, x, L, k=k, renorm=rn, residual=res)
        ref = omoe.layer(x, L, k, rn, src, residual=res)
        assert_close(out, ref["out"])
        again, *_ = _run(m, cfg, x, L, k=k, renorm=rn, residual=res)
        assert np.array_equal(out.view(np.uint16), again.view(np.uint16))
    # T = 0 is a no-op
    ws = m.workspace(0, 2)
    e = torch.empty((0, cfg.H), dtype=torch.float16, device="cuda")
    m.pw_moe_forward(0, e, torch.empty((0, cfg.E), dtype=torch.float32, device="cuda"), 2, 1, ws=ws)


def test_single_expert_layer():
    cfg = synth.CONFIGS["tiny"].with_(E=1, top_k=1, renorm=1, T=5)
    m = gpu_layer(cfg)
    x, L = synth.tokens(cfg), synth.logits(cfg)
    out, *_ = _run(m, cfg, x, L)
    ref = omoe.layer(x, L, 1, 1, oracle_blocks(SynthBlocks(cfg, 0), synth.block_bits(cfg)))
    assert_close(out, ref["out"])


def test_host_entry_matches_device_entry():
    import torch
    cfg = synth.CONFIGS["qwen_decode"]
    m = gpu_layer(cfg)
    x, L = synth.tokens(cfg), synth.logits(cfg)
    dev, *_ = _run(m, cfg, x, L)
    xh = torch.from_numpy(x).pin_memory()
    Lh = torch.from_numpy(L).pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    m.pw_moe_forward_host(0, xh, Lh, cfg.top_k, cfg.renorm, oh)
    assert np.array_equal(oh.numpy().view(np.uint16), dev.view(np.uint16))


def test_nan_logit_sets_status_not_fault():
    import torch
    import any_precision_weight_gb300 as pw
    cfg = synth.CONFIGS["tiny"]
    m = gpu_layer(cfg)
    x, L = synth.tokens(cfg), synth.logits(cfg)
    L[3, 2] = np.nan
    ws = m.workspace(cfg.T, cfg.top_k)
    m.pw_moe_forward(0, torch.from_numpy(x).cuda(), torch.from_numpy(L).cuda(), cfg.top_k, cfg.renorm, ws=ws)
    assert m.workspace_status(ws) & pw.PW_STATUS_NAN_LOGIT
    L[3, 2] = 0.0
    m.pw_moe_forward(0, torch.from_numpy(x).cuda(), torch.from_numpy(L).cuda(), cfg.top_k, cfg.renorm, ws=ws)
    assert m.workspace_status(ws) == 0


def test_forward_argument_errors():
    import torch
    import any_precision_weight_gb300 as pw
    cfg = synth.CONFIGS["tiny"]
    m = gpu_layer(cfg)
    x = torch.from_numpy(synth.tokens(cfg)).cuda()
    L = torch.from_numpy(synth.logits(cfg)).cuda()
    with pytest.raises(pw.PWError) as e:
        m.pw_moe_forward(0, x, L, cfg.E + 1, 1)
    assert e.value.code == pw.PW_EINVAL
    with pytest.raises(pw.PWError) as e:
        m.pw_moe_forward(1, x, L, 2, 1)
    assert e.value.code == pw.PW_EINVAL
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pw.PWError) as e:
        m.pw_moe_forward(0, x, L, 2, 1, ws=small)
    assert e.value.code == pw.PW_ENOMEM
    # a table with an unregistered block refuses to run
    m2 = pw.PagedMoE(1, cfg.E, cfg.H, cfg.I)
    with pytest.raises(pw.PWError) as e:
        m2.pw_moe_forward(0, x, L, 2, 1)
    assert e.value.code == pw.PW_EINVAL


@pytest.mark.parametrize("T", [16, 300])   # the fused decode kernel and the separate routing kernel
def test_routing_statistics_follow_the_oracle_moving_average(T):
    import torch
    cfg = synth.CONFIGS["tiny"]
    m = gpu_layer(cfg, n_layers=2, bits={0: synth.block_bits(cfg, 0), 1: synth.block_bits(cfg, 1)})
    stats = torch.full((2, cfg.E), 1.0 / cfg.E, dtype=torch.float32, device="cuda")
    alpha = 0.2
    m.pw_stats_attach(stats, alpha)
    want = np.full((2, cfg.E), 1.0 / cfg.E)
    for step in range(4):
        for l in range(2):
            x = torch.from_numpy(synth.tokens(cfg, step=step, T=T)).cuda()
            L = synth.logits(cfg, l, step=step, T=T)
            m.pw_moe_forward(l, x, torch.from_numpy(L).cuda(), cfg.top_k, cfg.renorm)
            idx, w = omoe.route(L, cfg.top_k, cfg.renorm)
            want[l] = omoe.stats_update(want[l], idx, w, cfg.E, alpha)
    torch.cuda.synchronize()
    got = stats.cpu().numpy().astype(np.float64)
    assert np.allclose(got, want, rtol=1e-5, atol=1e-7)
    assert np.allclose(got.sum(axis=1), 1.0, atol=1e-5)      # renorm: every batch adds mass 1
    # detached: forwards leave the statistics alone
    m.pw_stats_attach(None)
    before = stats.clone()
    m.pw_moe_forward(0, x, torch.from_numpy(L).cuda(), cfg.top_k, cfg.renorm)
    torch.cuda.synchronize()
    assert torch.equal(stats, before)


def test_stats_attach_rejects_bad_alpha():
    import torch
    import any_precision_weight_gb300 as pw
    cfg = synth.CONFIGS["tiny"]
    m = gpu_layer(cfg)
    s = torch.zeros((1, cfg.E), dtype=torch.float32, device="cuda")
    for a in (0.0, -0.5, 1.5):
        with pytest.raises(pw.PWError) as e:
            m.pw_stats_attach(s, a)
        assert e.value.code == pw.PW_EINVAL


# ----------------------------------------------------------------------------- edge cases

def test_empty_batch_is_a_no_op():
    import torch
    cfg = synth.CONFIGS["tiny"]
    m = gpu_layer(cfg)
    x = torch.empty((0, cfg.H), dtype=torch.float16, device="cuda")
    L = torch.empty((0, cfg.E), dtype=torch.float32, device="cuda")
    out = m.pw_moe_forward(0, x, L, cfg.top_k, cfg.renorm)
    torch.cuda.synchronize()
    assert out.shape == (0, cfg.H)
    oh = torch.empty((0, cfg.H), dtype=torch.float16).pin_memory()
    m.pw_moe_forward_host(0, x.cpu().pin_memory(), L.cpu().pin_memory(), cfg.top_k, cfg.renorm, oh)


@pytest.mark.parametrize("T", [64, 65])     # the largest fused batch and the first unfused one
def test_fused_path_boundary(T):
    cfg = synth.CONFIGS["tiny"].with_(T=T)
    m = gpu_layer(cfg)
    x, L = synth.tokens(cfg), synth.logits(cfg)
    out, ri, rw, ro, rp = _run(m, cfg, x, L)
    ref = omoe.layer(x, L, cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), synth.block_bits(cfg)))
    _check_routing(ref, ri, rw, ro, rp)
    assert_close(out, ref["out"])


@pytest.mark.parametrize("E", [78, 79])
def test_descriptor_cache_boundary(E):
    """The decode kernel keeps every block descriptor of the layer in shared
    memory while 2E descriptors fit (E <= 78) and reads them per item from
    global memory above that; both sides of the boundary against the oracle."""
    cfg = synth.CONFIGS["tiny"].with_(E=E, T=24, top_k=3, H=128, I=256)
    m = gpu_layer(cfg)
    x, L = synth.tokens(cfg), synth.logits(cfg)
    out, ri, rw, ro, rp = _run(m, cfg, x, L)
    ref = omoe.layer(x, L, cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), synth.block_bits(cfg)))
    _check_routing(ref, ri, rw, ro, rp)
    assert_close(out, ref["out"])


def test_largest_expert_count_and_pair_count():
    # E = 256 experts (the routing's limit) and T * k = 256 pairs (the fused kernel's limit)
    cfg = synth.CONFIGS["tiny"].with_(E=256, T=32, top_k=8, H=128, I=128)
    m = gpu_layer(cfg)
    x, L = synth.tokens(cfg), synth.logits(cfg)
    out, ri, rw, ro, rp = _run(m, cfg, x, L)
    ref = omoe.layer(x, L, cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), synth.block_bits(cfg)))
    _check_routing(ref, ri, rw, ro, rp)
    assert_close(out, ref["out"])


@pytest.mark.parametrize("T", [16, 300])
def test_every_token_routed_to_one_expert(T):
    # one expert far above the others takes every token (the hottest-expert extreme):
    # its tiles carry all T tokens, the others none
    cfg = synth.CONFIGS["tiny"].with_(T=T)
    m = gpu_layer(cfg)
    x = synth.tokens(cfg)
    L = synth.logits(cfg).copy()
    L[:, 5] += 40.0
    out, ri, rw, ro, rp = _run(m, cfg, x, L)
    ref = omoe.layer(x, L, cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), synth.block_bits(cfg)))
    assert (ref["idx"][:, 0] == 5).all()
    _check_routing(ref, ri, rw, ro, rp)
    assert_close(out, ref["out"])
