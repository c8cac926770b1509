"""The page table's reload / commit protocol on the GPU.

Pinned by: before a commit the output is bitwise that of a run that never
reloaded; after it, it equals the oracle at the new bitwidth and bitwise a
table registered at that bitwidth from the start; a reload writes only the
planes above the resident ones; every misuse returns its status code.
"""
import numpy as np
import pytest

import synth
from oracle import moe as omoe

from _layers import SynthBlocks, assert_close, gpu_layer, oracle_blocks, to_np

pytestmark = pytest.mark.gpu


def _fwd(m, cfg, x, L):
    import torch
    out = m.pw_moe_forward(0, x, L, cfg.top_k, cfg.renorm)
    torch.cuda.synchronize()
    return to_np(out)


def test_reload_then_commit_changes_bits_at_the_boundary():
    import torch
    cfg = synth.CONFIGS["tiny"]
    E = cfg.E
    lo = np.full((E, 2), 4, dtype=np.int32)
    hi = lo.copy()
    hi[:, 0] = 7                                  # every gate_up block goes 4 -> 7
    m = gpu_layer(cfg, bits={0: lo})
    fresh = gpu_layer(cfg, bits={0: hi})
    x = torch.from_numpy(synth.tokens(cfg)).cuda()
    L = torch.from_numpy(synth.logits(cfg)).cuda()
    before = _fwd(m, cfg, x, L)
    pages_before = [to_np(m.pages(0, e, 0)[0]).copy() for e in range(E)]

    copy = torch.cuda.Stream()
    for e in range(E):
        m.pw_reload_async(0, e, 0, 7, stream=copy)
        assert m.pw_block_state(0, e, 0)[2] == 7
    # still at q = 4: same bits as before, in flight or not
    during = _fwd(m, cfg, x, L)
    assert np.array_equal(during.view(np.uint16), before.view(np.uint16))
    for e in range(E):
        m.pw_set_commit(0, e, 0, 7)               # stream-ordered after the copies
    after = _fwd(m, cfg, x, L)
    want = _fwd(fresh, cfg, x, L)
    assert np.array_equal(after.view(np.uint16), want.view(np.uint16))
    ref = omoe.layer(to_np(x), to_np(L), cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), hi))
    assert_close(after, ref["out"])
    torch.cuda.synchronize()
    pb = m.pages(0, 0, 0)[0].numel() // 8
    for e in range(E):
        q, res, tgt = m.pw_block_state(0, e, 0)
        assert (q, res, tgt) == (7, 7, 0)
        now = to_np(m.pages(0, e, 0)[0])
        # resident planes untouched; reloaded planes equal the host backing store
        assert np.array_equal(now[:4 * pb], pages_before[e][:4 * pb])
        host = m._keep[(0, e, 0)][2].numpy().view(np.uint8).reshape(-1)
        assert np.array_equal(now[4 * pb:7 * pb], host[4 * pb:7 * pb])
    # lowering needs no reload
    for e in range(E):
        m.pw_set_commit(0, e, 0, 4)
    assert np.array_equal(_fwd(m, cfg, x, L).view(np.uint16), before.view(np.uint16))


def test_query_then_commit_and_state():
    import torch
    cfg = synth.CONFIGS["tiny"]
    bits = np.full((cfg.E, 2), 3, dtype=np.int32)
    m = gpu_layer(cfg, bits={0: bits})
    copy = torch.cuda.Stream()
    assert m.pw_reload_query(0, 1, 1) == 1            # nothing pending
    m.pw_reload_async(0, 1, 1, 8, stream=copy)
    copy.synchronize()
    assert m.pw_reload_query(0, 1, 1) == 1
    assert m.pw_block_state(0, 1, 1) == (3, 8, 0)     # resident, not committed
    m.pw_set_commit(0, 1, 1, 6)
    assert m.pw_block_state(0, 1, 1) == (6, 8, 0)
    m.pw_reload_async(0, 1, 1, 5)                     # below resident: no-op
    assert m.pw_block_state(0, 1, 1)[2] == 0


def test_commit_errors():
    import any_precision_weight_gb300 as pw
    cfg = synth.CONFIGS["tiny"]
    bits = np.full((cfg.E, 2), 5, dtype=np.int32)
    m = gpu_layer(cfg, bits={0: bits}, alloc_planes=lambda e, k: 6)
    with pytest.raises(pw.PWError) as e:
        m.pw_set_commit(0, 0, 0, 6)                   # not resident, no reload
    assert e.value.code == pw.PW_ENOTRESIDENT
    with pytest.raises(pw.PWError) as e:
        m.pw_set_commit(0, 0, 0, 2)                   # below b_min
    assert e.value.code == pw.PW_EINVAL
    with pytest.raises(pw.PWError) as e:
        m.pw_reload_async(0, 0, 0, 7)                 # no page for plane 6
    assert e.value.code == pw.PW_EINVAL
    m.pw_reload_async(0, 0, 0, 6)
    with pytest.raises(pw.PWError) as e:
        m.pw_reload_async(0, 0, 0, 6)                 # one pending reload per block
    assert e.value.code == pw.PW_EINVAL
    with pytest.raises(pw.PWError) as e:
        m.pw_set_commit(0, 0, 0, 7)                   # above the pending target
    assert e.value.code == pw.PW_ENOTRESIDENT
    m.pw_set_commit(0, 0, 0, 6)
    assert m.pw_block_state(0, 0, 0) == (6, 6, 0)


def test_failed_reload_refuses_commit_and_keeps_q():
    import torch
    import any_precision_weight_gb300 as pw
    cfg = synth.CONFIGS["tiny"]
    bits = np.full((cfg.E, 2), 4, dtype=np.int32)
    m = gpu_layer(cfg, bits={0: bits})
    x = torch.from_numpy(synth.tokens(cfg)).cuda()
    L = torch.from_numpy(synth.logits(cfg)).cuda()
    before = _fwd(m, cfg, x, L)
    m.pw_debug_fail_next_reload()
    with pytest.raises(pw.PWError) as e:
        m.pw_reload_async(0, 2, 0, 6)
    assert e.value.code == pw.PW_ECUDA
    with pytest.raises(pw.PWError) as e:
        m.pw_reload_query(0, 2, 0)
    assert e.value.code == pw.PW_ERELOAD
    with pytest.raises(pw.PWError) as e:
        m.pw_set_commit(0, 2, 0, 6)
    assert e.value.code == pw.PW_ERELOAD
    assert m.pw_block_state(0, 2, 0)[0] == 4
    assert np.array_equal(_fwd(m, cfg, x, L).view(np.uint16), before.view(np.uint16))
    # a retry succeeds
    m.pw_reload_async(0, 2, 0, 6)
    m.pw_set_commit(0, 2, 0, 6)
    assert m.pw_block_state(0, 2, 0) == (6, 6, 0)


def test_small_stack_recommit_midrun_matches_oracle_per_layer():
    """Three stacked layers with the residual fused into the combine; some blocks
    are reloaded on a side stream and re-committed between two passes.  Every
    layer's output is checked against the oracle on the GPU's own input to that
    layer, before (old bits) and after (new bits)."""
    import torch
    cfg = synth.CONFIGS["tiny"].with_(T=4, n_layers=3)
    L = 3
    bits = {l: synth.block_bits(cfg, l) for l in range(L)}
    raised = {l: bits[l].copy() for l in range(L)}
    plan = []
    for l in range(L):
        for e in range(cfg.E):
            for k in range(2):
                if (e + k + l) % 3 == 0 and bits[l][e, k] < 8:
                    raised[l][e, k] = min(8, bits[l][e, k] + 2)
                    plan.append((l, e, k, int(raised[l][e, k])))
    m = gpu_layer(cfg, n_layers=L, bits=bits)
    Ls = [synth.logits(cfg, l) for l in range(L)]
    x0 = synth.tokens(cfg)

    def run():
        xs = [x0]
        x = torch.from_numpy(x0).cuda()
        for l in range(L):
            out = m.pw_moe_forward(l, x, torch.from_numpy(Ls[l]).cuda(), cfg.top_k, cfg.renorm, residual=x)
            xs.append(to_np(out))
            x = out
        torch.cuda.synchronize()
        return xs

    def check(xs, bb):
        for l in range(L):
            ref = omoe.layer(xs[l], Ls[l], cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, l), bb[l]),
                             residual=xs[l])
            assert_close(xs[l + 1], ref["out"])

    check(run(), bits)
    copy = torch.cuda.Stream()
    for (l, e, k, q) in plan:
        m.pw_reload_async(l, e, k, q, stream=copy)
    for (l, e, k, q) in plan:
        m.pw_set_commit(l, e, k, q)      # waits on the reload's event on the compute stream
    check(run(), raised)


def test_batched_reload_and_commit_match_per_block_calls():
    """pw_reload_many + pw_set_commit_many leave the same pages, descriptors and
    outputs as the per-block calls; a batch with one bad entry commits nothing."""
    import torch
    import any_precision_weight_gb300 as pw
    cfg = synth.CONFIGS["tiny"]
    lo = np.full((cfg.E, 2), 3, dtype=np.int32)
    lo[:, 1] = 5
    items = [(0, e, k, 8 if k == 0 else 7) for e in range(cfg.E) for k in range(2) if e % 2 == 0]
    a = gpu_layer(cfg, bits={0: lo})
    b = gpu_layer(cfg, bits={0: lo})
    x = torch.from_numpy(synth.tokens(cfg)).cuda()
    L = torch.from_numpy(synth.logits(cfg)).cuda()
    copy = torch.cuda.Stream()
    for (l, e, k, q) in items:
        a.pw_reload_async(l, e, k, q, stream=copy)
        a.pw_set_commit(l, e, k, q)
    assert b.pw_reload_many(items, stream=copy) == len(items)
    bad = items[:3] + [(0, 1, 0, 8)]            # expert 1 was not reloaded
    with pytest.raises(pw.PWError) as err:
        b.pw_set_commit_many(bad)
    assert err.value.code == pw.PW_ENOTRESIDENT
    for (l, e, k, q) in items:
        assert b.pw_block_state(l, e, k)[0] == lo[e, k]
    b.pw_set_commit_many(items)
    for e in range(cfg.E):
        for k in range(2):
            assert a.pw_block_state(0, e, k)[:2] == b.pw_block_state(0, e, k)[:2]
    assert np.array_equal(_fwd(a, cfg, x, L).view(np.uint16), _fwd(b, cfg, x, L).view(np.uint16))
    hi = lo.copy()
    for (l, e, k, q) in items:
        hi[e, k] = q
    ref = omoe.layer(to_np(x), to_np(L), cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), hi))
    assert_close(_fwd(b, cfg, x, L), ref["out"])


def test_commit_many_spans_several_launches():
    """More blocks than one descriptor-batch launch carries (192)."""
    import torch
    cfg = synth.CONFIGS["tiny"]
    L_ = 30
    bits = {l: np.full((cfg.E, 2), 4, dtype=np.int32) for l in range(L_)}
    m = gpu_layer(cfg, n_layers=L_, bits=bits)
    items = [(l, e, k, 3 + (l + e + k) % 2) for l in range(L_) for e in range(cfg.E) for k in range(2)]
    assert len(items) > 192
    m.pw_set_commit_many(items)
    torch.cuda.synchronize()
    x = torch.from_numpy(synth.tokens(cfg)).cuda()
    for l in (0, 17, 29):
        Lg = torch.from_numpy(synth.logits(cfg, l)).cuda()
        got = to_np(m.pw_moe_forward(l, x, Lg, cfg.top_k, cfg.renorm))
        want_bits = np.array([[3 + (l + e + k) % 2 for k in range(2)] for e in range(cfg.E)], dtype=np.int32)
        ref = omoe.layer(to_np(x), to_np(Lg), cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, l), want_bits))
        assert_close(got, ref["out"])
        for e in range(cfg.E):
            for k in range(2):
                assert m.pw_block_state(l, e, k)[0] == want_bits[e, k]


def test_planner_thread_reloads_while_decode_thread_commits():
    """A second host thread enqueues reloads (pw_reload_many, chunk by chunk)
    while this thread runs forward passes, polls and commits whatever has
    landed; afterwards every block is at its raised bitwidth and the layer
    matches the oracle there."""
    import threading
    import torch
    cfg = synth.CONFIGS["tiny"]
    L_ = 6
    bits = {l: np.full((cfg.E, 2), 3, dtype=np.int32) for l in range(L_)}
    m = gpu_layer(cfg, n_layers=L_, bits=bits)
    items = [(l, e, k, 5 + (e + k) % 4) for l in range(L_) for e in range(cfg.E) for k in range(2)]
    issued, errors = [], []
    copy = torch.cuda.Stream()

    def planner():
        try:
            for j in range(0, len(items), 7):
                m.pw_reload_many(items[j:j + 7], stream=copy)
                issued.extend(items[j:j + 7])
        except Exception as ex:
            errors.append(ex)

    x = torch.from_numpy(synth.tokens(cfg)).cuda()
    Ls = [torch.from_numpy(synth.logits(cfg, l)).cuda() for l in range(L_)]
    th = threading.Thread(target=planner)
    th.start()
    done = 0
    for it in range(100000):
        for l in range(L_):
            m.pw_moe_forward(l, x, Ls[l], cfg.top_k, cfg.renorm)
        j = done
        while j < len(issued) and m.pw_reload_query(*items[j][:3]) == 1:
            j += 1
        if j > done:
            m.pw_set_commit_many(items[done:j])
            done = j
        if done == len(items):
            break
    th.join()
    assert not errors
    assert done == len(items)
    torch.cuda.synchronize()
    for l in range(L_):
        want = np.array([[5 + (e + k) % 4 for k in range(2)] for e in range(cfg.E)], dtype=np.int32)
        got = to_np(m.pw_moe_forward(l, x, Ls[l], cfg.top_k, cfg.renorm))
        ref = omoe.layer(to_np(x), to_np(Ls[l]), cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, l), want))
        assert_close(got, ref["out"])


def test_mover_commits_landed_reloads_at_step_boundaries():
    """The native mover carries out submitted reloads with a small in-flight
    bound while forward passes run; pw_commit_arrived commits what has landed.
    Before the first commit the outputs are those of the old bits; at the end
    every block is at its target and each layer matches the oracle there."""
    import torch
    import any_precision_weight_gb300 as pw
    cfg = synth.CONFIGS["tiny"]
    L_ = 6
    bits = {l: np.full((cfg.E, 2), 3, dtype=np.int32) for l in range(L_)}
    m = gpu_layer(cfg, n_layers=L_, bits=bits)
    x = torch.from_numpy(synth.tokens(cfg)).cuda()
    Ls = [torch.from_numpy(synth.logits(cfg, l)).cuda() for l in range(L_)]
    before = [to_np(m.pw_moe_forward(l, x, Ls[l], cfg.top_k, cfg.renorm)) for l in range(L_)]
    last = (L_ - 1, cfg.E - 1, 1)
    items = [(l, e, k, 5 + (e + k) % 4) for l in range(L_) for e in range(cfg.E) for k in range(2)
             if (l, e, k) != last]
    items.append(last + (3,))                     # at the resident planes: committed without a copy
    with pytest.raises(pw.PWError):
        m.pw_mover_submit(items)                  # not started
    copy = torch.cuda.Stream()
    m.pw_mover_start(copy, max_inflight_bytes=256 << 10)
    with pytest.raises(pw.PWError) as err:
        m.pw_mover_submit([(0, 0, 0, 9)])         # q out of range: nothing queued
    assert err.value.code == pw.PW_EINVAL
    m.pw_mover_submit(items[:-1])
    m.pw_mover_submit(items[-1:])
    total, outstanding = 0, len(items)
    for it in range(200000):
        for l in range(L_):
            m.pw_moe_forward(l, x, Ls[l], cfg.top_k, cfg.renorm)
        c, outstanding = m.pw_commit_arrived()
        total += c
        if outstanding == 0:
            break
    assert outstanding == 0 and total == len(items)
    torch.cuda.synchronize()
    for l in range(L_):
        want = np.array([[5 + (e + k) % 4 for k in range(2)] for e in range(cfg.E)], dtype=np.int32)
        if l == last[0]:
            want[last[1], last[2]] = 3
        for e in range(cfg.E):
            for k in range(2):
                assert m.pw_block_state(l, e, k)[:2] == (want[e, k], want[e, k])
        got = to_np(m.pw_moe_forward(l, x, Ls[l], cfg.top_k, cfg.renorm))
        ref = omoe.layer(to_np(x), to_np(Ls[l]), cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, l), want))
        assert_close(got, ref["out"])
        assert not np.array_equal(got, before[l])
    with pytest.raises(pw.PWError):
        m.pw_mover_start(copy)                    # already running


def test_planner_plan_applied_to_a_stack():
    """pw_plan_bits on the table's blocks, then pw_plan_apply: lowering (and raising
    within resident planes) commits at once, raising above them goes through the
    mover; each layer then matches the oracle at the planned bits."""
    import torch
    import any_precision_weight_gb300 as pw
    from oracle import planner as oplan
    cfg = synth.CONFIGS["tiny"]
    L_ = 3
    start = {l: np.full((cfg.E, 2), 4, dtype=np.int32) for l in range(L_)}
    m = gpu_layer(cfg, n_layers=L_, bits=start, alloc_planes=lambda e, k: 8)
    nb = L_ * cfg.E * 2
    R = np.array([cfg.rows(i % 2) for i in range(nb)])
    K = np.array([cfg.cols(i % 2) for i in range(nb)])
    rng = np.random.default_rng(3)
    sens = rng.lognormal(0.0, 1.0, nb)
    mass = np.repeat(rng.dirichlet(np.ones(cfg.E), size=L_).reshape(-1), 2)
    full = sum(oplan.resident_bytes(int(r), int(k), 8, 3) for r, k in zip(R, K))
    x = torch.from_numpy(synth.tokens(cfg)).cuda()
    Ls = [torch.from_numpy(synth.logits(cfg, l)).cuda() for l in range(L_)]
    copy = torch.cuda.Stream()
    m.pw_mover_start(copy)

    def run_plan(frac):
        bits, _ = pw.pw_plan_bits(R, K, sens, mass, cfg.E, 1.0 / cfg.E, 6, frac * full)
        want, _ = oplan.plan_bits(list(R), list(K), list(sens), list(mass), cfg.E, 1.0 / cfg.E, 6, 3, 8,
                                  frac * full)
        assert np.array_equal(bits, want)
        now, moved = m.pw_plan_apply(bits.reshape(L_, cfg.E, 2))
        left = moved
        for _ in range(100000):
            if left == 0:
                break
            _, left = m.pw_commit_arrived()
        assert left == 0
        torch.cuda.synchronize()
        b3 = bits.reshape(L_, cfg.E, 2)
        for l in range(L_):
            for e in range(cfg.E):
                for k in range(2):
                    assert m.pw_block_state(l, e, k)[0] == b3[l, e, k]
            got = to_np(m.pw_moe_forward(l, x, Ls[l], cfg.top_k, cfg.renorm))
            ref = omoe.layer(to_np(x), to_np(Ls[l]), cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, l), b3[l]))
            assert_close(got, ref["out"])
        return now, moved

    now, moved = run_plan(0.7)      # from 4 bits everywhere: most blocks go up through the mover
    assert moved > 0
    now, moved = run_plan(0.45)     # lowering only: everything commits at once
    assert moved == 0 and now > 0
    now, moved = run_plan(0.7)      # back up: the planes are still resident, no copy needed
    assert moved == 0 and now > 0


def test_offload_release_and_reattach_round_trip():
    """Planes above the committed q leave the GPU (their pages are released and
    freed), the layer keeps matching the oracle at q; fresh pages are attached,
    the planes are reloaded from the host store and committed again."""
    import torch
    import any_precision_weight_gb300 as pw
    cfg = synth.CONFIGS["tiny"]
    bits = np.full((cfg.E, 2), 6, dtype=np.int32)
    m = gpu_layer(cfg, bits={0: bits}, per_plane=True)
    x = torch.from_numpy(synth.tokens(cfg)).cuda()
    L = torch.from_numpy(synth.logits(cfg)).cuda()
    D, HP, HO, MV = pw.PW_PLANE_DEVICE, pw.PW_PLANE_HOST_PAGED, pw.PW_PLANE_HOST, pw.PW_PLANE_MOVING
    assert m.pw_plane_states(0, 3, 0) == [D] * 6 + [HP] * 2
    with pytest.raises(pw.PWError):
        m.pw_block_release(0, 3, 0, 5)                  # below the committed q
    before = m.device_bytes()
    for e in range(cfg.E):
        rel = m.pw_block_release(0, e, 0, 6)
        assert all(r for r in rel[6:]) and not any(rel[:6])
    assert m.device_bytes() == before - cfg.E * 2 * cfg.rows(0) * cfg.cols(0) // 8
    assert m.pw_plane_states(0, 3, 0) == [D] * 6 + [HO] * 2
    with pytest.raises(pw.PWError) as err:
        m.pw_reload_async(0, 3, 0, 8)                   # no page for plane 6
    assert err.value.code == pw.PW_EINVAL
    ref6 = omoe.layer(to_np(x), to_np(L), cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), bits))
    assert_close(_fwd(m, cfg, x, L), ref6["out"])
    # back: fresh pages, reload, commit
    copy = torch.cuda.Stream()
    for e in range(cfg.E):
        m.pw_block_attach_pages(0, e, 0)
        assert m.pw_plane_states(0, e, 0) == [D] * 6 + [HP] * 2
        m.pw_reload_async(0, e, 0, 8, stream=copy)
        st = m.pw_plane_states(0, e, 0)
        assert st[:6] == [D] * 6 and all(s in (MV, D) for s in st[6:])
        with pytest.raises(pw.PWError):
            m.pw_block_release(0, e, 0, 6)              # a reload is pending
        m.pw_set_commit(0, e, 0, 8)
    hi = bits.copy()
    hi[:, 0] = 8
    ref8 = omoe.layer(to_np(x), to_np(L), cfg.top_k, cfg.renorm, oracle_blocks(SynthBlocks(cfg, 0), hi))
    assert_close(_fwd(m, cfg, x, L), ref8["out"])
    assert m.pw_plane_states(0, 3, 0) == [D] * 8
