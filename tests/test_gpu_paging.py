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
