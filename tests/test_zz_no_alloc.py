"""pw_moe_forward_noalloc, the forward for callers that cannot allocate device
memory (their runtime reserves all GPU memory up front, or their host only
hands over input and output buffers): it must give exactly the layer output
of pw_moe_forward with a caller workspace (the forward is deterministic, so
bit for bit), call after call, although every call reuses the library's one
fixed scratch array and finds there whatever the previous call left.

Collected last on purpose, so that a run stopping at the first failure has
already run every other test."""
import numpy as np
import pytest

import synth
from oracle import moe as omoe

from _layers import SynthBlocks, assert_close, gpu_layer, oracle_blocks, to_np

pytestmark = pytest.mark.gpu


def _same(a, b):
    import torch
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "qwen_decode"])
def test_noalloc_matches_workspace_forward_on_consecutive_calls(name):
    import torch
    cfg = synth.CONFIGS[name]
    m = gpu_layer(cfg)
    inputs = [(torch.from_numpy(synth.tokens(cfg, step=s)).cuda(),
               torch.from_numpy(synth.logits(cfg, step=s)).cuda()) for s in (11, 12)]
    refs = []
    for x, L in inputs:
        refs.append(m.pw_moe_forward(0, x, L, cfg.top_k, cfg.renorm).clone())
    torch.cuda.synchronize()
    want = omoe.layer(synth.tokens(cfg, step=11), synth.logits(cfg, step=11), cfg.top_k, cfg.renorm,
                      oracle_blocks(SynthBlocks(cfg, 0), synth.block_bits(cfg)))
    assert_close(to_np(refs[0]), want["out"])
    # two calls in a row, different batches: the second must not see the first's leftovers
    for (x, L), ref in zip(inputs, refs):
        got = m.pw_moe_forward_noalloc(0, x, L, cfg.top_k, cfg.renorm)
        torch.cuda.synchronize()
        assert _same(got, ref)
        assert m.noalloc_status() == 0


def test_noalloc_alternating_shapes_and_paths():
    """Tensor-core path (300 tokens), decode path (16 tokens) and another table's
    shapes, one after the other on the shared scratch; each against a forward on
    a fresh workspace of its own."""
    import torch
    tiny = synth.CONFIGS["tiny"]
    big = tiny.with_(T=300)
    qwen = synth.CONFIGS["qwen_decode"]
    mt = gpu_layer(tiny)
    mq = gpu_layer(qwen)
    runs = [(mt, big, 21), (mt, tiny, 22), (mq, qwen, 23), (mt, big, 24), (mq, qwen, 25), (mt, tiny, 26)]
    for m, cfg, step in runs:
        x = torch.from_numpy(synth.tokens(cfg, step=step)).cuda()
        L = torch.from_numpy(synth.logits(cfg, step=step)).cuda()
        ref = m.pw_moe_forward(0, x, L, cfg.top_k, cfg.renorm, ws=m.workspace(cfg.T, cfg.top_k)).clone()
        got = m.pw_moe_forward_noalloc(0, x, L, cfg.top_k, cfg.renorm)
        torch.cuda.synchronize()
        assert _same(got, ref), (cfg.name, cfg.T, step)
        assert m.noalloc_status() == 0


def test_noalloc_reports_device_status():
    import torch
    import any_precision_weight_gb300 as pw
    cfg = synth.CONFIGS["tiny"]
    m = gpu_layer(cfg)
    x = torch.from_numpy(synth.tokens(cfg)).cuda()
    L = synth.logits(cfg)
    L[2, 5] = np.nan
    m.pw_moe_forward_noalloc(0, x, torch.from_numpy(L).cuda(), cfg.top_k, cfg.renorm)
    assert m.noalloc_status() & pw.PW_STATUS_NAN_LOGIT
    L[2, 5] = 0.0
    m.pw_moe_forward_noalloc(0, x, torch.from_numpy(L).cuda(), cfg.top_k, cfg.renorm)
    assert m.noalloc_status() == 0


def test_noalloc_rejects_batches_beyond_its_scratch():
    import torch
    import any_precision_weight_gb300 as pw
    cfg = synth.CONFIGS["tiny"]
    m = gpu_layer(cfg)
    T = 4096                                   # needs far more than the 8 MiB reserved
    x = torch.zeros((T, cfg.H), dtype=torch.float16, device="cuda")
    L = torch.zeros((T, cfg.E), dtype=torch.float32, device="cuda")
    with pytest.raises(pw.PWError) as e:
        m.pw_moe_forward_noalloc(0, x, L, cfg.top_k, cfg.renorm)
    assert e.value.code == pw.PW_ENOMEM
    assert "8388608" in str(e.value)
