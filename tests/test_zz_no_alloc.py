"""pw_moe_forward_noalloc, the forward for callers that cannot allocate device
memory (their runtime reserves all GPU memory up front, or their host only
hands over input and output buffers): it must give the same layer output as
pw_moe_forward with a caller workspace, call after call, although every call
reuses the library's one fixed scratch array.

Collected last on purpose, so that a run stopping at the first failure has
already run every other test."""
import numpy as np
import pytest

import synth

from _layers import assert_close, gpu_layer, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "qwen_decode"])
def test_noalloc_matches_workspace_forward_on_consecutive_calls(name):
    import torch
    cfg = synth.CONFIGS[name]
    m = gpu_layer(cfg)
    inputs = [(torch.from_numpy(synth.tokens(cfg, step=s)).cuda(),
               torch.from_numpy(synth.logits(cfg, step=s)).cuda()) for s in (11, 12)]
    refs = []
    for x, L in inputs:
        refs.append(to_np(m.pw_moe_forward(0, x, L, cfg.top_k, cfg.renorm)))
    torch.cuda.synchronize()
    # two calls in a row, different batches: the second must not see the first's leftovers
    for (x, L), ref in zip(inputs, refs):
        got = m.pw_moe_forward_noalloc(0, x, L, cfg.top_k, cfg.renorm)
        torch.cuda.synchronize()
        assert_close(to_np(got), ref.astype(np.float64))


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
