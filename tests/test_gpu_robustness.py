"""The decode forward against what its caller may hand it: workspaces holding
anything (fresh memory, another forward's leftovers, adversarial patterns),
and a GPU of which another kernel holds half the SMs while the forward runs.
In every case the output must equal the forward on a zeroed workspace bit for
bit (the forward is deterministic) and the oracle within tolerance, with no
status bit raised."""
import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import synth
from oracle import moe as omoe

from _layers import SynthBlocks, assert_close, gpu_layer, oracle_blocks, to_np

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _inputs(cfg, step=0):
    import torch
    return (torch.from_numpy(synth.tokens(cfg, step=step)).cuda(),
            torch.from_numpy(synth.logits(cfg, step=step)).cuda())


def _fills(nbytes, stale):
    """name -> uint8 numpy array of nbytes: the contents a fresh workspace gets."""
    rng = np.random.default_rng(1234)
    n4 = nbytes // 4
    out = {
        "zeros": np.zeros(nbytes, np.uint8),
        "ones": np.full(nbytes, 0xFF, np.uint8),
        "iota_0_4096": (np.arange(n4, dtype=np.int64) % 4097).astype(np.int32).view(np.uint8),
        "small_counters_1_64": (np.arange(n4, dtype=np.int64) % 64 + 1).astype(np.int32).view(np.uint8),
        "random_bytes": rng.integers(0, 256, size=nbytes, dtype=np.uint8),
        "stale_forward": stale[:nbytes].copy(),
    }
    # every 8-byte word = a ticket word an earlier forward left behind (top byte 0xA5)
    w8 = stale[: (len(stale) // 8) * 8].view(np.uint64)
    tagged = w8[(w8 >> np.uint64(56)) == np.uint64(0xA5)]
    assert len(tagged) >= 1
    out["earlier_ticket_words"] = np.resize(tagged, nbytes // 8).astype(np.uint64).view(np.uint8)
    return out


@pytest.mark.parametrize("name", ["tiny", "qwen_decode"])
def test_forward_ignores_whatever_the_workspace_holds(name):
    import torch
    cfg = synth.CONFIGS[name]
    m = gpu_layer(cfg)
    x, L = _inputs(cfg, 3)
    ws0 = m.workspace(cfg.T, cfg.top_k)
    ws0.zero_()
    ref = m.pw_moe_forward(0, x, L, cfg.top_k, cfg.renorm, ws=ws0).clone()
    torch.cuda.synchronize()
    assert m.workspace_status(ws0) == 0
    want = omoe.layer(synth.tokens(cfg, step=3), synth.logits(cfg, step=3), cfg.top_k, cfg.renorm,
                      oracle_blocks(SynthBlocks(cfg, 0), synth.block_bits(cfg)))
    assert_close(to_np(ref), want["out"])
    # a workspace a forward of another batch size used (its sections sit elsewhere)
    big = 64
    wsb = m.workspace(big, cfg.top_k)
    xb = torch.from_numpy(synth.tokens(cfg, step=5, T=big)).cuda()
    Lb = torch.from_numpy(synth.logits(cfg, step=5, T=big)).cuda()
    m.pw_moe_forward(0, xb, Lb, cfg.top_k, cfg.renorm, ws=wsb)
    m.pw_moe_forward(0, x, L, cfg.top_k, cfg.renorm, ws=wsb)
    torch.cuda.synchronize()
    stale = wsb.cpu().numpy()
    for fill, data in _fills(ws0.numel(), stale).items():
        ws = torch.from_numpy(data).cuda()
        got = m.pw_moe_forward(0, x, L, cfg.top_k, cfg.renorm, ws=ws)
        torch.cuda.synchronize()
        assert m.workspace_status(ws) == 0, fill
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), fill
        # and again on the same workspace: the first forward's leftovers
        got2 = m.pw_moe_forward(0, x, L, cfg.top_k, cfg.renorm, ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(got2.view(torch.int16), ref.view(torch.int16)), fill


def _occupier():
    src = os.path.join(HERE, "gpu_occupy.cu")
    so = os.path.join(tempfile.mkdtemp(prefix="pw_occupy_"), "occupy.so")
    nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    subprocess.run([nvcc, "-shared", "-Xcompiler", "-fPIC", "-gencode", "arch=compute_103a,code=sm_103a",
                    src, "-o", so], check=True, capture_output=True)
    lib = ctypes.CDLL(so)
    lib.occupy.restype = ctypes.c_int
    lib.occupy.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_ulonglong, ctypes.c_void_p, ctypes.c_void_p]
    return lib


@pytest.mark.parametrize("name", ["tiny", "qwen_decode"])
def test_forward_beside_a_kernel_holding_half_the_sms(name):
    """Another stream's kernel holds half the SMs for 0.6 s, longer than any
    device-side wait of the forward (about 0.3 s): the forward's CTAs on the
    free SMs must finish the layer themselves, correctly."""
    import torch
    cfg = synth.CONFIGS[name]
    m = gpu_layer(cfg)
    x, L = _inputs(cfg, 4)
    ref = m.pw_moe_forward(0, x, L, cfg.top_k, cfg.renorm).clone()
    torch.cuda.synchronize()
    occ = _occupier()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    done = torch.zeros(1, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    ws = m.workspace(cfg.T, cfg.top_k)
    for rep in range(2):
        with torch.cuda.stream(side):
            assert occ.occupy(sms // 2, 120 * 1024, 600_000_000, done.data_ptr(), side.cuda_stream) == 0
        torch.cuda._sleep(2_000_000)     # let the holder's CTAs land before the forward is launched
        got = m.pw_moe_forward(0, x, L, cfg.top_k, cfg.renorm, ws=ws)
        torch.cuda.synchronize()
        assert int(done.item()) == (rep + 1) * (sms // 2)
        assert m.workspace_status(ws) == 0
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "qwen_decode"])
def test_graph_replays_of_one_forward(name):
    """One decode forward captured in a CUDA graph and replayed four times in a
    row on the same workspace (every replay carries the tag of the capture):
    each replay equals an eager forward bit for bit, with no status bit."""
    import torch
    cfg = synth.CONFIGS[name]
    m = gpu_layer(cfg)
    x, L = _inputs(cfg, step=31)
    ws = m.workspace(cfg.T, cfg.top_k)
    ref = m.pw_moe_forward(0, x, L, cfg.top_k, cfg.renorm, ws=ws).clone()
    out = torch.empty_like(x)
    m.pw_moe_forward(0, x, L, cfg.top_k, cfg.renorm, out=out, ws=ws)   # warm the launch path
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        m.pw_moe_forward(0, x, L, cfg.top_k, cfg.renorm, out=out, ws=ws)
    for _ in range(4):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert m.workspace_status(ws) == 0
