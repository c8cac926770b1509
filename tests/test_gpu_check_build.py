"""The PW_CHECK build (libpw_check.so: the same kernels with device-side bounds
checks that report PW_STATUS_BOUNDS instead of trapping) on the decode path,
the K-split down items and the tensor-core path: no check fires, and the
outputs equal the normal build's bit for bit.  Runs the check build in a
child process (a process loads one of the two libraries)."""
import os
import subprocess
import sys

import numpy as np
import pytest

import synth

from _layers import gpu_layer, to_np

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CASES = [("tiny", {}), ("qwen_decode", {}), ("tiny", {"H": 256, "I": 6144, "T": 5}), ("tiny", {"T": 300})]

CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, ROOT); sys.path.insert(0, ROOT + "/tests")
import synth
import any_precision_weight_gb300 as pw
from _layers import gpu_layer, to_np
out = {}
for i, (name, kw) in enumerate(CASES):
    cfg = synth.CONFIGS[name].with_(**kw)
    m = gpu_layer(cfg)
    ws = m.workspace(cfg.T, cfg.top_k)
    o = m.pw_moe_forward(0, torch.from_numpy(synth.tokens(cfg, step=5)).cuda(),
                         torch.from_numpy(synth.logits(cfg, step=5)).cuda(), cfg.top_k, cfg.renorm, ws=ws)
    torch.cuda.synchronize()
    out[f"out{i}"] = to_np(o).view(np.uint16)
    out[f"status{i}"] = np.array([m.workspace_status(ws)])
np.savez(PATH, **out)
"""


def _forward(cfg):
    import torch
    m = gpu_layer(cfg)
    o = m.pw_moe_forward(0, torch.from_numpy(synth.tokens(cfg, step=5)).cuda(),
                         torch.from_numpy(synth.logits(cfg, step=5)).cuda(), cfg.top_k, cfg.renorm)
    torch.cuda.synchronize()
    return to_np(o).view(np.uint16)


def test_check_build_agrees_and_reports_nothing(tmp_path):
    import any_precision_weight_gb300 as pw
    path = str(tmp_path / "check.npz")
    code = f"ROOT = {ROOT!r}\nCASES = {CASES!r}\nPATH = {path!r}\n" + CHILD
    env = dict(os.environ, PW_CHECK="1")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    got = np.load(path)
    for i, (name, kw) in enumerate(CASES):
        cfg = synth.CONFIGS[name].with_(**kw)
        assert int(got[f"status{i}"][0]) & pw.PW_STATUS_BOUNDS == 0, (name, kw)
        assert int(got[f"status{i}"][0]) == 0, (name, kw)
        assert np.array_equal(got[f"out{i}"], _forward(cfg)), (name, kw)
