#!/usr/bin/env python
"""Throughput of the fused APL MoE layer (decode), one JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mixtral_decode_t4|mixtral_decode_t1|qwen_decode|tiny|
                                mixtral_prefill|qwen_stack]
                    [--per-config all|none|name,name]

A step is one pass of the whole hot path (routing, permutation, gate_up
dequant GEMV + SiLU*up, down dequant GEMV, combine) over one batch.  The
default workload is the largest single-GPU decode configuration: the
Mixtral-8x7B-shaped layer (hidden 4096, 8 experts, intermediate 14336, top-2,
batch 4, per-block bits in {3, 4, 5, 6, 8}).  Inputs are seeded synthetic
tensors resident in HBM.  Consecutive steps walk through ``--instances``
distinct layers of that shape (as a model walks its layers), so the weights a
step reads were last touched several hundred MB earlier and are not served
from the 129 MB L2.

Each timed step is one forward bracketed by CUDA events on its stream, so
steps do not overlap and every launch has its own duration: ``value`` and
``roofline`` come from the same region.  The back-to-back rate (forwards
overlapping through programmatic dependent launch) is reported beside it,
labelled.  ``per_q`` sweeps every block of the layer through uniform
bitwidths 3..8 (a commit, no reload).  ``per_config`` measures the other
workloads of the list the same way in the same run, each with its clocks.
The 24-layer stack replays each step as one CUDA graph and reloads a quarter
of its lower-bit blocks mid-run (tokens/s before, during and after each
reload window).

Multi-GPU (torchrun): the layer does not shard here, so every rank runs an
independent replica ("scaling": "weak"); value = all ranks' tokens / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused APL MoE layer decode tokens/s; weight-byte HBM GB/s vs GB300 peak"
FALLBACK_HBM = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixtral_decode_t4")
    ap.add_argument("--instances", type=int, default=0,
                    help="distinct layer instances cycled (default 8 for decode, 1 for prefill)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-q", action="store_true", help="skip the uniform-bitwidth sweep")
    ap.add_argument("--per-config", default="all",
                    help="other workloads measured into the same line: all, none, or a comma list")
    ap.add_argument("--uniform-bits", action="store_true",
                    help="every block at the byte-weighted mean bitwidth (mixed vs uniform check)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--reload-at", type=int, default=100, help="stack workload: step of the mid-run reload")
    ap.add_argument("--reload-inflight-mb", type=int, default=64,
                    help="stack workload: bound on the mover's copies in flight")
    ap.add_argument("--stack-reps", type=int, default=3, help="stack workload: reload windows measured")
    ap.add_argument("--read-store-first", action="store_true",
                    help="stack workload: copy the whole pinned host store to the GPU once before measuring "
                         "(checks whether the first reload window is slow because its host pages are read for "
                         "the first time)")
    ap.add_argument("--eager-steps", action="store_true",
                    help="stack workload: launch each step's 48 kernels from Python instead of one CUDA graph")
    ap.add_argument("--independent-logits", action="store_true",
                    help="stack workload: precomputed logits (lets consecutive layers overlap)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- distributed

def dist_init(n):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    """The maximum of v over all ranks (a host value: one small all-reduce)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks

class Clocks:
    """nvidia-smi samples of the SM clock and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = tempfile.mktemp(prefix="pw_clocks_", suffix=".csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.dev)], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
            time.sleep(1.0)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [s.strip() for s in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel, or
    None when there is none or the kernel sources changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"k_layer_{workload}.md")
    if kernel != "layer_fused" or not os.path.exists(path):
        return None
    txt = open(path).read()
    want = hashlib.sha256()
    for f in ("pw_decode.cu", "pw_route.cuh"):
        want.update(open(os.path.join(ROOT, "any_precision_weight_gb300", "csrc", f), "rb").read())
    fields = dict(l.split(":", 1) for l in txt.splitlines() if ":" in l and " " not in l.split(":", 1)[0])
    if fields.get("kernel_sources_sha256_16", "").strip() != want.hexdigest()[:16]:
        return None
    try:
        return int(fields["traffic_bytes_per_launch"].strip())
    except (KeyError, ValueError):
        return None


def tensor_peak():
    """Dense fp16/bf16 tensor peak (same rate on GB300): the measured burst figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(p))["bf16_tflops"]), "measured (bf16 burst; fp16 same rate)"
    except Exception:
        return 1900.0, "fallback"


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(p))["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM, "fallback"


# ----------------------------------------------------------------------------- workload

def uniform_bits(cfg, n_inst):
    """The byte-weighted mean committed bitwidth over the instances' blocks, rounded."""
    import numpy as np
    import synth
    num = den = 0.0
    for l in range(n_inst):
        b = synth.block_bits(cfg, l)
        for kind in (0, 1):
            w = cfg.rows(kind) * cfg.cols(kind)
            num += float(b[:, kind].sum()) * w
            den += b.shape[0] * w
    return int(np.floor(num / den + 0.5))


def build_model(cfg, n_inst, device, uniform=None):
    import numpy as np
    import any_precision_weight_gb300 as pw
    from any_precision_weight_gb300.model import load_expert_layer
    import synth
    m = pw.PagedMoE(n_inst, cfg.E, cfg.H, cfg.I, device=device)
    bits = {}
    for l in range(n_inst):
        bits[l] = synth.block_bits(cfg, l)
        if uniform is not None:
            bits[l] = np.full_like(bits[l], uniform)
        src = lambda e, k, l=l: (synth.parent_indices(cfg, l, e, k), synth.parent_lut(cfg, l, e, k))
        load_expert_layer(m, l, src, bits[l])
    return m, bits


def algorithmic_bytes(cfg, bits, counts):
    """Bytes each kernel must move at least, for one layer forward.

    gate_up: planes (q/8 byte per weight) + LUT_q of every active expert's
    gate_up block, its tokens' x rows, the h rows it writes;
    down: same for the down block, h rows read, fp32 y rows written;
    layer: both plus logits, out and the routing weights.
    """
    H, I, T, k, E = cfg.H, cfg.I, cfg.T, cfg.top_k, cfg.E
    gu = dn = 0
    for e in range(E):
        n = int(counts[e])
        if n == 0:
            continue
        qg, qd = int(bits[e][0]), int(bits[e][1])
        gu += 2 * I * H * qg // 8 + 2 * I * (1 << qg) * 2 + n * H * 2 + n * I * 2
        dn += H * I * qd // 8 + H * (1 << qd) * 2 + n * I * 2 + n * H * 4
    pairs = T * k
    layer = gu + dn + T * E * 4 + pairs * H * 4 + T * H * 2
    return {"gate_up": gu, "down": dn, "layer": layer}


# ----------------------------------------------------------------------------- CPU oracle

def oracle_rate(cfg, layer, seconds, sample_pairs=None):
    """Runs the fp64 oracle on one layer for about ``seconds``; returns
    (tokens/s, reps, seconds).  Input drawing is outside the timed part."""
    import numpy as np
    import synth
    from oracle import moe as omoe
    bits = synth.block_bits(cfg, layer)
    cache = {}

    def blocks(e):
        if e not in cache:
            cache[e] = tuple(omoe.Block(synth.parent_indices(cfg, layer, e, k), synth.parent_lut(cfg, layer, e, k),
                                        bits[e][k]) for k in (0, 1))
        return cache[e]
    x, L = synth.tokens(cfg), synth.logits(cfg, layer)
    omoe.layer(x, L, cfg.top_k, cfg.renorm, blocks)   # untimed: draws the inputs, builds tables
    t0 = time.perf_counter()
    reps = 0
    toks = 0.0
    while True:
        if sample_pairs is None:
            omoe.layer(x, L, cfg.top_k, cfg.renorm, blocks)
            toks += cfg.T
        else:
            t = reps % cfg.T
            omoe.layer(x, L, cfg.top_k, cfg.renorm, blocks, out_tokens=[t])
            toks += 1
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return toks / dt, reps, dt


def oracle_rate_one_thread(cfg, seconds):
    """oracle_rate in a child process whose BLAS and OpenMP pools have one thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json, sys; sys.path.insert(0, %r); import bench, synth; "
            "print(json.dumps(bench.oracle_rate(synth.CONFIGS[%r], 0, %r)))" % (ROOT, cfg.name, seconds))
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                             timeout=seconds * 4 + 120)
        rate, reps, dt = json.loads(out.stdout.strip().splitlines()[-1])
        return rate
    except Exception:
        return None


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


# ----------------------------------------------------------------------------- measurement

def commit_uniform(m, n_inst, q, stream=None):
    """Every block of every instance committed at q (all planes are resident)."""
    items = [(l, e, k, q) for l in range(n_inst) for e in range(m.E) for k in (0, 1)]
    for i in range(0, len(items), 4096):
        m.pw_set_commit_many(items[i:i + 4096], stream=stream)


def commit_bits(m, bits, stream=None):
    items = [(l, e, k, int(bits[l][e][k])) for l in bits for e in range(m.E) for k in (0, 1)]
    for i in range(0, len(items), 4096):
        m.pw_set_commit_many(items[i:i + 4096], stream=stream)


def timed_forwards(m, cfg, X, Lg, ws, out, n, start=0, serial=True):
    """n forwards cycling the instances.  serial: each forward's kernels are
    bracketed by CUDA events recorded on the launching stream
    (pw_profile_attach), so consecutive forwards do not overlap and every
    launch has its own duration; otherwise the forwards go back to back
    (programmatic dependent launch lets one forward's routing overlap the
    previous one's tail).  Returns (region ms, [per-forward event lists])."""
    import torch
    import any_precision_weight_gb300 as pw
    n_inst = len(X)
    stream = torch.cuda.current_stream()
    evs = []
    if serial:
        # the decode path is one kernel: an event before it and one right after it
        # (no other events between two forwards); the prefill path has four
        # kernels and five boundary events
        ne = 2 if is_fused(cfg) else 5
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(ne)] for _ in range(n)]
        for row in evs:              # torch creates the CUDA event at its first record
            for e in row:
                e.record(stream)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(n):
        l = (start + i) % n_inst
        if serial:
            pw.pw_profile_attach(evs[i] if len(evs[i]) == 5 else evs[i] + [None, None, None])
        m.pw_moe_forward(l, X[l], Lg[l], cfg.top_k, cfg.renorm, out=out, ws=ws)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1), evs


def kernel_times(cfg, evs):
    """Average ms per launch of each kernel from the per-forward events."""
    fused = is_fused(cfg)
    if fused:
        return {"layer_fused": sum(r[0].elapsed_time(r[1]) for r in evs) / len(evs)}
    names = ["route_permute", "gate_up", "down", "combine"]   # route_permute: routing + permutation launches
    return {nm: sum(r[j].elapsed_time(r[j + 1]) for r in evs) / len(evs) for j, nm in enumerate(names)}


def is_fused(cfg):
    return cfg.T <= 64 and cfg.T * cfg.top_k <= 256     # one persistent kernel per layer


def roofline(cfg, kms, byt_avg):
    """The dominant kernel against its roof: HBM bytes/s for the decode kernel,
    fp16 tensor FLOP/s for the prefill GEMMs.  Duration = the kernel's own
    CUDA-event time per launch."""
    if is_fused(cfg):
        peak, kind = hbm_peak()
        ms = kms["layer_fused"]
        b = byt_avg["layer"]
        a = b / (ms / 1e3) / 1e9
        return {"bound": "hbm", "kernel": "k_layer (whole decode layer, one launch)",
                "duration": "CUDA events around each launch, launches serialised", "ms_per_launch": ms,
                "achieved": a, "peak": peak, "unit": "GB/s", "frac": a / peak, "peak_kind": peak_kind_note(kind),
                "traffic": profiled_traffic("layer_fused", cfg.name), "bytes_per_launch": b}
    dom = max(("gate_up", "down"), key=lambda n: kms[n])
    P = cfg.T * cfg.top_k
    fl = {"gate_up": 2.0 * P * 2 * cfg.I * cfg.H, "down": 2.0 * P * cfg.H * cfg.I}[dom]
    peak, kind = tensor_peak()
    a = fl / (kms[dom] / 1e3) / 1e12
    return {"bound": "tensor", "kernel": f"k_prefill<{dom}>", "duration": "CUDA events around each launch",
            "ms_per_launch": kms[dom], "achieved": a, "peak": peak, "unit": "TFLOP/s", "frac": a / peak,
            "peak_kind": kind, "traffic": None, "flops_per_launch": fl}


def peak_kind_note(kind):
    return f"{kind} (HBM copy bandwidth, MEASURED_PEAKS.json)" if kind == "measured" else kind


def routed_bytes(m, cfg, X, Lg, ws, bits):
    """Algorithmic bytes of each instance's forward (its routing is fixed by its logits)."""
    import numpy as np
    import torch
    byt = []
    for l in range(len(X)):
        _, _, _, off, _ = m.pw_moe_forward(l, X[l], Lg[l], cfg.top_k, cfg.renorm, ws=ws, routing=True)
        counts = np.diff(off.cpu().numpy())
        byt.append(algorithmic_bytes(cfg, bits[l], counts))
    torch.cuda.synchronize()
    return byt


def avg_bytes(byt, n, start=0):
    keys = byt[0].keys()
    return {k: sum(byt[(start + i) % len(byt)][k] for i in range(n)) / n for k in keys}


def measure_layer(cfg, dev, local, steps, warmup, n_inst, world=1, uniform=None, per_q=False, e2e_steps=0,
                  overlapped=True):
    """Builds n_inst seeded layers of cfg and measures them.  Returns a dict:
    timed region (serialised forwards, per-launch events), roofline of the
    dominant kernel, the back-to-back step rate, optional host-buffer end to
    end rate and per-bitwidth sweep."""
    import torch
    import synth
    m, bits = build_model(cfg, n_inst, dev, uniform=uniform)
    X = [torch.from_numpy(synth.tokens(cfg, step=l)).to(dev) for l in range(n_inst)]
    Lg = [torch.from_numpy(synth.logits(cfg, l)).to(dev) for l in range(n_inst)]
    out = torch.empty((cfg.T, cfg.H), dtype=torch.float16, device=dev)
    ws = m.workspace(cfg.T, cfg.top_k)
    byt = routed_bytes(m, cfg, X, Lg, ws, bits)
    timed_forwards(m, cfg, X, Lg, ws, out, warmup, serial=False)
    res = {"workload": cfg.name, "instances": n_inst}

    clocks = Clocks(local)
    clocks.start()
    barrier(world)
    w0 = time.perf_counter()
    ms, evs = timed_forwards(m, cfg, X, Lg, ws, out, steps, serial=True)
    wall = time.perf_counter() - w0
    barrier(world)
    res["clocks"] = clocks.stop()
    res["region_ms"] = ms
    res["wall_s"] = wall
    res["ms_per_step"] = ms / steps
    res["tokens_per_s"] = cfg.T * steps / (ms / 1e3)
    kms = kernel_times(cfg, evs)
    res["kernel_ms"] = kms
    b = avg_bytes(byt, steps)
    res["layer_bytes_per_step"] = b["layer"]
    res["roofline"] = roofline(cfg, kms, b)
    if overlapped and is_fused(cfg):
        oms, _ = timed_forwards(m, cfg, X, Lg, ws, out, steps, serial=False)
        res["step_rate_overlapped"] = {
            "tokens_per_s": cfg.T * steps / (oms / 1e3), "ms_per_step": oms / steps,
            "note": "the same forwards back to back with no events between them: each forward routes its "
                    "batch while the previous one finishes (programmatic dependent launch), possible only "
                    "because the logits are ready in advance; in a model other layers sit between two MoE "
                    "layers, so this overlap is not counted in value or roofline"}
    if per_q and is_fused(cfg):
        # every plane of every block onto the device first (a reload from the
        # pinned host copies), so that any uniform bitwidth is one commit away
        items = [(l, e, k, 8) for l in range(n_inst) for e in range(cfg.E) for k in (0, 1)]
        copy = torch.cuda.Stream(device=dev)
        for i in range(0, len(items), 4096):
            m.pw_reload_many(items[i:i + 4096], stream=copy)
        copy.synchronize()
        sweep = {}
        for q in (3, 4, 5, 6, 7, 8):
            commit_uniform(m, n_inst, q)
            ubits = {l: [[q, q] for _ in range(cfg.E)] for l in range(n_inst)}
            ub = routed_bytes(m, cfg, X, Lg, ws, ubits)
            timed_forwards(m, cfg, X, Lg, ws, out, max(3, warmup), serial=False)
            n = max(50, min(steps, 200))
            qms, qevs = timed_forwards(m, cfg, X, Lg, ws, out, n, serial=True)
            kq = kernel_times(cfg, qevs)["layer_fused"]
            bq = avg_bytes(ub, n)["layer"]
            gbs = bq / (kq / 1e3) / 1e9
            sweep[str(q)] = {"ms_per_launch": kq, "bytes_per_launch": bq, "achieved_gbs": gbs,
                             "frac": gbs / hbm_peak()[0], "tokens_per_s": cfg.T / (kq / 1e3)}
        commit_bits(m, bits)
        torch.cuda.synchronize()
        res["per_q"] = sweep
    if e2e_steps:
        xh = [torch.from_numpy(synth.tokens(cfg, step=l)).pin_memory() for l in range(n_inst)]
        lh = [torch.from_numpy(synth.logits(cfg, l)).pin_memory() for l in range(n_inst)]
        oh = torch.empty((cfg.T, cfg.H), dtype=torch.float16).pin_memory()
        for i in range(min(10, e2e_steps)):
            m.pw_moe_forward_host(i % n_inst, xh[i % n_inst], lh[i % n_inst], cfg.top_k, cfg.renorm, oh, ws=ws)
        barrier(world)
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            l = i % n_inst
            m.pw_moe_forward_host(l, xh[l], lh[l], cfg.top_k, cfg.renorm, oh, ws=ws)
        res["e2e_s"] = max_over_ranks(time.perf_counter() - t0, world)
    res["bits"] = (f"uniform q={uniform} (byte-weighted mean of the mixed assignment)" if uniform is not None
                   else "per block from the config's set" + (", hot experts >= 6" if cfg.hot_bits else ""))
    del m, X, Lg, ws, out
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------- arms

def run_reference(args, cfg, rank, world):
    """The oracle, as it stands, on the host cores: full layer forwards of the
    same workload for a bounded time (0.03 s per requested step, 10..120 s)."""
    if rank != 0:
        return
    budget = min(120.0, max(10.0, 0.03 * (args.steps + args.warmup)))
    rate, reps, dt = oracle_rate(cfg, 0, budget)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / reps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "I": cfg.I, "top_k": cfg.top_k},
        "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{reps} full layer forwards (batch {cfg.T}) of layer instance 0 in "
                                   f"{dt:.1f} s, fp64 numpy; each a step"},
        "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


PER_CONFIG = ["tiny", "qwen_decode", "mixtral_decode_t1", "mixtral_decode_t4", "mixtral_prefill", "qwen_stack"]


def per_config_entries(args, head, dev, local, world):
    """Every other config of the workload list, each measured the same way on a
    short run (its own clocks), for the same JSON line."""
    import synth
    out = {}
    names = [n for n in PER_CONFIG if n != head] if args.per_config == "all" else \
        [n for n in args.per_config.split(",") if n and n != "none" and n != head]
    for name in names:
        cfg = synth.CONFIGS[name]
        t0 = time.perf_counter()
        try:
            if cfg.n_layers > 1:
                r = measure_stack(args, cfg, dev, local, world, steps=max(200, args.reload_at + 100))
                ent = {"workload": name, "ms_per_step": r["ms_per_step"], "tokens_per_s": r["tokens_per_s"],
                       "roofline": r["roofline"], "stack": r["stack"], "clocks": r["clocks"]}
            else:
                n_inst = 8 if is_fused(cfg) else 1
                steps = 200 if is_fused(cfg) else 5
                r = measure_layer(cfg, dev, local, steps, 5, n_inst, world=world)
                ent = {k: r[k] for k in ("workload", "ms_per_step", "tokens_per_s", "kernel_ms", "roofline",
                                         "clocks") if k in r}
                if "step_rate_overlapped" in r:
                    ent["step_rate_overlapped_tokens_per_s"] = r["step_rate_overlapped"]["tokens_per_s"]
                if not is_fused(cfg) or cfg.name == "tiny":
                    ent["l2"] = ("one layer instance; its 1.5 GB of planes exceed L2" if not is_fused(cfg)
                                 else "8 instances of 2 MB: L2-resident, a latency check")
        except Exception as ex:      # one config failing does not lose the others
            ent = {"workload": name, "error": f"{type(ex).__name__}: {ex}"}
        ent["setup_and_run_s"] = time.perf_counter() - t0
        out[name] = ent
    return out


def run_ours(args, cfg, rank, world, local):
    import torch

    dev = torch.device("cuda", local)
    n_inst = args.instances or (8 if is_fused(cfg) else 1)
    uq = uniform_bits(cfg, n_inst) if args.uniform_bits else None
    r = measure_layer(cfg, dev, local, args.steps, args.warmup, n_inst, world=world, uniform=uq,
                      per_q=not args.no_per_q, e2e_steps=min(args.steps, 1000))
    ms_max = max_over_ranks(r["region_ms"], world)
    value = world * cfg.T * args.steps / (ms_max / 1e3)
    e2e = world * cfg.T * min(args.steps, 1000) / r["e2e_s"]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, reps, dt = oracle_rate(cfg, 0, args.cpu_seconds)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
               "value_1_thread": oracle_rate_one_thread(cfg, min(10.0, args.cpu_seconds)),
               "sample": f"{reps} full layer forwards (batch {cfg.T}) of layer instance 0 in {dt:.1f} s, "
                         "fp64 numpy (BLAS matmuls threaded, gathers single-threaded)"}
    per = per_config_entries(args, cfg.name, dev, local, world) if args.per_config != "none" else None

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "I": cfg.I,
                   "top_k": cfg.top_k, "renorm": cfg.renorm, "bits": r["bits"],
                   "accumulate": "f32", "parallelism": f"replicas x{world}",
                   "l2": f"{n_inst} distinct layer instances cycled; inputs larger than L2 between reuses",
                   "timing": "each step one forward bracketed by CUDA events on its stream (no overlap "
                             "between steps)",
                   "layer_weight_bytes_per_step": r["layer_bytes_per_step"], "kernel_ms": r["kernel_ms"]},
        "roofline": r["roofline"],
        "step_rate_overlapped": r.get("step_rate_overlapped"),
        "per_q": r.get("per_q"),
        "cpu_baseline": cpu,
        "e2e": {"value": e2e, "unit": "tokens/s", "h2d_bytes_per_step": cfg.T * cfg.H * 2 + cfg.T * cfg.E * 4,
                "d2h_bytes_per_step": cfg.T * cfg.H * 2 + 4},
        "gpu_launches": (1 if is_fused(cfg) else 6) * args.steps,   # route, permute, gather, two GEMMs, combine
        "clocks": r["clocks"],
        "wall_s": r["wall_s"],
        "per_config": per,
    }
    print(json.dumps(line), flush=True)


def measure_stack(args, cfg, dev, local, world, steps):
    """24-layer Qwen-shaped stack, decode batch 4: bits fitted to 40% of the fp16
    bytes.  Each layer's logits are made by a small kernel that reads the
    previous layer's output (their values stay the config's seeded logits), so
    a layer's routing cannot start before the previous layer is done, as in a
    model.  At step reload_at a seeded 25% of the blocks below 8 bits start an
    asynchronous host->device reload of two more planes on a side stream
    (native mover), each committed (stream ordered) at the first step boundary
    after its copy completed.  The reload is run ``args.stack_reps`` times (the
    reloaded planes are released again in between); reports tokens/s before,
    during and after each window and the spread of the loss."""
    import numpy as np
    import torch
    import any_precision_weight_gb300 as pw
    from any_precision_weight_gb300.model import HostStore, load_expert_layer
    import synth

    L = cfg.n_layers
    bits = synth.stack_bits(cfg)
    plan = synth.reload_plan(cfg, bits)
    target = {(l, e, k): qn for (l, e, k, qo, qn) in plan}
    m = pw.PagedMoE(L, cfg.E, cfg.H, cfg.I, device=dev)
    store = HostStore()
    t_setup = time.perf_counter()
    for l in range(L):
        src = lambda e, k, l=l: (synth.parent_indices(cfg, l, e, k), synth.parent_lut(cfg, l, e, k))
        load_expert_layer(m, l, src, bits[l], store=store,
                          alloc_planes=lambda e, k, l=l: target.get((l, e, k), int(bits[l, e, k])))
    t_setup = time.perf_counter() - t_setup
    Lg = [torch.from_numpy(synth.logits(cfg, l)).to(dev) for l in range(L)]
    X0 = [torch.from_numpy(synth.tokens(cfg, step=i)).to(dev) for i in range(8)]
    bufs = [torch.empty((cfg.T, cfg.H), dtype=torch.float16, device=dev) for _ in range(2)]
    lbuf = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device=dev)
    ws = m.workspace(cfg.T, cfg.top_k)
    stream = torch.cuda.current_stream()
    copy = torch.cuda.Stream(device=dev)
    dependent = not args.independent_logits

    def step_body(i):
        x = X0[i % len(X0)]
        for l in range(L):
            o = bufs[l & 1]
            if dependent:
                # logits_l = seeded logits + 0 * (the previous layer's output): the values do not
                # change, but this kernel cannot run before that output exists
                torch.add(Lg[l], x[:, :cfg.E].float(), alpha=0.0, out=lbuf)
                lg = lbuf
            else:
                lg = Lg[l]
            m.pw_moe_forward(l, x, lg, cfg.top_k, cfg.renorm, residual=x, out=o, ws=ws)
            x = o

    bits_after = bits.copy()
    for (l, e, kind, qo, qn) in plan:
        bits_after[l, e, kind] = qn
    step_bytes = [0, 0]
    for l in range(L):
        _, _, _, off, _ = m.pw_moe_forward(l, X0[0], Lg[l], cfg.top_k, cfg.renorm, ws=ws, routing=True)
        counts = np.diff(off.cpu().numpy())
        step_bytes[0] += algorithmic_bytes(cfg, bits[l], counts)["layer"]
        step_bytes[1] += algorithmic_bytes(cfg, bits_after[l], counts)["layer"]
    reload_bytes = 0
    for (l, e, kind, qo, qn) in plan:
        R, K = m.rows_cols(kind)
        reload_bytes += (qn - qo) * R * K // 8 + R * 2 * sum(1 << b for b in range(qo + 1, qn + 1))
    items = [(l, e, kind, qn) for (l, e, kind, qo, qn) in plan]
    n = steps
    reload_at = min(args.reload_at, n - 1)
    m.pw_mover_start(copy, max_inflight_bytes=args.reload_inflight_mb << 20)
    for i in range(3):
        step_body(i)
    torch.cuda.synchronize()
    # One CUDA graph per token set holds a whole step (the 24 layers' logits
    # kernels and forwards), so a step costs the host one launch: with 48
    # launches from Python a step takes about 1 ms of host time against 1.4 ms
    # of GPU time, and the mover's copy calls during a reload window then make
    # the host, not the GPU, the bottleneck.  Commits stay outside the graphs
    # (the forwards read the descriptors when they run).
    graphs, launch_mode = [], "eager (48 launches per step from Python)"
    if not args.eager_steps:
        try:
            for j in range(len(X0)):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    step_body(j)
                graphs.append(g)
            torch.cuda.synchronize()
            launch_mode = "one CUDA graph per step"
        except Exception as ex:   # capture refused: measure the eager loop
            graphs, launch_mode = [], f"eager (graph capture failed: {str(ex)[:120]})"
            torch.cuda.synchronize()

    def step(i):
        if graphs:
            graphs[i % len(graphs)].replay()
        else:
            step_body(i)
    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    # host->device rate of plain copies from the pinned store on the copy stream:
    # the last chunk (the last layers' planes) twice in a row (its pages first
    # untouched by the GPU since packing, then just read), then the same copy
    # while the decode steps run
    probe = {}
    chunk = store._chunks[-1]
    dbuf = torch.empty(chunk.numel(), dtype=torch.uint8, device=dev)
    for name in ("first", "again"):
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(copy)
        with torch.cuda.stream(copy):
            dbuf.copy_(chunk, non_blocking=True)
        p1.record(copy)
        p1.synchronize()
        probe[f"h2d_{name}_gbs"] = chunk.numel() / (p0.elapsed_time(p1) / 1e3) / 1e9
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(copy)
    with torch.cuda.stream(copy):
        dbuf.copy_(chunk, non_blocking=True)
    p1.record(copy)
    k = 0
    while not p1.query() and k < 1000:
        step(k)
        k += 1
    p1.synchronize()
    probe["h2d_beside_decode_gbs"] = chunk.numel() / (p0.elapsed_time(p1) / 1e3) / 1e9
    probe["probe_bytes"] = chunk.numel()
    torch.cuda.synchronize()
    try:
        probe["host_page_bytes"] = os.sysconf("SC_PAGE_SIZE")
        probe["thp"] = open("/sys/kernel/mm/transparent_hugepage/enabled").read().strip()
    except Exception:
        pass
    if args.read_store_first:
        t_rd = time.perf_counter()
        for c in store._chunks:
            dbuf[:c.numel()].copy_(c, non_blocking=True)
        torch.cuda.synchronize()
        probe["store_read_first_gbs"] = store.nbytes() / (time.perf_counter() - t_rd) / 1e9
    del dbuf
    clocks = Clocks(local)
    clocks.start()
    reps = []
    released = {}
    for rep in range(args.stack_reps):
        if rep:
            # back to the fitted bits, the reloaded planes offloaded again (their pages
            # re-attached empty), so the next window copies the same bytes
            m.pw_set_commit_many([(l, e, k, qo) for (l, e, k, qo, qn) in plan])
            torch.cuda.synchronize()
            for (l, e, k, qo, qn) in plan:
                rel = m.pw_block_release(l, e, k, qo)
                ptrs = (pw._vp * pw.MAX_BITS)(*[rel[p] for p in range(pw.MAX_BITS)])
                pw._check(pw.lib().pw_block_attach_pages(m._t, l, e, k, ptrs), "pw_block_attach_pages")
            for i in range(3):
                step(i)
            torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        for e_ in ev + [c0, c1]:          # torch creates the CUDA event at its first record
            e_.record(stream)
        torch.cuda.synchronize()
        committed = 0
        commit_launches = 0
        last = reload_at
        landed = False
        w0 = time.perf_counter()
        ev[0].record(stream)
        enq = np.zeros(n)                    # host seconds spent enqueueing each step
        for i in range(n):
            if i >= 2:
                ev[i - 1].synchronize()      # at most two steps in flight, as a decode loop that
                                             # needs step i-2's tokens before launching step i
            h0 = time.perf_counter()
            if i == reload_at:
                c0.record(copy)
                m.pw_mover_submit(items)
            if i >= reload_at and committed < len(items):
                c, left = m.pw_commit_arrived()
                if c:
                    committed += c
                    commit_launches += -(-c // 192)
                    last = i
                if left == 0:
                    c1.record(stream)        # the boundary at which the last block was committed
                    landed = True
            step(3 + i)
            ev[i + 1].record(stream)
            enq[i] = time.perf_counter() - h0
        torch.cuda.synchronize()
        wall = time.perf_counter() - w0
        # a window longer than the run: its remaining blocks committed untimed,
        # so that the next window starts from the same state
        t_drain = time.perf_counter()
        while committed < len(items):
            c, left = m.pw_commit_arrived()
            committed += c
            if left == 0 and committed >= len(items):
                break
            if time.perf_counter() - t_drain > 120:
                raise RuntimeError("stack reload did not complete within 120 s")
            time.sleep(0.001)
        torch.cuda.synchronize()
        t = np.array([ev[i].elapsed_time(ev[i + 1]) for i in range(n)])
        copy_ms = c0.elapsed_time(c1) if landed else None
        before, during, after = t[:reload_at], t[reload_at:last + 1], t[last + 1:]
        tps = lambda a: float(cfg.T / (a.mean() / 1e3)) if len(a) else None
        reps.append({
            "tokens_per_s_before": tps(before), "tokens_per_s_during": tps(during),
            "tokens_per_s_after": tps(after),
            "loss_pct_during": (1 - tps(during) / tps(before)) * 100 if len(during) and len(before) else None,
            "last_commit_step": last, "committed": committed, "window_within_run": landed,
            "submit_to_last_commit_ms": copy_ms,
            "reload_gbs": reload_bytes / (copy_ms / 1e3) / 1e9 if copy_ms else None,
            "ms_total": float(t.sum()), "before_ms_per_step": float(before.mean()) if len(before) else None,
            "after_ms_per_step": float(after.mean()) if len(after) else None,
            "commit_launches": commit_launches, "wall_s": wall,
            "host_enqueue_ms_before": float(enq[:reload_at].mean() * 1e3),
            "host_enqueue_ms_during": float(enq[reload_at:last + 1].mean() * 1e3)})
    clk = clocks.stop()
    losses = [r["loss_pct_during"] for r in reps if r["loss_pct_during"] is not None]
    gbs = [r["reload_gbs"] for r in reps if r["reload_gbs"]]
    before_ms = float(np.mean([r["before_ms_per_step"] for r in reps]))
    after_ms = [r["after_ms_per_step"] for r in reps if r["after_ms_per_step"]]
    res = {
        "ms_per_step": float(np.mean([r["ms_total"] for r in reps])) / n,
        "tokens_per_s": cfg.T * n * len(reps) / (sum(r["ms_total"] for r in reps) / 1e3),
        "clocks": clk, "setup_s": t_setup, "steps": n, "reps": len(reps),
        "gpu_launches": n * L * (2 if dependent else 1) * len(reps) + sum(r["commit_launches"] for r in reps),
        "stack": {"logits": "from a kernel reading the previous layer's output" if dependent
                            else "precomputed (the forwards may overlap)",
                  "reload_at_step": reload_at, "reloaded_blocks": len(plan), "reload_bytes": reload_bytes,
                  "mover": f"native mover thread, at most {args.reload_inflight_mb} MiB of copies in flight",
                  "step_launch": launch_mode,
                  "loss_pct_during_mean": float(np.mean(losses)) if losses else None,
                  "loss_pct_first_window": losses[0] if losses else None,
                  "loss_pct_later_windows_mean": float(np.mean(losses[1:])) if len(losses) > 1 else None,
                  "loss_pct_during_min": float(np.min(losses)) if losses else None,
                  "loss_pct_during_max": float(np.max(losses)) if losses else None,
                  "reload_gbs_mean": float(np.mean(gbs)) if gbs else None,
                  "reload_gbs_min": float(np.min(gbs)) if gbs else None,
                  "reload_gbs_max": float(np.max(gbs)) if gbs else None,
                  "copy_probe": probe, "runs": reps},
        "roofline": {"bound": "hbm", "kernel": "k_layer (whole step of 24 layers)",
                     "duration": "CUDA events around each step",
                     "achieved": step_bytes[0] / (before_ms / 1e3) / 1e9,
                     "peak": hbm_peak()[0], "unit": "GB/s", "peak_kind": peak_kind_note(hbm_peak()[1]),
                     "traffic": None, "bytes_per_step_before": step_bytes[0],
                     "bytes_per_step_after": step_bytes[1],
                     "achieved_after": step_bytes[1] / (float(np.mean(after_ms)) / 1e3) / 1e9 if after_ms else None},
    }
    res["roofline"]["frac"] = res["roofline"]["achieved"] / res["roofline"]["peak"]
    m.close()
    del m, store, ws
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_stack(args, cfg, rank, world, local):
    import torch
    dev = torch.device("cuda", local)
    r = measure_stack(args, cfg, dev, local, world, steps=args.steps)
    ms_max = max_over_ranks(r["ms_per_step"] * r["steps"], world)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": world * cfg.T * r["steps"] / (ms_max / 1e3), "unit": "tokens/s",
        "n_gpus": world, "steps": r["steps"], "warmup": args.warmup, "ms_per_step": ms_max / r["steps"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": cfg.name, "layers": cfg.n_layers, "T": cfg.T, "H": cfg.H, "E": cfg.E, "I": cfg.I,
                   "top_k": cfg.top_k, "bits": "greedy fit to 40% of fp16 bytes",
                   "l2": "24 layers of weights (about 10 GB) between reuses, larger than L2"},
        "stack": r["stack"], "roofline": r["roofline"], "gpu_launches": r["gpu_launches"],
        "clocks": r["clocks"], "setup_s": r["setup_s"],
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    import synth
    cfg = synth.CONFIGS[args.workload]
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, cfg, rank, int(os.environ.get("WORLD_SIZE", "1")))
        return
    rank, world, local = dist_init(args.gpus)
    if cfg.n_layers > 1:
        run_stack(args, cfg, rank, world, local)
    else:
        run_ours(args, cfg, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
