#!/usr/bin/env python
"""Throughput of the fused APL MoE layer (decode), one JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload qwen_decode|mixtral_decode_t1|mixtral_decode_t4|tiny]

A step is one pass of the whole hot path (routing, permutation, gate_up
dequant GEMV + SiLU*up, down dequant GEMV, combine) over one decode batch of
the Qwen1.5-MoE-A2.7B-shaped layer (hidden 2048, 60 experts, intermediate
1408, top-4, batch 4, per-block bits in {3..8}, hot experts >= 6).  Inputs are
seeded synthetic tensors resident in HBM.  Consecutive steps walk through
``--instances`` distinct layers of that shape (as a model walks its layers),
so the weights a step reads were last touched several hundred MB earlier and
are not served from the 129 MB L2.

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
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen_decode")
    ap.add_argument("--instances", type=int, default=0,
                    help="distinct layer instances cycled (default 8 for decode, 1 for prefill)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--uniform-bits", action="store_true",
                    help="every block at the byte-weighted mean bitwidth (mixed vs uniform check)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--reload-at", type=int, default=100, help="stack workload: step of the mid-run reload")
    ap.add_argument("--reload-inflight-mb", type=int, default=64,
                    help="stack workload: bound on the mover's copies in flight")
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


def run_ours(args, cfg, rank, world, local):
    import numpy as np
    import torch
    import any_precision_weight_gb300 as pw
    import synth

    dev = torch.device("cuda", local)
    n_inst = args.instances or (8 if cfg.T <= 64 else 1)
    uq = uniform_bits(cfg, n_inst) if args.uniform_bits else None
    m, bits = build_model(cfg, n_inst, dev, uniform=uq)
    X = [torch.from_numpy(synth.tokens(cfg, step=l)).to(dev) for l in range(n_inst)]
    Lg = [torch.from_numpy(synth.logits(cfg, l)).to(dev) for l in range(n_inst)]
    out = torch.empty((cfg.T, cfg.H), dtype=torch.float16, device=dev)
    ws = m.workspace(cfg.T, cfg.top_k)
    stream = torch.cuda.current_stream()

    # routing of each instance (fixed logits): algorithmic bytes per step
    byt = []
    for l in range(n_inst):
        _, _, _, off, _ = m.pw_moe_forward(l, X[l], Lg[l], cfg.top_k, cfg.renorm, ws=ws, routing=True)
        counts = np.diff(off.cpu().numpy())
        byt.append(algorithmic_bytes(cfg, bits[l], counts))
    torch.cuda.synchronize()

    def step(i):
        l = i % n_inst
        m.pw_moe_forward(l, X[l], Lg[l], cfg.top_k, cfg.renorm, out=out, ws=ws)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    clocks = Clocks(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - w0
    barrier(world)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    ms_max = max_over_ranks(ms, world)
    value = world * cfg.T * args.steps / (ms_max / 1e3)

    # per-kernel boundary events over a second region of the same steps
    kn = min(args.steps, 2000)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(kn)]
    for row in evs:                 # torch creates the CUDA event at its first record
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(kn):
        pw.pw_profile_attach(evs[i])
        step(i)
    torch.cuda.synchronize()
    fused = cfg.T <= 64 and cfg.T * cfg.top_k <= 256     # one persistent kernel per layer
    if fused:
        names = ["layer_fused"]
        tot = {"layer_fused": sum(evs[i][0].elapsed_time(evs[i][4]) for i in range(kn))}
        dom = "layer_fused"
    else:
        names = ["route_permute", "gate_up", "down", "combine"]
        tot = {n: 0.0 for n in names}
        for i in range(kn):
            for j, n in enumerate(names):
                tot[n] += evs[i][j].elapsed_time(evs[i][j + 1])
        dom = max(("gate_up", "down"), key=lambda n: tot[n])
    avg_ms = {n: tot[n] / kn for n in names}
    key = "layer" if fused else dom
    dom_bytes = sum(byt[i % n_inst][key] for i in range(kn)) / kn
    achieved = dom_bytes / (avg_ms[dom] / 1e3) / 1e9
    duration = "CUDA events around each launch"
    if fused:
        # one launch per step and nothing else on the stream: the launch's average
        # duration in the timed region is the step time (consecutive launches overlap
        # the next one's routing with this one's tail; events between launches, as in
        # the per-kernel pass above, would serialise them)
        dom_bytes = sum(byt[i % n_inst]["layer"] for i in range(args.steps)) / args.steps
        achieved = dom_bytes / (ms / args.steps / 1e3) / 1e9
        duration = "timed region / launches (one launch per step)"
    peak, peak_kind = hbm_peak()
    bound, unit = "hbm", "GB/s"
    if not fused:
        # tensor-core GEMM path: roofline on fp16 FLOP/s of the dominant kernel
        P = cfg.T * cfg.top_k
        fl = {"gate_up": 2.0 * P * 2 * cfg.I * cfg.H, "down": 2.0 * P * cfg.H * cfg.I}[dom]
        achieved = fl / (avg_ms[dom] / 1e3) / 1e12
        peak, peak_kind = tensor_peak()
        bound, unit, dom_bytes = "tensor", "TFLOP/s", None
    layer_bytes = sum(byt[i % n_inst]["layer"] for i in range(args.steps)) / args.steps
    layer_gbs = layer_bytes / (ms / args.steps / 1e3) / 1e9

    # end to end through the host-buffer entry point (copies inside the region)
    ne = min(args.steps, 1000)
    xh = [torch.from_numpy(synth.tokens(cfg, step=l)).pin_memory() for l in range(n_inst)]
    lh = [torch.from_numpy(synth.logits(cfg, l)).pin_memory() for l in range(n_inst)]
    oh = torch.empty((cfg.T, cfg.H), dtype=torch.float16).pin_memory()
    for i in range(min(10, ne)):
        m.pw_moe_forward_host(i % n_inst, xh[i % n_inst], lh[i % n_inst], cfg.top_k, cfg.renorm, oh, ws=ws)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(ne):
        l = i % n_inst
        m.pw_moe_forward_host(l, xh[l], lh[l], cfg.top_k, cfg.renorm, oh, ws=ws)
    e2e_dt = max_over_ranks(time.perf_counter() - t0, world)
    e2e = world * cfg.T * ne / e2e_dt

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, reps, dt = oracle_rate(cfg, 0, args.cpu_seconds)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
               "value_1_thread": oracle_rate_one_thread(cfg, min(10.0, args.cpu_seconds)),
               "sample": f"{reps} full layer forwards (batch {cfg.T}) of layer instance 0 in {dt:.1f} s, "
                         "fp64 numpy (BLAS matmuls threaded, gathers single-threaded)"}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "I": cfg.I,
                   "top_k": cfg.top_k, "renorm": cfg.renorm, "bits": (f"uniform q={uq} (byte-weighted mean of the mixed assignment)" if uq is not None
                            else "per block in {3..8}, hot experts >= 6"),
                   "accumulate": "f32", "parallelism": f"replicas x{world}",
                   "l2": f"{n_inst} distinct layer instances cycled; inputs larger than L2 between reuses",
                   "layer_weight_bytes_per_step": layer_bytes, "layer_gbs": layer_gbs,
                   "kernel_ms": avg_ms},
        "roofline": {"bound": bound, "kernel": dom, "duration": duration, "achieved": achieved, "peak": peak,
                     "unit": unit,
                     "frac": achieved / peak, "peak_kind": peak_kind, "traffic": profiled_traffic(dom, cfg.name),
                     "bytes_per_launch": dom_bytes},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e, "unit": "tokens/s", "h2d_bytes_per_step": cfg.T * cfg.H * 2 + cfg.T * cfg.E * 4,
                "d2h_bytes_per_step": cfg.T * cfg.H * 2 + 4},
        "gpu_launches": (1 if fused else 4) * args.steps,
        "clocks": clk,
        "wall_s": wall,
    }
    print(json.dumps(line), flush=True)


def run_stack(args, cfg, rank, world, local):
    """24-layer Qwen-shaped stack, decode batch 4: bits fitted to 40% of the fp16
    bytes; at step --reload-at a seeded 25% of the blocks below 8 bits start an
    asynchronous host->device reload of two more planes on a side stream, and
    each is committed (stream ordered) at the first step boundary after its copy
    completed.  Reports tokens/s before, during and after the reload window."""
    import numpy as np
    import torch
    import any_precision_weight_gb300 as pw
    from any_precision_weight_gb300.model import HostStore, load_expert_layer
    import synth

    dev = torch.device("cuda", local)
    L = cfg.n_layers
    bits = synth.stack_bits(cfg)
    plan = synth.reload_plan(cfg, bits)
    target = {(l, e, k): qn for (l, e, k, qo, qn) in plan}
    m = pw.PagedMoE(L, cfg.E, cfg.H, cfg.I, device=dev)
    store = HostStore()
    for l in range(L):
        src = lambda e, k, l=l: (synth.parent_indices(cfg, l, e, k), synth.parent_lut(cfg, l, e, k))
        load_expert_layer(m, l, src, bits[l], store=store,
                          alloc_planes=lambda e, k, l=l: target.get((l, e, k), int(bits[l, e, k])))
    Lg = [torch.from_numpy(synth.logits(cfg, l)).to(dev) for l in range(L)]
    X0 = [torch.from_numpy(synth.tokens(cfg, step=i)).to(dev) for i in range(8)]
    bufs = [torch.empty((cfg.T, cfg.H), dtype=torch.float16, device=dev) for _ in range(2)]
    ws = m.workspace(cfg.T, cfg.top_k)
    stream = torch.cuda.current_stream()
    copy = torch.cuda.Stream(device=dev)

    def step(i):
        x = X0[i % len(X0)]
        for l in range(L):
            o = bufs[l & 1]
            m.pw_moe_forward(l, x, Lg[l], cfg.top_k, cfg.renorm, residual=x, out=o, ws=ws)
            x = o

    # routing depends only on each layer's fixed logits: weight bytes per step
    bits_after = bits.copy()
    for (l, e, kind, qo, qn) in plan:
        bits_after[l, e, kind] = qn
    step_bytes = [0, 0]
    for l in range(L):
        _, _, _, off, _ = m.pw_moe_forward(l, X0[0], Lg[l], cfg.top_k, cfg.renorm, ws=ws, routing=True)
        counts = np.diff(off.cpu().numpy())
        step_bytes[0] += algorithmic_bytes(cfg, bits[l], counts)["layer"]
        step_bytes[1] += algorithmic_bytes(cfg, bits_after[l], counts)["layer"]

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    n = args.steps
    reload_at = min(args.reload_at, n - 1)
    clocks = Clocks(local)
    clocks.start()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    for e_ in ev + [c0, c1]:          # torch creates the CUDA event at its first record
        e_.record(stream)
    torch.cuda.synchronize()
    reload_bytes = 0
    for (l, e, kind, qo, qn) in plan:
        R, K = m.rows_cols(kind)
        reload_bytes += (qn - qo) * R * K // 8 + R * 2 * sum(1 << b for b in range(qo + 1, qn + 1))
    items = [(l, e, kind, qn) for (l, e, kind, qo, qn) in plan]
    m.pw_mover_start(copy, max_inflight_bytes=args.reload_inflight_mb << 20)
    committed = 0
    commit_launches = 0
    last = reload_at
    landed = False
    w0 = time.perf_counter()
    ev[0].record(stream)
    for i in range(n):
        if i >= 2:
            ev[i - 1].synchronize()      # at most two steps in flight, as a decode loop that
                                         # needs step i-2's tokens before launching step i
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
        step(args.warmup + i)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - w0
    clk = clocks.stop()
    t = np.array([ev[i].elapsed_time(ev[i + 1]) for i in range(n)])
    copy_ms = c0.elapsed_time(c1) if landed else None
    before = t[:reload_at]
    during = t[reload_at:last + 1]
    after = t[last + 1:]
    tps = lambda a: float(cfg.T / (a.mean() / 1e3)) if len(a) else None
    ms_total = float(t.sum())
    ms_max = max_over_ranks(ms_total, world)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": world * cfg.T * n / (ms_max / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": n, "warmup": args.warmup, "ms_per_step": ms_max / n, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": cfg.name, "layers": L, "T": cfg.T, "H": cfg.H, "E": cfg.E, "I": cfg.I,
                   "top_k": cfg.top_k, "bits": "greedy fit to 40% of fp16 bytes",
                   "device_weight_bytes": m.device_bytes(), "host_store_bytes": store.nbytes(),
                   "l2": "24 layers of weights (about 10 GB) between reuses, larger than L2"},
        "stack": {"tokens_per_s_before": tps(before), "tokens_per_s_during": tps(during),
                  "tokens_per_s_after": tps(after),
                  "loss_pct_during": (1 - tps(during) / tps(before)) * 100 if len(during) and len(before) else None,
                  "reload_at_step": reload_at, "last_commit_step": last, "reloaded_blocks": len(plan),
                  "reload_bytes": reload_bytes, "committed": committed, "submit_to_last_commit_ms": copy_ms,
                  "mover": f"native mover thread, at most {args.reload_inflight_mb} MiB of copies in flight",
                  "reload_gbs": reload_bytes / (copy_ms / 1e3) / 1e9 if copy_ms else None},
        "roofline": {"bound": "hbm", "kernel": "layer_fused (whole step)",
                     "achieved": step_bytes[0] / (before.mean() / 1e3) / 1e9 if len(before) else None,
                     "peak": hbm_peak()[0], "unit": "GB/s", "peak_kind": hbm_peak()[1], "traffic": None,
                     "bytes_per_step_before": step_bytes[0], "bytes_per_step_after": step_bytes[1],
                     "achieved_after": step_bytes[1] / (after.mean() / 1e3) / 1e9 if len(after) else None},
        "gpu_launches": n * L + commit_launches, "clocks": clk, "wall_s": wall,
    }
    r = line["roofline"]
    if r["achieved"] is not None:
        r["frac"] = r["achieved"] / r["peak"]
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
