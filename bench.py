#!/usr/bin/env python
"""Benchmark: the routed-MoE FFN decode step on a 43-layer Q8_0 stack (GB300).

Workload (``decode_stack43``): 43 resident decode MoE layers, each H=2048,
I=1024, 64 routed experts (top-6) + 1 shared expert, Q8_0 weights (18.7 GB
in HBM), 1 token per step, router logits skewed by a Zipf(1.1) per-expert
offset; the step ends with the greedy argmax over 129,280 vocabulary logits.
One step = one token through all 43 layers (route, quantize, group, gate/up
pair + SwiGLU, down + combine per layer) + the argmax: every kernel of the
path.  Inputs are pre-drawn for 64 steps (x and logits per layer) and cycle.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead, on
a bounded sample (one layer of one token per step), on the host cores.

Timing: W warm-up steps, then K steps bracketed by a barrier and a device
synchronize, timed with CUDA events on the launch stream; max over ranks.
L2: every step reads ~2.0 GB of distinct expert weights (> 129 MB L2).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_moe_decode_luce_gb300 import workloads as W  # noqa: E402
from quantized_moe_decode_luce_gb300.replicas import job_throughput, rank_seed  # noqa: E402

METRIC = "MoE-FFN layer µs, tokens/s and expert-weight HBM GB/s vs GB300 peak"
UNIT = "tokens/s"
VOCAB = 129280
SPEC_HBM_GBS = 8000.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-graph", action="store_true", help="launch eagerly instead of replaying CUDA graphs")
    p.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-edge-ops", action="store_true", help="skip timing the router and vocabulary-split steps")
    p.add_argument("--no-configs", action="store_true",
                   help="skip timing the single decode, verify and prefill layer workloads")
    p.add_argument("--path", choices=["layer", "split"], default="layer",
                   help="layer: each MoE layer is one launch (luce_moe_layer); split: prep, gate/up, down launches")
    p.add_argument("--layers", type=int, default=None, help="(debug) fewer layers; invalid as a bench number")
    p.add_argument("--input-steps", type=int, default=None,
                   help="pre-drawn input steps to cycle (default 64; fewer keeps profiling runs short)")
    p.add_argument("--layer-only", choices=["decode_layer", "verify_layer", "prefill_layer", "q4k_decode_layer",
                                             "decode_chain"],
                   default=None,
                   help="(profiling) run one layer workload --reps times through luce_moe_layer (or, for "
                        "q4k_decode_layer, the two Q4_K launches) and print its event-timed µs per layer; no "
                        "bench line")
    p.add_argument("--reps", type=int, default=1)
    return p.parse_args()


def chain_only(args):
    """(profiling) The chained 43-layer decode stack (router + layer per layer,
    final add, argmax), `reps` steps launched eagerly after one untimed step:
    the command of the chained stack's launch list."""
    import torch

    from quantized_moe_decode_luce_gb300 import binding as Bd
    from quantized_moe_decode_luce_gb300 import build as Bl
    from quantized_moe_decode_luce_gb300.layer import Argmax, MoEStep
    Bl.build()
    Bd.lib()
    Bd.luce_set_pdl(not args.no_pdl)
    dev = torch.device("cuda")
    wl = W.Workload(**{**W.WORKLOADS["decode_stack43"].__dict__, "steps": 8})
    layers = args.layers or wl.layers
    wls = W.Workload(**{**wl.__dict__, "layers": 1})
    dls = [W.device_layer(wls, wl.seed * 1000 + l, dev) for l in range(layers)]
    xs, lg, biases, vocab = draw_inputs(wl, layers, 0)
    xs_d, b_d, vocab_d = (torch.from_numpy(a).to(dev) for a in (xs, biases, vocab))
    bufs = MoEStep(wl.T, wl.H, wl.I, wl.E, wl.k, wl.shared, wl.clamp, device=dev)
    am = Argmax(1, VOCAB, device=dev)
    stream = torch.cuda.Stream(device=dev)
    chain_measure(dev, 1.0, stream, wl, layers, dls, b_d, xs_d, vocab_d, bufs, am, 0, eager_steps=1)
    r = chain_measure(dev, 1.0, stream, wl, layers, dls, b_d, xs_d, vocab_d, bufs, am, 0,
                      eager_steps=max(1, args.reps))
    print(json.dumps({"workload": "decode_chain", "layers": layers, "launches_per_step": 2 * layers + 2, **r,
                      "device_faults": Bd.luce_get_fault()}))


def q4k_layer_only(args):
    """The Q4_K decode-shape layer (T=1, H=2048, I=1024, 64 experts + shared,
    230 MB of Q4_K weights, six distinct experts drawn per rep): gate/up with
    its q8_1 blocks of h, then down + combine, `reps` times after one untimed
    call; for the ncu summary of those two kernels."""
    import torch

    from quantized_moe_decode_luce_gb300 import binding as Bd
    from quantized_moe_decode_luce_gb300 import build as Bl
    Bl.build()
    Bd.lib()
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    E, H, I, k = 64, 2048, 1024, 6

    def q4k(rows, K):
        b = torch.randint(0, 256, (rows, K // 256, 144), generator=g, device=dev, dtype=torch.uint8)
        dd = (torch.rand((rows, K // 256, 2), generator=g, device=dev) * 1.9e-3 + 1e-4).half()
        b[..., 0:4] = dd.view(torch.uint8).reshape(rows, K // 256, 4)
        return b

    wg, wu, wd = q4k(E * I, H), q4k(E * I, H), q4k(E * H, I)
    wsg, wsu, wsd = q4k(I, H), q4k(I, H), q4k(H, I)
    n = args.reps + 1
    ids = torch.stack([torch.randperm(E, generator=g, device=dev)[:k] for _ in range(n)]).int().view(n, 1, k)
    wts = torch.full((1, k), 1.0 / k, device=dev)
    xq = torch.zeros((1, H // 32, 36), dtype=torch.uint8, device=dev)
    Bd.luce_quantize_q8_1(torch.randn((1, H), generator=g, device=dev), xq)
    h = torch.zeros((k + 1, I), device=dev)
    hq = torch.zeros((k + 1, I // 32, 36), dtype=torch.uint8, device=dev)
    out = torch.empty((1, H), device=dev)

    def one(i):
        Bd.luce_moe_glu_q4k(wg, wu, wsg, wsu, xq, ids[i], E, H, I, 0.0, h, hq)
        Bd.luce_moe_down_combine_q4k(wd, wsd, hq, ids[i], wts, E, H, I, out)

    one(0)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record()
    for i in range(1, n):
        one(i)
    ev[1].record()
    torch.cuda.synchronize()
    print(json.dumps({"workload": "q4k_decode_layer", "path": "k_glu_q4k (with hq) + k_down_combine_q4k",
                      "reps": args.reps, "us_per_layer": ev[0].elapsed_time(ev[1]) * 1e3 / max(1, args.reps),
                      "device_faults": Bd.luce_get_fault()}))


def layer_only(args):
    """One layer workload (the parity-test inputs) through luce_moe_layer, `reps`
    times after one untimed call: the short, self-contained command that the
    ncu summaries in profiles/ are taken from."""
    import torch

    from quantized_moe_decode_luce_gb300 import binding as Bd
    from quantized_moe_decode_luce_gb300 import build as Bl
    from quantized_moe_decode_luce_gb300.layer import MoEStep
    Bl.build()
    Bd.lib()
    wl = W.WORKLOADS[args.layer_only]
    dl = W.device_layer(wl, wl.seed, "cuda")
    x = torch.from_numpy(W.activations(W.rng(wl.seed, 2), wl.T, wl.H)).cuda()
    lg, b = W.router_logits(W.rng(wl.seed, 3), wl)
    lg = torch.from_numpy(lg).cuda()
    b = torch.from_numpy(b).cuda() if b is not None else None
    st = MoEStep(wl.T, wl.H, wl.I, wl.E, wl.k, wl.shared, wl.clamp)
    if args.path == "split":
        st.path = "split"
    st.run(dl, x, lg, b)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record()
    for _ in range(args.reps):
        st.run(dl, x, lg, b)
    ev[1].record()
    torch.cuda.synchronize()
    print(json.dumps({"workload": wl.name, "path": _path_label(st), "reps": args.reps,
                      "us_per_layer": ev[0].elapsed_time(ev[1]) * 1e3 / max(1, args.reps),
                      "device_faults": Bd.luce_get_fault()}))


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def config_dict(wl, layers, graph):
    return {"workload": "decode_stack43", "tokens_per_step": wl.T, "layers": layers, "hidden": wl.H,
            "expert_intermediate": wl.I, "routed_experts": wl.E, "top_k": wl.k, "shared_experts": 1,
            "weights": "Q8_0 (34 B / 32 values)", "activations": "q8_1", "argmax_vocab": VOCAB,
            "input_steps": wl.steps, "graph": graph,
            "l2": "inputs larger than L2: each step reads ~2.0 GB of distinct expert weights (18.7 GB resident)"}


# ----------------------------------------------------------------------------- inputs
def draw_inputs(wl, layers, rank):
    """Per layer bias, per (step, layer) x and logits, per step vocab logits."""
    seed = rank_seed(wl.seed, rank)
    xs = np.empty((wl.steps, layers, wl.T, wl.H), np.float32)
    lg = np.empty((wl.steps, layers, wl.T, wl.E), np.float32)
    biases = []
    for l in range(layers):
        g = W.rng(seed, 10_000 + l)
        wl_l = W.Workload(**{**wl.__dict__})
        # one Zipf ranking and bias per layer; fresh N(0, 1) draws per step
        logits_all, bias = W.router_logits(g, wl_l, T=wl.T * wl.steps)
        biases.append(bias)
        lg[:, l] = logits_all.reshape(wl.steps, wl.T, wl.E)
        xs[:, l] = W.activations(W.rng(seed, 20_000 + l), wl.T * wl.steps, wl.H).reshape(wl.steps, wl.T, wl.H)
    vocab = W.vocab_logits(W.rng(seed, 30_000), wl.steps, VOCAB).reshape(wl.steps, 1, VOCAB)
    return xs, lg, np.stack(biases), vocab


def layer_bytes(wl, n_active):
    """Algorithmic bytes of one layer: touched expert weights + activations."""
    wts = W.touched_weight_bytes(wl, n_active)
    rows = wl.T * wl.k + wl.T
    act = (wl.T * wl.H * 4 + wl.T * wl.E * 4 + wl.T * wl.H // 32 * 36 * 2 + rows * wl.I * 4 * 2
           + rows * wl.I // 32 * 36 * 2 + wl.T * wl.H * 4)
    return wts + act


def glu_bytes(wl, n_active):
    """Algorithmic bytes of one gate/up launch: gate+up rows of the touched
    experts, the q8_1 input, h and hq written."""
    n = n_active + 1
    rows = wl.T * wl.k + wl.T
    return (n * 2 * wl.I * wl.H // 32 * 34 + wl.T * wl.H // 32 * 36 + rows * wl.I * 4
            + rows * wl.I // 32 * 36)


def down_bytes(wl, n_active):
    n = n_active + 1
    rows = wl.T * wl.k + wl.T
    return n * wl.H * wl.I // 32 * 34 + rows * wl.I // 32 * 36 + wl.T * wl.H * 4 + wl.T * wl.k * 8


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            p = [s.strip() for s in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle (CPU) timing
def oracle_layer_times(wl, n_layers, budget_s, host_layer_fn):
    """Time the CPU oracle on up to n_layers decode layers (one token each),
    stopping after budget_s seconds of oracle work."""
    import oracle
    times = []
    spent = 0.0
    for l in range(n_layers):
        args = host_layer_fn(l)
        t = time.perf_counter()
        oracle.moe_layer(*args)
        dt = time.perf_counter() - t
        times.append(dt)
        spent += dt
        if spent >= budget_s:
            break
    return times


def host_layer_sampler(wl, layers, seed):
    """Host-drawn layer inputs for the oracle: only the experts the router
    selects are drawn (the oracle never reads the others)."""
    xs, lg, biases, _ = draw_inputs(wl, layers, 0)

    def make(l):
        import oracle
        ids, _ = oracle.route_topk(lg[0, l], biases[l], wl.k)
        used = sorted(set(ids.reshape(-1).tolist()))
        g = W.rng(seed, 40_000 + l)
        E = wl.E
        nb_h, nb_i = wl.H // 32, wl.I // 32
        wg = np.zeros((E, wl.I, nb_h, 34), np.uint8)
        wu = np.zeros_like(wg)
        wd = np.zeros((E, wl.H, nb_i, 34), np.uint8)
        for e in used:
            wg[e] = W.q8_0_blocks(g, wl.I, wl.H)
            wu[e] = W.q8_0_blocks(g, wl.I, wl.H)
            wd[e] = W.q8_0_blocks(g, wl.H, wl.I)
        wsg, wsu, wsd = W.q8_0_blocks(g, wl.I, wl.H), W.q8_0_blocks(g, wl.I, wl.H), W.q8_0_blocks(g, wl.H, wl.I)
        return (wg, wu, wd, wsg, wsu, wsd, xs[0, l], lg[0, l], biases[l], wl.k, wl.clamp)

    return make


def run_reference(args, wl, layers):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    make = host_layer_sampler(wl, layers, wl.seed)
    steps = max(1, args.steps)
    warm = max(0, args.warmup)
    # each step: one decode layer of one token (a bounded sample of the token)
    per = []
    budget = 150.0
    t_all = time.perf_counter()
    prepared = {}
    for i in range(warm + steps):
        l = i % layers
        if l not in prepared:
            prepared[l] = make(l)
        t = time.perf_counter()
        oracle.moe_layer(*prepared[l])
        dt = time.perf_counter() - t
        if i >= warm:
            per.append(dt)
        if time.perf_counter() - t_all > budget and len(per) >= 1:
            break
    layer_s = float(np.mean(per))
    value = 1.0 / (layer_s * layers)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": len(per), "warmup": warm, "ms_per_step": layer_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "i8 codes, f64 accumulation", "data": "synthetic",
            "config": {**config_dict(wl, layers, False), "pdl": False},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{len(per)} steps, each one decode layer of one token "
                                       f"(x {layers} layers = 1 token); single-threaded C oracle"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "layer_us": layer_s * 1e6}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm
def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_files, kernel):
    """dram bytes per launch of `kernel` from the committed ncu summaries, if
    they were taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        entries = d if isinstance(d, list) else [d]
        for ent in entries:
            if ent.get("kernel") == kernel and ent.get("source_hash") == source_hash(kernel_files):
                return ent.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def edge_ops_measure(dev, peak, stream):
    """Device time of the steps either side of the layer at the decode sizes,
    inputs rotating over more distinct buffers than L2 holds: the RMS norm +
    router logits (T=1, E=64, H=2048, F32 router matrix) and the greedy token
    of a 129,280-entry vocabulary split into two shards (two shard argmaxes
    and the pick).  Returns kernels-dict entries."""
    import torch
    from quantized_moe_decode_luce_gb300 import binding as Bd

    g = torch.Generator(device=dev)
    g.manual_seed(77)
    out = {}
    T, E, H, N = 1, 64, 2048, 320  # 320 x 0.5 MB router matrices: 168 MB > L2
    wr = torch.randn((N, E, H), generator=g, device=dev) * 0.02
    xs = torch.randn((N, T, H), generator=g, device=dev)
    gamma = torch.ones(H, device=dev)
    xn = torch.empty((T, H), device=dev)
    lg = torch.empty((T, E), device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed_graph(body, n):
        # the n calls captured once and replayed: device time, no host launch cost
        with torch.cuda.stream(stream):
            body(0, 8)
            torch.cuda.synchronize()
            gph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gph, stream=stream):
                body(0, n)
            gph.replay()
            torch.cuda.synchronize()
            ev[0].record(stream)
            gph.replay()
            ev[1].record(stream)
            torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) * 1e3 / n

    wr_v = [wr[i] for i in range(N)]
    xs_v = [xs[i] for i in range(N)]

    def router_calls(a, b):
        for i in range(a, b):
            Bd.luce_rmsnorm_router(xs_v[i], gamma, 1e-6, wr_v[i], xn, lg)

    us = timed_graph(router_calls, N)
    nbytes = E * H * 4 + 2 * T * H * 4 + H * 4 + T * E * 4
    out["k_rmsnorm_router"] = {"workload": "T=1 E=64 H=2048 fp32 router", "avg_launch_us": us,
                               "bytes_per_launch": nbytes, "GBps": nbytes / (us * 1e-6) / 1e9,
                               "frac": nbytes / (us * 1e-6) / 1e9 / peak, "bound": "hbm (latency-bound at this size)"}
    del wr, xs
    V, R, N2 = 129280, 1, 300  # 300 vocabulary rows of 517 KB: 155 MB > L2
    half = V // 2
    vocab = torch.randn((N2, 2, R, half), generator=g, device=dev)
    ws = [torch.zeros(Bd.luce_argmax_workspace_bytes(R, half), dtype=torch.uint8, device=dev) for _ in range(2)]
    vals = torch.empty((2, R), device=dev)
    idxs = torch.empty((2, R), dtype=torch.int32, device=dev)
    idx = torch.empty(R, dtype=torch.int32, device=dev)
    val = torch.empty(R, device=dev)

    shards = [[vocab[i, s] for s in range(2)] for i in range(N2)]
    idx_v = [idxs[s] for s in range(2)]
    val_v = [vals[s] for s in range(2)]

    def pick_steps(a, b):
        for i in range(a, b):
            for s in range(2):
                Bd.luce_argmax_shard(shards[i][s], s * half, idx_v[s], val_v[s], ws[s])
            Bd.luce_argmax_pick(vals, idxs, idx, val)

    us = timed_graph(pick_steps, N2)
    nbytes = V * 4 * R
    out["k_argmax_shard x2 + k_argmax_pick"] = {"workload": "1 x 129,280 fp32 logits in two shards",
                                                "avg_step_us": us, "launches": 3, "bytes_per_step": nbytes,
                                                "GBps": nbytes / (us * 1e-6) / 1e9,
                                                "frac": nbytes / (us * 1e-6) / 1e9 / peak,
                                                "bound": "hbm (latency-bound at this size)"}

    # the Q4_K path at the decode shape: 64 routed experts + shared (230 MB,
    # more than L2), six distinct routed experts drawn per step
    E, H, I, k, N3 = 64, 2048, 1024, 6, 200

    def q4k(rows, K):
        b = torch.randint(0, 256, (rows, K // 256, 144), generator=g, device=dev, dtype=torch.uint8)
        dd = (torch.rand((rows, K // 256, 2), generator=g, device=dev) * 1.9e-3 + 1e-4).half()
        b[..., 0:4] = dd.view(torch.uint8).reshape(rows, K // 256, 4)
        return b

    wg, wu, wd = q4k(E * I, H), q4k(E * I, H), q4k(E * H, I)
    wsg, wsu, wsd = q4k(I, H), q4k(I, H), q4k(H, I)
    ids_all = torch.stack([torch.randperm(E, generator=g, device=dev)[:k] for _ in range(N3)]).int().view(N3, 1, k)
    wts = torch.full((1, k), 1.0 / k, device=dev)
    xq = torch.zeros((1, H // 32, 36), dtype=torch.uint8, device=dev)
    Bd.luce_quantize_q8_1(torch.randn((1, H), generator=g, device=dev), xq)
    hbuf = torch.zeros((k + 1, I), device=dev)
    hq = torch.zeros((k + 1, I // 32, 36), dtype=torch.uint8, device=dev)
    o = torch.empty((1, H), device=dev)
    ids_v = [ids_all[i] for i in range(N3)]

    def q4k_steps(a, b):
        for i in range(a, b):
            Bd.luce_moe_glu_q4k(wg, wu, wsg, wsu, xq, ids_v[i], E, H, I, 0.0, hbuf, hq)
            Bd.luce_moe_down_combine_q4k(wd, wsd, hq, ids_v[i], wts, E, H, I, o)

    us = timed_graph(q4k_steps, N3)
    nbytes = (k + 1) * 3 * I * (H // 256) * 144 + H // 32 * 36 + (k + 1) * I * 4 + H * 4
    out["Q4_K layer (k_glu_q4k with its q8_1 blocks of h + k_down_combine_q4k)"] = {
        "workload": "T=1 H=2048 I=1024 E=64 k=6 + shared, Q4_K weights", "avg_step_us": us, "launches": 2,
        "bytes_per_step": nbytes, "GBps": nbytes / (us * 1e-6) / 1e9, "frac": nbytes / (us * 1e-6) / 1e9 / peak,
        "bound": "hbm"}
    return out


def chain_measure(dev, peak, stream, wl, layers, dls, b_d, xs_d, vocab_d, bufs, am, lb, eager_steps=0):
    """The decode stack with the step before each layer in the chain: per
    layer the residual add that makes the layer's input (the previous layer's
    input + output), its RMS norm and the router logits (F32 router matrix
    [E][H]) in one launch, then the one-launch MoE layer on the normed row;
    after the last layer its residual add, then the greedy token.  Each
    layer's routing therefore depends on the previous layer's output, as in a
    real decode (attention is not part of this path and is left out).
    Launches chain through programmatic launch; 8 input slots are captured
    as graphs and replayed in turn.  Returns a kernels-dict entry."""
    import torch
    from quantized_moe_decode_luce_gb300 import binding as Bd

    g = torch.Generator(device=dev)
    g.manual_seed(91)
    T, H, E = wl.T, wl.H, wl.E
    wr = torch.randn((layers, E, H), generator=g, device=dev) * 0.02
    gamma = 1.0 + 0.1 * torch.randn((layers, H), generator=g, device=dev)
    xres = torch.empty((layers + 1, T, H), device=dev)
    xn = torch.empty((T, H), device=dev)
    lg = torch.empty((T, E), device=dev)
    outc = torch.empty((2, T, H), device=dev)
    S = min(8, xs_d.shape[0])

    def chain_step(s):
        x = xs_d[s, 0]
        for l in range(layers):
            lay = dls[l]
            if l == 0:
                Bd.luce_rmsnorm_router(x, gamma[l], 1e-6, wr[l], xn, lg)
            else:
                Bd.luce_add_rmsnorm_router(x, outc[(l - 1) % 2], xres[l], gamma[l], 1e-6, wr[l], xn, lg)
                x = xres[l]
            Bd.luce_moe_layer(lg, b_d[l], xn, wl.k, wl.I, lay.wg, lay.wu, lay.wd, lay.wsg, lay.wsu, lay.wsd,
                              wl.clamp, bufs.ids, bufs.weights, bufs.xq, bufs.counts, bufs.offsets, bufs.routes,
                              bufs.h, bufs.hq, outc[l % 2], bufs.workspace)
        Bd.luce_add_f32(x, outc[(layers - 1) % 2], xres[layers])
        am.run(vocab_d[s])

    if eager_steps:  # (profiling) launches only, no graphs
        with torch.cuda.stream(stream):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for s in range(eager_steps):
                chain_step(s % S)
            e1.record(stream)
            torch.cuda.synchronize()
        return {"eager_steps": eager_steps, "us_per_step": e0.elapsed_time(e1) * 1e3 / eager_steps}
    gs = []
    with torch.cuda.stream(stream):
        for s in range(S):  # eager once: every call checked
            chain_step(s)
        torch.cuda.synchronize()
        for s in range(S):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                chain_step(s)
            gs.append(gr)
        for i in range(3 * S):
            gs[i % S].replay()
        torch.cuda.synchronize()
        n = 400
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            gs[i % S].replay()
        e1.record(stream)
        torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / n
    finite = bool(torch.isfinite(xres[layers]).all().item())
    router_b = E * H * 4 + 2 * T * H * 4 + H * 4 + T * E * 4
    step_b = layers * (lb + router_b + 3 * T * H * 4) + VOCAB * 4 * T
    return {"workload": f"{layers} x (residual add + RMS norm + router [E={E}][H={H}] fp32 in one launch, "
                        f"MoE layer) + final residual add + {VOCAB}-entry argmax, T={T}, layer l+1 routed on "
                        f"layer l's output",
            "tokens_per_s": T / (us * 1e-6), "us_per_step": us, "us_per_layer": us / layers,
            "launches_per_step": 2 * layers + 2, "bytes_per_step": step_b,
            "GBps": step_b / (us * 1e-6) / 1e9, "frac": step_b / (us * 1e-6) / 1e9 / peak,
            "input_slots": S, "steps": n, "residual_finite": finite}


def _path_label(st):
    """What luce_moe_layer (or the split launches) runs for this step's shape."""
    if st.path != "layer":
        return "prep + gate/up + down launches"
    if st.T > 8 or st.T * st.k > 64:
        return ("grouped tensor-core launches: route, quantize, group, work lists + gathered codes, "
                "gate/up GEMM, down GEMM, combine")
    return "one launch per layer"


def configs_measure(dev, peak, stream):
    """Device time of the other layer workloads, one launch sequence per
    workload captured in a CUDA graph and replayed (device time, no host
    launch cost):

    * decode_layer (T=1, H=2048, I=1024, E=64, top-6 + shared, seed 1):
      8 resident copies of the layer (3.5 GB) and 64 input draws rotate, so
      consecutive launches touch different weights (each 46.8 MB);
    * verify_layer (T=5, H=4096, I=2048, E=128, top-8 + shared, clamp 10,
      seed 2): 2 resident copies (6.9 GB) and 8 input draws (each its own
      shared column means); each launch touches (U+1) x 26.7 MB, U the
      unique routed experts, counted from the launch's own selection; plus
      the greedy argmax over 5 x 129,280 logits rotating over 64 buffers;
    * prefill_layer (T=512, H=4096, I=1536, E=128, top-8 + shared, clamp 10,
      seed 4): one copy (2.59 GB, all of it touched by every launch).

    Returns a dict of per-workload entries (µs per layer, tokens/s, GB/s and
    the fraction of the measured copy bandwidth)."""
    import torch

    from quantized_moe_decode_luce_gb300.layer import Argmax, MoEStep

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed(body, n, reps=5):
        with torch.cuda.stream(stream):
            body(0, n)  # eager once: kernel attributes, argument checks
            torch.cuda.synchronize()
            gph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gph, stream=stream):
                body(0, n)
            for _ in range(2):
                gph.replay()
            torch.cuda.synchronize()
            us = []
            for _ in range(reps):
                ev[0].record(stream)
                gph.replay()
                ev[1].record(stream)
                torch.cuda.synchronize()
                us.append(ev[0].elapsed_time(ev[1]) * 1e3 / n)
        return statistics.median(us)

    def draw(wl, n_inputs, seed):
        xs, lgs, bias = [], [], None
        for i in range(n_inputs):
            g = W.rng(seed, 50_000 + i)
            lg, b = W.router_logits(g, wl)
            if bias is None:
                bias = b
            lgs.append(lg)
            xs.append(W.activations(W.rng(seed, 60_000 + i), wl.T, wl.H))
        xs_d = torch.from_numpy(np.stack(xs)).to(dev)
        lg_d = torch.from_numpy(np.stack(lgs)).to(dev)
        b_d = torch.from_numpy(bias).to(dev) if bias is not None else None
        return xs_d, lg_d, b_d

    out = {}
    plan = [("decode_layer", 8, 64, 64), ("verify_layer", 2, 8, 16), ("prefill_layer", 1, 2, 4)]
    for name, n_copies, n_inputs, n_launch in plan:
        wl = W.WORKLOADS[name]
        lays = [W.device_layer(wl, wl.seed * 1000 + 500 + c, dev) for c in range(n_copies)]
        xs_d, lg_d, b_d = draw(wl, n_inputs, wl.seed)
        st = MoEStep(wl.T, wl.H, wl.I, wl.E, wl.k, wl.shared, wl.clamp, device=dev)
        o = torch.empty((n_launch, wl.T, wl.H), device=dev)
        # unique routed experts of each input (from the launch's own selection)
        uniq = []
        with torch.cuda.stream(stream):
            for i in range(n_inputs):
                st.run(lays[i % n_copies], xs_d[i], lg_d[i], b_d, stream=stream, out=o[0])
                uniq.append(int(torch.unique(st.ids).numel()))
        torch.cuda.synchronize()

        def body(a, b):
            for i in range(a, b):
                st.run(lays[i % n_copies], xs_d[i % n_inputs], lg_d[i % n_inputs], b_d, stream=stream, out=o[i])

        us = timed(body, n_launch)
        nb = float(np.mean([W.touched_weight_bytes(wl, uniq[i % n_inputs]) + _act_bytes(wl)
                            for i in range(n_launch)]))
        gbs = nb / (us * 1e-6) / 1e9
        ent = {"T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k, "clamp": wl.clamp,
               "path": _path_label(st),
               "us_per_layer": us, "tokens_per_s": wl.T / (us * 1e-6), "bytes_per_layer": nb,
               "GBps": gbs, "frac_of_measured_hbm": gbs / peak, "frac_of_8TBps_spec": gbs / SPEC_HBM_GBS,
               "l2": f"{n_copies} resident weight copies x {n_inputs} input draws rotate "
                     f"({n_copies * (wl.E + 1) * wl.expert_bytes / 1e9:.1f} GB resident)"}
        if name == "verify_layer":
            ent["unique_routed_experts"] = uniq
            ent["unique_routed_experts_mean"] = float(np.mean(uniq))
        if name == "prefill_layer":
            ops = 2.0 * (wl.T * wl.k + wl.T) * 3 * wl.H * wl.I
            ent["int8_ops_per_layer"] = ops
            ent["int8_tops"] = ops / (us * 1e-6) / 1e12
            # the same layer on the dp4a launches (prep, gate/up pair, down + combine), for comparison
            st.path = "split"
            us_split = timed(body, n_launch)
            ent["dp4a_split_path"] = {"us_per_layer": us_split, "int8_tops": ops / (us_split * 1e-6) / 1e12,
                                      "GBps": nb / (us_split * 1e-6) / 1e9,
                                      "tensor_core_speedup": us_split / us}
        out[name] = ent
        del lays, st, o
        torch.cuda.empty_cache()
        if name == "verify_layer":
            V, R, N = 129280, 5, 64
            g = torch.Generator(device=dev)
            g.manual_seed(wl.seed)
            vocab = torch.randn((N, R, V), generator=g, device=dev)
            am = Argmax(R, V, device=dev)
            vv = [vocab[i] for i in range(N)]

            def am_body(a, b):
                for i in range(a, b):
                    am.run(vv[i], stream=stream)

            us = timed(am_body, N)
            nbytes = R * V * 4
            out["verify_argmax"] = {"R": R, "V": V, "us": us, "bytes": nbytes,
                                    "GBps": nbytes / (us * 1e-6) / 1e9,
                                    "frac_of_measured_hbm": nbytes / (us * 1e-6) / 1e9 / peak,
                                    "l2": f"{N} logit buffers rotate ({N * nbytes / 1e6:.0f} MB)"}
            del vocab, vv, am
            torch.cuda.empty_cache()
    return out


def _act_bytes(wl):
    """Activation bytes of one layer: x and logits read, xq, h, hq written and
    read once, out written."""
    rows = wl.T * wl.k + (wl.T if wl.shared else 0)
    return (wl.T * wl.H * 4 + wl.T * wl.E * 4 + wl.T * wl.H // 32 * 36 * 2 + rows * wl.I * 4 * 2
            + rows * wl.I // 32 * 36 * 2 + wl.T * wl.H * 4)


def _oracle_worker(job):
    """One host process of the all-core oracle row: times `n` decode layers
    (inputs drawn outside the timed calls).  Returns the seconds spent in the
    oracle and the layers done."""
    wl_name, layers, seed, start, n = job
    import oracle
    wl = W.WORKLOADS[wl_name]
    make = host_layer_sampler(wl, layers, seed)
    spent, done = 0.0, 0
    for j in range(n):
        args = make((start + j) % layers)
        t = time.perf_counter()
        oracle.moe_layer(*args)
        spent += time.perf_counter() - t
        done += 1
    return spent, done


def oracle_all_cores(wl, layers, per_core_layers):
    """The oracle on every host core at once: one process per core, each
    running its own decode layers (independent work, nothing shared)."""
    import multiprocessing as mp
    ncores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    jobs = [(wl.name, layers, wl.seed, c * per_core_layers, per_core_layers) for c in range(ncores)]
    with ctx.Pool(ncores) as pool:
        res = pool.map(_oracle_worker, jobs)
    slowest = max(s for s, _ in res)
    done = sum(d for _, d in res)
    return done, slowest, ncores


def run_ours(args, wl, layers):
    import torch
    import torch.distributed as dist

    from quantized_moe_decode_luce_gb300 import binding as Bd
    from quantized_moe_decode_luce_gb300 import build as Bl
    from quantized_moe_decode_luce_gb300.layer import Argmax, MoEStep

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    Bl.build()
    Bd.lib()

    # resident weights: 43 layers x (64 routed + 1 shared) experts
    wls = W.Workload(**{**wl.__dict__, "layers": 1})
    t_gen = time.time()
    dls = [W.device_layer(wls, wl.seed * 1000 + l, dev) for l in range(layers)]
    torch.cuda.synchronize()
    t_gen = time.time() - t_gen
    xs, lg, biases, vocab = draw_inputs(wl, layers, rank)
    # active experts per (step, layer): the router's selection (T=1: always k)
    n_active = wl.k
    xs_d = torch.from_numpy(xs).to(dev)
    lg_d = torch.from_numpy(lg).to(dev)
    b_d = torch.from_numpy(biases).to(dev)
    vocab_d = torch.from_numpy(vocab).to(dev)
    outs = torch.empty((layers, wl.T, wl.H), dtype=torch.float32, device=dev)
    step_bufs = MoEStep(wl.T, wl.H, wl.I, wl.E, wl.k, wl.shared, wl.clamp, device=dev)
    am = Argmax(1, VOCAB, device=dev)
    graph = not args.no_graph
    Bd.luce_set_pdl(not args.no_pdl)

    # per-kernel timing events (recorded inside the graphs as external events)
    ev_kind = {"glu": [], "down": []}

    def make_events():
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return torch.cuda.Event(enable_timing=True)

    one_launch = args.path == "layer"

    def run_step(s, x_src, lg_src, v_src, out_dst, record, am_=None):
        bufs = step_bufs
        for l in range(layers):
            lay = dls[l]
            if one_launch:
                if record is not None:
                    record[l][0].record()
                Bd.luce_moe_layer(lg_src[s, l], b_d[l], x_src[s, l], wl.k, wl.I, lay.wg, lay.wu, lay.wd, lay.wsg,
                                  lay.wsu, lay.wsd, wl.clamp, bufs.ids, bufs.weights, bufs.xq, bufs.counts,
                                  bufs.offsets, bufs.routes, bufs.h, bufs.hq, out_dst[l], bufs.workspace)
                if record is not None:
                    record[l][1].record()
                continue
            Bd.luce_moe_prep(lg_src[s, l], b_d[l], x_src[s, l], wl.k, bufs.ids, bufs.weights, bufs.xq, bufs.counts,
                             bufs.offsets, bufs.routes)
            if record is not None:
                e0, e1, e2 = record[l]
                e0.record()
            Bd.luce_moe_glu_pair(lay.wg, lay.wu, lay.wsg, lay.wsu, bufs.xq, bufs.offsets, bufs.routes, wl.T,
                                 wl.k, wl.E, wl.H, wl.I, wl.clamp, bufs.h, bufs.hq)
            if record is not None:
                e1.record()
            Bd.luce_moe_down_combine(lay.wd, lay.wsd, bufs.hq, bufs.ids, bufs.weights, bufs.offsets, bufs.routes,
                                     wl.T, wl.k, wl.E, wl.H, wl.I, out_dst[l])
            if record is not None:
                e2.record()
        (am_ or am).run(v_src[s])

    # per layer: one launch, or prep + gate/up + down; then the argmax
    launches_per_step = layers * (1 if one_launch else 3) + 1
    S = wl.steps
    stream = torch.cuda.Stream(device=dev)
    # per-kernel timing: only the graph of input slot 0 carries event records
    # (an event node between two kernels also removes their programmatic
    # overlap, so instrumenting every step would slow the timed region)
    records = [[(make_events(), make_events(), make_events()) for _ in range(layers)] if s == 0 else None
               for s in range(S)]
    graphs = []
    with torch.cuda.stream(stream):
        for s in range(S):  # eager once: sets kernel attributes, checks every call
            run_step(s, xs_d, lg_d, vocab_d, outs, None)
        torch.cuda.synchronize()
        if graph:
            for s in range(S):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    run_step(s, xs_d, lg_d, vocab_d, outs, records[s])
                graphs.append(g)
        torch.cuda.synchronize()

    def step(i):
        if graph:
            graphs[i % S].replay()
        else:
            run_step(i % S, xs_d, lg_d, vocab_d, outs, records[i % S])

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
        barrier()
        clocks = ClockSampler(dev.index)
        time.sleep(0.3)
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        barrier()
        start.record(stream)
        for i in range(args.steps):
            step(args.warmup + i)
        end.record(stream)
        barrier()
        clk = clocks.stop()
    ms = start.elapsed_time(end)
    # per-kernel durations: the last execution of every recorded pair
    glu_ms, down_ms = [], []
    for rec in records:
        for (e0, e1, e2) in (rec or []):
            try:
                glu_ms.append(e0.elapsed_time(e1))
                if not one_launch:
                    down_ms.append(e1.elapsed_time(e2))
            except Exception:
                pass
    value, ms = job_throughput(ms, args.steps * wl.T, world, dev)
    ms_per_step = ms / args.steps
    lb = layer_bytes(wl, n_active)
    step_bytes = layers * lb + VOCAB * 4
    peak, peak_kind = measured_peaks()
    glu_avg = float(np.mean(glu_ms)) if glu_ms else None
    down_avg = float(np.mean(down_ms)) if down_ms else None
    # the argmax's share of a step, timed alone (a graph of argmax launches
    # over the rotating vocabulary rows), so that the layer kernel's time
    # follows from the timed region: (step - argmax) / layers
    am_us = None
    with torch.cuda.stream(stream):
        gam = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gam, stream=stream):
            for s in range(S):
                am.run(vocab_d[s])
        gam.replay()
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        gam.replay()
        a1.record(stream)
        torch.cuda.synchronize()
        am_us = a0.elapsed_time(a1) * 1e3 / S
    layer_us_timed = (ms_per_step * 1e3 - am_us) / layers
    kernels = {}
    roofline = None
    if one_launch:
        # the dominant (and only) layer kernel: all of the layer's algorithmic
        # bytes over its share of the timed region
        kernel_files = ["quantized_moe_decode_luce_gb300/csrc/moe_layer.cu",
                        "quantized_moe_decode_luce_gb300/csrc/common.cuh"]
        ach = lb / (layer_us_timed * 1e-6) / 1e9
        roofline = {"kernel": "k_moe_layer", "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                    "frac": ach / peak, "peak_kind": f"{peak_kind} (STREAM-style copy, burst)",
                    "frac_of_8TBps_spec": ach / SPEC_HBM_GBS, "bytes_per_launch": lb,
                    "launch_us_from_timed_region": layer_us_timed,
                    "how": "achieved = bytes_per_launch / ((ms_per_step - argmax_us) / layers)",
                    "argmax_us": am_us,
                    "traffic": profiled_traffic(kernel_files, "k_moe_layer")}
        if glu_avg:
            roofline["diag_event_bracketed_launch_us"] = glu_avg * 1e3
    else:
        gb = glu_bytes(wl, n_active)
        kernel_files = ["quantized_moe_decode_luce_gb300/csrc/glu_pair.cu",
                        "quantized_moe_decode_luce_gb300/csrc/common.cuh"]
        if glu_avg:
            ach = gb / (glu_avg * 1e-3) / 1e9
            roofline = {"kernel": "k_glu_pair", "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                        "frac": ach / peak, "peak_kind": f"{peak_kind} (STREAM-style copy)",
                        "frac_of_8TBps_spec": ach / SPEC_HBM_GBS, "bytes_per_launch": gb,
                        "avg_launch_us": glu_avg * 1e3, "traffic": profiled_traffic(kernel_files, "k_glu_pair")}
        if down_avg:
            db = down_bytes(wl, n_active)
            kernels["k_down_combine"] = {"avg_launch_us": down_avg * 1e3, "bytes_per_launch": db,
                                         "GBps": db / (down_avg * 1e-3) / 1e9}

    # e2e: host inputs -> device, the same step, result back to the host.
    # Double-buffered like a serving loop: step i+1's inputs are copied in on
    # one stream and step i's outputs and token copied out on another while
    # the device computes; every step's copies stay inside the timed region.
    e2e = None
    if rank == 0 or world > 1:
        NB = 2
        pin_x = torch.from_numpy(xs).pin_memory()
        pin_l = torch.from_numpy(lg).pin_memory()
        pin_v = torch.from_numpy(vocab).pin_memory()
        host_out = [torch.empty((layers, wl.T, wl.H), dtype=torch.float32).pin_memory() for _ in range(NB)]
        host_idx = [torch.empty(1, dtype=torch.int32).pin_memory() for _ in range(NB)]
        stage_x = [torch.empty_like(xs_d[0:1]) for _ in range(NB)]
        stage_l = [torch.empty_like(lg_d[0:1]) for _ in range(NB)]
        stage_v = [torch.empty_like(vocab_d[0:1]) for _ in range(NB)]
        outs_b = [torch.empty_like(outs) for _ in range(NB)]
        ams = [Argmax(1, VOCAB, device=dev) for _ in range(NB)]
        h2d_s = torch.cuda.Stream(device=dev)
        d2h_s = torch.cuda.Stream(device=dev)
        copied = [torch.cuda.Event() for _ in range(NB)]
        computed = [torch.cuda.Event() for _ in range(NB)]
        drained = [torch.cuda.Event() for _ in range(NB)]
        e2e_graphs = []
        with torch.cuda.stream(stream):
            for b in range(NB):  # real inputs in the staging buffers before the first (checked) calls
                stage_x[b].copy_(xs_d[0:1])
                stage_l[b].copy_(lg_d[0:1])
                stage_v[b].copy_(vocab_d[0:1])
                run_step(0, stage_x[b], stage_l[b], stage_v[b], outs_b[b], None, ams[b])
            torch.cuda.synchronize()
            if graph:
                for b in range(NB):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        run_step(0, stage_x[b], stage_l[b], stage_v[b], outs_b[b], None, ams[b])
                    e2e_graphs.append(g)
            torch.cuda.synchronize()
        K2 = max(10, min(args.steps, 500))
        h2d = (xs[0].nbytes + lg[0].nbytes + vocab[0].nbytes)
        d2h = host_out[0].numel() * 4 + 4

        def e2e_step(i):
            s, b = i % S, i % NB
            with torch.cuda.stream(h2d_s):
                h2d_s.wait_event(drained[b])  # set b's last step is computed and read back
                stage_x[b].copy_(pin_x[s:s + 1], non_blocking=True)
                stage_l[b].copy_(pin_l[s:s + 1], non_blocking=True)
                stage_v[b].copy_(pin_v[s:s + 1], non_blocking=True)
                copied[b].record(h2d_s)
            stream.wait_event(copied[b])
            with torch.cuda.stream(stream):
                if graph:
                    e2e_graphs[b].replay()
                else:
                    run_step(0, stage_x[b], stage_l[b], stage_v[b], outs_b[b], None, ams[b])
            computed[b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(computed[b])
                host_out[b].copy_(outs_b[b], non_blocking=True)
                host_idx[b].copy_(ams[b].idx, non_blocking=True)
                drained[b].record(d2h_s)

        for i in range(3):
            e2e_step(i)
        barrier()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        h2d_s.wait_event(s0)
        for i in range(K2):
            e2e_step(i)
        for b in range(NB):
            stream.wait_event(drained[b])
        s1.record(stream)
        barrier()
        e_value, _ = job_throughput(s0.elapsed_time(s1), K2 * wl.T, world, dev)
        e2e = {"value": e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": K2,
               "path": "pinned host x/logits/vocab -> device copies -> C-ABI step -> outputs + token to pinned "
                       "host, double-buffered (copies of step i+1 in and step i out overlap the device's work)"}

    if rank == 0 and not args.no_edge_ops and one_launch:
        try:
            kernels["decode_stack43_chain"] = chain_measure(dev, peak, stream, wl, layers, dls, b_d, xs_d, vocab_d,
                                                            step_bufs, am, lb)
        except Exception as exc:  # a report, never a reason to fail the bench
            kernels["decode_stack43_chain"] = {"failed": str(exc)}

    if rank == 0 and not args.no_edge_ops:
        try:
            kernels.update(edge_ops_measure(dev, peak, stream))
        except Exception as exc:  # a report, never a reason to fail the bench
            kernels["edge_ops"] = {"failed": str(exc)}

    configs = None
    if rank == 0 and not args.no_configs:
        del dls, graphs
        torch.cuda.empty_cache()
        try:
            configs = configs_measure(dev, peak, stream)
        except Exception as exc:  # a report, never a reason to fail the bench
            configs = {"failed": str(exc)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            make = host_layer_sampler(wl, layers, wl.seed)
            times = oracle_layer_times(wl, layers, 12.0, make)
            layer_s = float(np.mean(times))
            cpu = {"value": 1.0 / (layer_s * layers), "unit": UNIT, "cores": 1, "kind": "oracle",
                   "sample": f"{len(times)} decode layers of one token (T=1, H=2048, I=1024, E=64, top-6 + shared); "
                             f"tokens/s = 1 / (mean layer time x {layers})",
                   "layer_us": layer_s * 1e6}
            done, slowest, ncores = oracle_all_cores(wl, layers, max(2, len(times) // 2))
            cpu["all_cores"] = {"value": done / slowest / layers, "unit": UNIT, "cores": ncores,
                                "kind": "oracle",
                                "sample": f"{done} decode layers, one process per core, each its own layers "
                                          f"(independent tokens); tokens/s = layers done / slowest process's "
                                          f"oracle seconds / {layers}"}
        except Exception as exc:  # the baseline is a report, never a reason to fail the bench
            cpu = {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": f"failed: {exc}"}

    fault = Bd.luce_get_fault()
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "i8 codes (dp4a int32 block sums), f32 scales/accumulation",
                "data": "synthetic (seeded Q8_0 weights, N(0,1) activations, Zipf-skewed router logits)",
                "config": {**config_dict(wl, layers, graph), "pdl": not args.no_pdl,
                           "path": "one launch per layer" if one_launch else "prep + gate/up + down launches"},
                "layer_us": ms_per_step * 1e3 / layers,
                "stack_weight_GBps": step_bytes / (ms_per_step * 1e-3) / 1e9,
                "stack_frac_of_measured_hbm": step_bytes / (ms_per_step * 1e-3) / 1e9 / peak,
                "roofline": roofline, "kernels": kernels, "configs": configs, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches_per_step * args.steps, "clocks": clk,
                "device_faults": fault, "weights_gen_s": round(t_gen, 2)}
        if layers != 43:
            line["invalid"] = f"debug run with {layers} layers"
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    args = parse()
    if args.layer_only == "q4k_decode_layer":
        q4k_layer_only(args)
        return
    if args.layer_only == "decode_chain":
        chain_only(args)
        return
    if args.layer_only:
        layer_only(args)
        return
    wl = W.WORKLOADS["decode_stack43"]
    if args.input_steps:
        wl = W.Workload(**{**wl.__dict__, "steps": args.input_steps})
    layers = args.layers or wl.layers
    if args.impl == "reference":
        run_reference(args, wl, layers)
    else:
        run_ours(args, wl, layers)


if __name__ == "__main__":
    main()
