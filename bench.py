#!/usr/bin/env python
"""Benchmark of the MoL ("virtual experts") LoRA layer on GB300.

One step = one MoE layer's MoL LoRA path over one batch: remap + align once,
then the gate_up stage (shrink, expand) and the down stage (shrink, expand)
reusing the routing. The workload is the bs=23 decode configuration (23
tokens, 128 experts x 8 adapters = 1024 virtual experts, top-8, rank 32,
gate_up 2048 -> 2x32 -> 2x768, down 768 -> 32 -> 2048), synthetic seeded data.

The first stage computes the routing with compute_routing = 1 (--routing-mode):
the top-k and adapter ids may come from the kernel that precedes the layer; the
line also reports the layer time with mode 2 (ids declared ready before that
kernel, as when the router ran earlier in the MoE layer).

Steps rotate over --layers distinct layers (own weights, routing and
activations) so that a step never finds its weights in L2: 8 decode layers
touch ~0.7 GB per cycle, over 5x the 129 MB L2. As in a real decode step, one
CUDA graph holds those layers back to back; exactly K steps are timed.

Prints one JSON line (rank 0). Under torchrun every rank runs an independent
replica (the path has no exchange step): weak scaling, value summed over ranks
against the slowest rank's time.

--impl reference times the CPU oracle on the same workload and metric.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "MoL LoRA layer (token,vexpert) pairs/s at 1 GB300"
UNIT = "pairs/s"


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=500)
    p.add_argument("--impl", choices=["mol", "reference"], default="mol")
    p.add_argument("--config", default="decode")
    p.add_argument("--layers", type=int, default=8, help="distinct layers rotated across steps")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--ranks", default=None,
                   help="per-adapter ranks, comma separated (one per adapter; scaling 16/rank)")
    p.add_argument("--routing-mode", type=int, choices=[1, 2], default=1,
                   help="compute_routing of each layer's first stage: 1 = the top-k and adapter "
                        "ids may come from the kernel preceding the layer, 2 = they are ready "
                        "before it (as after a router that ran earlier in the layer)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-kernels", action="store_true", help="skip the per-kernel timing phase")
    p.add_argument("--extra", default="wide,wide1k,ep,prefill,dense",
                   help="other workloads timed briefly after the main line (comma separated; "
                        "'none' to skip)")
    p.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    p.add_argument("--cpu-budget", type=float, default=15.0, help=argparse.SUPPRESS)
    return p.parse_args(argv)


# --------------------------------------------------------------------------- helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle samples, kept with host timestamps."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [f.strip() for f in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        win = [s for t, s in self.samples if t0 - 0.1 <= t <= t1 + 0.1]
        if not win and self.samples:  # a very short region: the samples around it
            near = sorted(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))[:2]
            win = [s for _, s in near]
        if not win:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=[], samples=0)
        sm = [float(s[1]) for s in win if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in win if s[2].replace(".", "").isdigit()]
        reasons = set()
        for s in win:
            for name, val in zip(self.NAMES, s[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(mx) if mx else None,
                    reasons=sorted(reasons), samples=len(win))


# --------------------------------------------------------------------------- ranks

def combine_ranks(ms: float, pairs: float, device=None):
    """Weak scaling over independent replicas: slowest rank's time, sum of every rank's pairs."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms, pairs
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    p = torch.tensor([pairs], dtype=torch.float64, device=device)
    dist.all_reduce(p, op=dist.ReduceOp.SUM)
    return float(t.item()), float(p.item())


def shard_tokens(num_tokens: int, world: int, rank: int):
    """Contiguous token range of `rank` when one batch is split over `world` replicas."""
    base, extra = divmod(num_tokens, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


# --------------------------------------------------------------------------- GPU arm

class LayerState:
    """Device tensors of one layer: routing, workspace, per-stage inputs and outputs."""

    # compute_routing of the first stage (the others reuse its routing)
    routing_mode = 1

    def __init__(self, wl, li, dev, mol, torch, ranks=None):
        self.wl, self.li = wl, li
        self.ranks = None if ranks is None else np.asarray(ranks, np.int32)
        self.ranks_d = self.scal_d = None
        if ranks is not None:
            self.ranks_d = torch.from_numpy(self.ranks).to(dev)
            scal = np.array([16.0 / r if r > 0 else 0.0 for r in self.ranks], np.float32)
            self.scal_d = torch.from_numpy(scal).to(dev)
        self.topk = torch.from_numpy(li.topk_ids).to(dev)
        self.lora = torch.from_numpy(li.lora_ids).to(dev)
        self.routing = mol.alloc_routing(wl.numel, wl.V, wl.BM, dev)
        self.ws = mol.alloc_workspace(wl.numel, wl.V, wl.BM, dev)
        self.stages = []
        for st in li.stages:
            self.stages.append(dict(
                st=st, x=st.x.to_device(dev), A=st.A.to_device(dev), B=st.B.to_device(dev),
                out=st.out0.to_device(dev),
                inter=torch.zeros((wl.numel, st.stage.R), dtype=torch.float32, device=dev)))

    def forward(self, mol):
        wl = self.wl
        for si, d in enumerate(self.stages):
            mol.mol_lora_forward(d["x"], d["st"].x_row_div, self.topk, self.lora, wl.E, wl.L,
                                 d["A"], d["B"], d["st"].stage.S, wl.scale, d["out"], self.routing,
                                 d["inter"], compute_routing=(self.routing_mode if si == 0 else 0),
                                 workspace=self.ws,
                                 lora_ranks=self.ranks_d, lora_scalings=self.scal_d)

    def counts(self):
        """Pairs that get a delta, their touched virtual experts' adapters and distinct token
        rows, from the routing output (pairs of rank-0 adapters get none)."""
        vt = self.routing.vtopk_ids.cpu().numpy().reshape(-1)
        valid = vt >= 0
        if self.ranks is not None:
            valid &= self.ranks[np.maximum(vt, 0) // self.wl.E] > 0
        touched = np.unique(vt[valid])
        rows = np.unique(np.nonzero(valid)[0] // self.wl.topk)
        return int(valid.sum()), int(touched.size), int(rows.size), touched // self.wl.E

    def stage_bytes(self, si, pairs, touched, token_rows, adapters):
        """Algorithmic HBM bytes of one stage's shrink and expand (an adapter of rank r_l needs
        r_l of the r rows of each slice of lora_a and r_l of the r columns of lora_b)."""
        st = self.stages[si]["st"].stage
        x_rows = token_rows if self.stages[si]["st"].x_row_div > 1 else pairs
        rank_sum = touched * st.r if self.ranks is None else \
            int(np.minimum(self.ranks[adapters], st.r).sum())
        shrink = st.S * rank_sum * st.K * 2 + x_rows * st.K * 2 + pairs * st.R * 4
        expand = st.N * rank_sum * 2 + pairs * st.R * 4 + pairs * st.N * 2 * 2
        return shrink, expand

    def align_bytes(self):
        wl = self.wl
        return wl.numel * (4 + 4) + wl.T * 4 + self.routing.capacity * 4 + self.routing.expert_ids.numel() * 4 + 4


def time_graphs(torch, graphs, steps, warmup):
    """Replay graphs round-robin; return ms per replay from CUDA events on the current stream."""
    n = len(graphs)
    for i in range(warmup):
        graphs[i % n].replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for i in range(steps):
        graphs[i % n].replay()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / steps


def event_ms(torch, fn, reps):
    """ms per call of fn() (which enqueues work on the current stream), CUDA events around
    `reps` calls, synchronized on both sides."""
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record()
    for _ in range(reps):
        fn()
    ev1.record()
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1) / reps


def capture(torch, fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def layer_steps_timer(torch, mol, layers, steps):
    """Graphs that run exactly `steps` layer steps, step i on layer i % len(layers): graphs of
    GRAPH_ROTATIONS rotations of the layers back to back (replayed steps // that many times)
    and, for the remainder, one graph of the next steps (one graph for up to that many steps,
    as a model's layers captured together would run). Returns (run, warm): run() enqueues the
    K steps; warm(w) replays every graph the timed region uses at least twice and covers at
    least w warm-up steps."""
    nl = len(layers)
    cap = nl * GRAPH_ROTATIONS
    full, rest = divmod(steps, cap)
    multi = capture(torch, lambda: [layers[i % nl].forward(mol) for i in range(cap)]) if full else None
    tail = capture(torch, lambda: [layers[i % nl].forward(mol) for i in range(rest)]) if rest else None

    def run():
        for _ in range(full):
            multi.replay()
        if tail is not None:
            tail.replay()

    def warm(w):
        done = 0
        for g, n in ((multi, cap), (tail, rest)):
            if g is None:
                continue
            for _ in range(2):
                g.replay()
                done += n
        while done < w:
            (multi or tail).replay()
            done += cap if multi else rest
        torch.cuda.synchronize()

    return run, warm


# rotations of the layers in one graph of the timed loop (the remainder: one more graph)
GRAPH_ROTATIONS = 64


def kernel_times(torch, mol, wl, layers, cnt, ranks, steps, config):
    """Each stage kernel (and the align, the per-token adapter ids) alone in its own graphs,
    over the same rotation of layers; the dominant kernel against the HBM roofline and the
    first stage's shrink against the bf16 tensor peak."""
    peaks = measured_peaks()
    dev = layers[0].topk.device
    kern = {}

    def stage_call(L_, si, which):
        d = L_.stages[si]
        st = d["st"]
        if which == "shrink":
            return lambda: mol.mol_lora_shrink(d["x"], st.x_row_div, d["A"], st.stage.S,
                                               L_.routing, d["inter"], lora_ranks=L_.ranks_d,
                                               num_experts=wl.E)
        return lambda: mol.mol_lora_expand(d["inter"], d["B"], st.stage.S, wl.scale,
                                           L_.routing, d["out"], lora_ranks=L_.ranks_d,
                                           lora_scalings=L_.scal_d, num_experts=wl.E)

    def align_call(L_):
        return lambda: mol.mol_align_block_size(L_.routing.vtopk_ids, wl.V, wl.BM,
                                                routing=L_.routing, workspace=L_.ws)

    reps = 4  # launches per graph = layers x reps, back to back on one stream

    def per_launch_us(calls):
        g = capture(torch, lambda: [f() for _ in range(reps) for f in calls])
        n = max(20, min(steps, 2000) // (reps * len(calls)))
        return time_graphs(torch, [g], n, 3) * 1e3 / (reps * len(calls))

    kern["align"] = per_launch_us([align_call(L_) for L_ in layers])
    # per-token adapter ids of the batch: one request per token (decode) or
    # requests of 64 tokens, adapter slots of the layer's tokens
    req_len = 1 if wl.T <= 256 else 64
    nreq = (wl.T + req_len - 1) // req_len
    wi = torch.from_numpy(layers[0].li.lora_ids[::req_len].astype(np.int32)).to(dev)
    seg = torch.from_numpy(np.minimum(np.arange(nreq + 1) * req_len, wl.T).astype(np.int32)).to(dev)
    tok_ids = torch.empty(wl.T, dtype=torch.int32, device=dev)
    kern["token_lora_ids"] = per_launch_us(
        [lambda: mol.mol_token_lora_ids(wi, seg, wl.T, wl.L, layers[0].ranks_d, tok_ids)])
    for si, st in enumerate(wl.stages):
        for which in ("shrink", "expand"):
            kern[f"{which}_{st.name}"] = per_launch_us([stage_call(L_, si, which) for L_ in layers])
    # dominant kernel: the stage kernel with the most algorithmic bytes
    best = None
    for si, st in enumerate(wl.stages):
        sb = [L_.stage_bytes(si, *c) for L_, c in zip(layers, cnt)]
        for j, which in enumerate(("shrink", "expand")):
            b = float(np.mean([x[j] for x in sb]))
            if best is None or b > best[1]:
                best = (f"{which}_{st.name}", b)
    name, nbytes = best
    us = kern[name]
    achieved = nbytes / (us * 1e-6) / 1e9
    cap = None if ranks is not None else TRAFFIC.get((config, name))
    fresh = cap is not None and cap[3] == kernel_source_digest(cap[2])
    roof = dict(kernel=name, bound="hbm", achieved=round(achieved, 1), peak=peaks["hbm_gbs"],
                unit="GB/s", frac=round(achieved / peaks["hbm_gbs"], 4),
                traffic=cap[0] if fresh else None,
                traffic_launch_alg_bytes=cap[1] if fresh else None,
                traffic_note=None if fresh else (
                    "no ncu capture of this kernel and workload" if cap is None else
                    "kernel sources changed since the ncu capture"),
                bytes_per_launch=int(nbytes), us_per_launch=round(us, 3),
                peak_source=peaks["source"])
    # the first stage's shrink against the bf16 tensor peak (a real dense
    # contraction only when the routed blocks are full, as in `dense`)
    pairs_per_step = float(np.mean([c[0] for c in cnt]))
    st0 = wl.stages[0]
    sname = f"shrink_{st0.name}"
    flops = 2.0 * pairs_per_step * st0.K * st0.R
    tflops = flops / (kern[sname] * 1e-6) / 1e12
    tc_path = (st0.R % 64 == 0 and st0.K % 64 == 0 and wl.BM in (64, 128) and ranks is None
               and wl.numel >= 32 * min(wl.numel, wl.V))
    shrink_tensor = dict(kernel=sname, bound="tensor", achieved=round(tflops, 1),
                         peak=peaks["bf16_tflops"], unit="TFLOP/s",
                         frac=round(tflops / peaks["bf16_tflops"], 4),
                         path="tcgen05" if tc_path else "mma.sync",
                         flops_per_launch=flops, peak_source=peaks["source"])
    return kern, roof, shrink_tensor


def make_layers(torch, mol, wl, n, seed, dev, ranks=None, first=0):
    from synth import make_layer

    layers = [LayerState(wl, make_layer(wl, seed, layer=i), dev, mol, torch, ranks)
              for i in range(first, first + n)]
    for L_ in layers:
        L_.forward(mol)
    torch.cuda.synchronize()
    return layers


def layer_alg_bytes(L_, c):
    """Algorithmic HBM bytes of one layer (both stages and the align) for its counts c."""
    return sum(sum(L_.stage_bytes(si, *c)) for si in range(len(L_.stages))) + L_.align_bytes()


L2_BYTES = 129e6


def measure_workload(torch, mol, name, seed, dev, budget_s=0.15):
    """Short figures for one more workload, same method as the main line: layers rotated
    past L2, graphs warmed, then a CUDA-event-timed run of whole rotations."""
    from synth import WORKLOADS

    wl = WORKLOADS[name]
    layers = make_layers(torch, mol, wl, 1, seed, dev)
    # distinct layers so that one rotation moves over 3x the L2 (at most 8)
    nl = int(min(8, max(1, -(-3 * L2_BYTES // layer_alg_bytes(layers[0], layers[0].counts())))))
    layers += make_layers(torch, mol, wl, nl - 1, seed, dev, first=1)
    cnt = [L_.counts() for L_ in layers]
    pairs = float(np.mean([c[0] for c in cnt]))
    probe_run, probe_warm = layer_steps_timer(torch, mol, layers, nl)
    probe_warm(nl)
    ms_rotation = event_ms(torch, probe_run, 3)
    steps = nl * max(2, int(budget_s / max(ms_rotation * 1e-3, 1e-6)))
    run, warm = layer_steps_timer(torch, mol, layers, steps)
    warm(3)
    ms = event_ms(torch, run, 1) / steps
    kern, roof, shrink_tensor = kernel_times(torch, mol, wl, layers, cnt, None, steps, name)
    layer_bytes = float(np.mean([layer_alg_bytes(L_, c) for L_, c in zip(layers, cnt)]))
    peaks = measured_peaks()
    out = dict(workload=f"{name}: {wl.note}", steps=steps, layers_rotated=nl,
               us_per_layer=round(ms * 1e3, 3), value=round(pairs / (ms * 1e-3), 1), unit=UNIT,
               pairs_per_layer=pairs,
               layer_hbm=dict(bytes=int(layer_bytes),
                              achieved_gbs=round(layer_bytes / (ms * 1e-3) / 1e9, 1),
                              frac=round(layer_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)),
               kernels_us={k: round(v, 3) for k, v in kern.items()}, roofline=roof,
               shrink_tensor=shrink_tensor)
    del layers
    torch.cuda.empty_cache()
    return out


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import moe_lora_virtual_gb300 as mol
    from moe_lora_virtual_gb300.build import build_library
    from synth import WORKLOADS, make_layer

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    if rank == 0:
        build_library()
    if world > 1:
        dist.barrier()
    mol.library()

    wl = WORKLOADS[args.config]
    LayerState.routing_mode = args.routing_mode
    ranks = None
    if args.ranks:
        ranks = [int(v) for v in args.ranks.split(",")]
        if len(ranks) != wl.L:
            raise SystemExit(f"--ranks: expected {wl.L} values (one per adapter)")
    layers = [LayerState(wl, make_layer(wl, args.seed + 1000 * rank, layer=i), dev, mol, torch,
                         ranks) for i in range(args.layers)]
    for L_ in layers:
        L_.forward(mol)
    torch.cuda.synchronize()
    cnt = [L_.counts() for L_ in layers]
    pairs_per_step = float(np.mean([c[0] for c in cnt]))
    # kernels per layer, counted by the library over one eager layer
    n0 = mol.mol_launch_count()
    layers[0].forward(mol)
    torch.cuda.synchronize()
    launches_per_step = mol.mol_launch_count() - n0

    # A real decode step replays all MoE layers inside one graph; here one graph
    # holds the rotating layers back to back, and one more graph holds the first
    # K mod layers of them, so exactly K steps (layers) are timed and no step runs
    # as an isolated single-layer graph. Every graph the timed region replays is
    # replayed before it (at least twice), whatever --warmup is.
    run_steps, warm_steps = layer_steps_timer(torch, mol, layers, args.steps)

    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(local)
    try:
        gpu_id = "GPU-" + str(props.uuid)
    except Exception:
        pass
    clocks = ClockSampler(gpu_id)
    time.sleep(0.3)

    # ---- timed region: exactly K steps -----------------------------------------------
    warm_steps(args.warmup)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    ev0.record()
    run_steps()
    ev1.record()
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        dist.barrier()
    ms = ev0.elapsed_time(ev1) / args.steps
    time.sleep(0.15)
    clk = clocks.summary(t0, t1)
    clocks.stop()

    ms, pairs_all = combine_ranks(ms, pairs_per_step, dev if world > 1 else None)
    value = pairs_all / (ms * 1e-3)

    # ---- the same layers with the other routing mode (context, not the metric) -----------
    other_mode = 3 - args.routing_mode
    LayerState.routing_mode = other_mode
    g_other = capture(torch, lambda: [L_.forward(mol) for L_ in layers])
    LayerState.routing_mode = args.routing_mode
    for _ in range(3):
        g_other.replay()
    other_reps = max(1, 800 // len(layers))
    us_other = time_graphs(torch, [g_other], other_reps, 2) * 1e3 / len(layers)
    del g_other

    # ---- per-kernel timing (each kernel alone in its own graphs, same rotation) -------
    peaks = measured_peaks()
    kern, roof, shrink_tensor = {}, None, None
    if not args.no_kernels:
        kern, roof, shrink_tensor = kernel_times(torch, mol, wl, layers, cnt, ranks, args.steps,
                                                 args.config)

    layer_bytes = float(np.mean([sum(sum(L_.stage_bytes(si, *c)) for si in range(len(wl.stages)))
                                 + L_.align_bytes() for L_, c in zip(layers, cnt)]))

    # ---- end to end through the public API with host buffers -------------------------
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, torch, mol, wl, layers, pairs_per_step, world, dev)

    # ---- the other workloads, short (rank 0 of a single-process run) ------------------
    extra = {}
    names = [] if args.extra in ("", "none") else [n for n in args.extra.split(",") if n]
    if world == 1 and names:
        del layers
        torch.cuda.empty_cache()
        for name in names:
            if name == args.config:
                continue
            extra[name] = measure_workload(torch, mol, name, args.seed, dev)

    out = dict(metric=METRIC, value=round(value, 1), unit=UNIT, n_gpus=world, steps=args.steps,
               warmup=args.warmup, ms_per_step=round(ms, 6), us_per_layer=round(ms * 1e3, 3),
               higher_is_better=True, scaling="weak", vs_baseline=None, dtype="bf16",
               data="synthetic",
               config=dict(workload=f"{args.config}: {wl.note}", T=wl.T, E=wl.E, topk=wl.topk,
                           max_loras=wl.L, num_vexperts=wl.V, block_m=wl.BM,
                           stages=[f"{s.name} K={s.K} R={s.R} N={s.N}" for s in wl.stages],
                           pairs_per_layer=pairs_per_step, layers_rotated=args.layers,
                           adapter_ranks=ranks,
                           routing_mode=args.routing_mode,
                           l2="inputs larger than L2: steps rotate over distinct layers",
                           graph=f"graphs of {GRAPH_ROTATIONS * args.layers} layer steps "
                                 f"({GRAPH_ROTATIONS} rotations of the {args.layers} layers), "
                                 "the K mod that remainder in one more graph; every graph "
                                 "replayed at least twice before the timed region",
                           parallelism=f"replicas{world}"),
               layer_hbm=dict(bytes=int(layer_bytes),
                              achieved_gbs=round(layer_bytes / (ms * 1e-3) / 1e9, 1),
                              frac=round(layer_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)),
               us_per_layer_other_routing_mode={"routing_mode": other_mode,
                                                "us": round(us_other, 3)},
               kernels_us={k: round(v, 3) for k, v in kern.items()},
               roofline=roof, shrink_tensor=shrink_tensor, e2e=e2e,
               gpu_launches=launches_per_step * args.steps,
               clocks=dict(sm_mhz=clk["sm_mhz"], sm_max_mhz=clk["sm_max_mhz"],
                           reasons=clk["reasons"], samples=clk["samples"]),
               workloads=extra or None)
    if rank == 0 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline(args)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))


def run_e2e(args, torch, mol, wl, layers, pairs_per_step, world, dev):
    """Per step: one pinned host -> device copy of the step's inputs, the layer, one device ->
    host copy of its outputs; the rotating steps, E2E_ROUNDS times over, captured (copies
    included) in one graph whose copies run on their own streams, ordered by events, beside
    the compute of other steps.

    Each layer's inputs (top-k ids, adapter ids, every stage's activations and the output rows
    the expand updates) live in one device buffer, 256-byte aligned segments with the outputs
    last, mirrored by a pinned host buffer: a step moves the same bytes as per-tensor copies
    in one copy each way. The library receives ordinary tensor views of that buffer."""
    def rup(n):
        return (n + 255) // 256 * 256

    packs = []
    for L_ in layers:
        segs = [("topk", L_.topk), ("lora", L_.lora)]
        segs += [(f"x{i}", d["x"]) for i, d in enumerate(L_.stages)]
        segs += [(f"out{i}", d["out"]) for i, d in enumerate(L_.stages)]
        offs, total = {}, 0
        for name, t in segs:
            offs[name] = total
            total += rup(t.numel() * t.element_size())
        dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
        host_in = torch.empty(total, dtype=torch.uint8).pin_memory()

        def view(buf, name, t, offs=offs):
            nb = t.numel() * t.element_size()
            return buf[offs[name]:offs[name] + nb].view(t.dtype).view(t.shape)

        for name, t in segs:
            view(host_in, name, t).copy_(t.cpu())
        L_.topk, L_.lora = view(dev_buf, "topk", L_.topk), view(dev_buf, "lora", L_.lora)
        for i, d in enumerate(L_.stages):
            d["x"] = view(dev_buf, f"x{i}", d["x"])
            d["out"] = view(dev_buf, f"out{i}", d["out"])
        out_lo = offs["out0"]
        host_out = torch.empty(total - out_lo, dtype=torch.uint8).pin_memory()
        packs.append((dev_buf, host_in, host_out, out_lo))

    def step(L_, pk):
        dev_buf, host_in, host_out, out_lo = pk
        dev_buf.copy_(host_in, non_blocking=True)
        L_.forward(mol)
        host_out.copy_(dev_buf[out_lo:], non_blocking=True)

    # The rotating layers, E2E_ROUNDS times over, in one graph on three streams:
    # the inputs of a group of E2E_GROUP steps are copied in on s_in, the group's
    # layers run on the capturing stream once they have landed (one wait per group,
    # so the launches inside a group stay one chain of programmatic dependent
    # launches), and each step's outputs go back on s_out once its layer is done; the
    # copies of neighbouring steps and groups overlap the layers (whole-job
    # throughput). A layer's buffers are reused by the step one rotation later, whose
    # copy-in waits for this step's copy-out (a group is shorter than a rotation, so
    # no copy-in waits on a layer of its own group). More steps per graph spread the
    # first copy-in and the last copy-out over more steps, as a graph of a whole
    # model's layers would.
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    nl = len(layers)
    n_steps = E2E_ROUNDS * nl
    group = max(1, min(E2E_GROUP, nl))

    def all_steps():
        main = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(main)
        s_in.wait_event(start)
        s_out.wait_event(start)
        copied_out = []
        for k0 in range(0, n_steps, group):
            ks = range(k0, min(k0 + group, n_steps))
            landed = torch.cuda.Event()
            with torch.cuda.stream(s_in):
                for k in ks:
                    dev_buf, host_in = packs[k % nl][0], packs[k % nl][1]
                    if k >= nl:
                        s_in.wait_event(copied_out[k - nl])
                    dev_buf.copy_(host_in, non_blocking=True)
                landed.record(s_in)
            main.wait_event(landed)
            for k in ks:
                L_, (dev_buf, host_in, host_out, out_lo) = layers[k % nl], packs[k % nl]
                done, back = torch.cuda.Event(), torch.cuda.Event()
                L_.forward(mol)
                done.record(main)
                s_out.wait_event(done)
                with torch.cuda.stream(s_out):
                    host_out.copy_(dev_buf[out_lo:], non_blocking=True)
                    back.record(s_out)
                copied_out.append(back)
        main.wait_stream(s_in)
        main.wait_stream(s_out)

    graph = capture(torch, all_steps)
    replays = max(4, min(args.steps, 5000) // n_steps)
    ms = time_graphs(torch, [graph], replays, max(1, min(args.warmup, 50) // n_steps)) / n_steps
    steps = replays * n_steps
    # one step at a time (copy in, layer, copy out in order), graph per layer, for reference
    graphs = [capture(torch, lambda L_=L_, pk=pk: step(L_, pk)) for L_, pk in zip(layers, packs)]
    ms_serial = time_graphs(torch, graphs, min(args.steps, 5000), min(args.warmup, 50))
    bi = packs[0][1].numel()
    bo = packs[0][2].numel()
    # eager calls (no graph) for reference
    n_e = min(steps, 500)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n_e):
        step(layers[i % len(layers)], packs[i % len(packs)])
    torch.cuda.synchronize()
    ms_eager = (time.perf_counter() - t0) * 1e3 / n_e
    return dict(value=round(pairs_per_step * world / (ms * 1e-3), 1), unit=UNIT,
                h2d_bytes_per_step=int(bi), d2h_bytes_per_step=int(bo), ms_per_step=round(ms, 6),
                mode=f"graph replay of {n_steps} steps ({E2E_ROUNDS} rotations of the layers): per "
                     "step one pinned-host copy of the packed inputs, the mol_lora_forward calls, "
                     "one copy of the outputs back; copies on their own streams overlap "
                     f"neighbouring steps' compute; the layers wait for their inputs in groups of "
                     f"{group} steps",
                serial_value=round(pairs_per_step * world / (ms_serial * 1e-3), 1),
                serial_ms_per_step=round(ms_serial, 6),
                eager_value=round(pairs_per_step * world / (ms_eager * 1e-3), 1),
                eager_ms_per_step=round(ms_eager, 6), steps=steps)


# rotations of the layers inside the end-to-end graph
E2E_ROUNDS = 16
# steps whose inputs the layers wait for together (at most one rotation)
E2E_GROUP = 4


# traffic (dram bytes read + written) of one captured launch, with the algorithmic bytes of
# that same launch (the first layer of the workload, seed 0), the source file of the kernel
# and the digest of that file (with the shared device header) when it was captured, keyed by
# (workload, kernel). An entry whose digest differs from the current sources is stale and
# reported as null. Sources: the ncu summaries under profiles/.
TRAFFIC = {
    ("decode", "shrink_gate_up"): (35516416 + 0, 35506176, "mol_lora.cu", "bc84f759162e7992"),
    ("wide", "expand_down"): (41627648 + 37376, 43469824, "mol_lora.cu", "bc84f759162e7992"),
    ("wide1k", "expand_down"): (172901632 + 7897088, 184738816, "mol_lora.cu", "bc84f759162e7992"),
    ("ep", "shrink_gate_up"): (569616384 + 6232320, 572089984, "mol_lora.cu", "bc84f759162e7992"),
    ("dense", "expand_down"): (344882688 + 210326528, 612368384, "mol_expand_tc.cu", "7b034bb8c0282707"),
}


def kernel_source_digest(src: str) -> str:
    """sha256 (first 16 hex digits) of a kernel's source file and the shared device headers
    it includes (the tcgen05 helpers for the tensor-core kernels)."""
    import hashlib

    csrc = os.path.join(ROOT, "moe_lora_virtual_gb300", "csrc")
    h = hashlib.sha256()
    tc = ("mol_tc.cuh",) if src in ("mol_umma.cu", "mol_expand_tc.cu") else ()
    for f in (src, "mol_device.cuh") + tc:
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------------------- CPU (oracle)

def oracle_layer_sample(wl, li, blocks_per_step, step_idx, routing_cache):
    """Oracle on one step's sample of the layer: the routing, then both stages on a rotating
    window of routed blocks. Returns the number of (token, vexpert) pairs processed."""
    import oracle

    key = id(li)
    if key not in routing_cache:
        vt = oracle.virtual_topk(li.topk_ids, li.lora_ids, wl.E, wl.L).reshape(-1)
        s, e, n = oracle.align_block_size(vt, wl.V, wl.BM)
        real = np.nonzero(e[: n // wl.BM] >= 0)[0]
        routing_cache[key] = (s, e, n, real)
    s, e, n, real = routing_cache[key]
    if blocks_per_step >= real.size:
        pick = real
    else:
        start = (step_idx * blocks_per_step) % real.size
        pick = np.take(real, np.arange(start, start + blocks_per_step), mode="wrap")
    e_s = np.full_like(e, -1)
    e_s[pick] = e[pick]
    pairs = 0
    for t in pick:
        ids = s[t * wl.BM:(t + 1) * wl.BM]
        pairs += int(np.sum(ids < wl.numel))
    for st in li.stages:
        if not hasattr(st, "_host_out0"):
            st._host_out0 = st.out0.host_all()
        inter = oracle.lora_shrink(st.x, st.x_row_div, st.A, s, e_s, n, wl.BM, wl.numel,
                                   np.zeros((wl.numel, st.stage.R), np.float32))
        oracle.lora_expand(inter, st.B, st.stage.S, st.stage.r, st.stage.Ns, wl.scale, None, s,
                           e_s, n, wl.BM, wl.numel, st._host_out0)
    return pairs


def cpu_worker(args):
    """Runs in a child process with one BLAS thread: the oracle on a bounded sample."""
    from synth import WORKLOADS, make_layer

    wl = WORKLOADS[args.config]
    li = make_layer(wl, args.seed, layer=0)
    cache = {}
    oracle_layer_sample(wl, li, 4, 0, cache)          # warm: routing + conversions
    t0 = time.perf_counter()
    pairs = 0
    k = 0
    while time.perf_counter() - t0 < args.cpu_budget:
        pairs += oracle_layer_sample(wl, li, 1 << 30, k, cache)
        k += 1
    dt = time.perf_counter() - t0
    print(json.dumps(dict(pairs=pairs, seconds=dt, layers=k)))


def cpu_baseline(args):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-worker", "--config", args.config,
           "--seed", str(args.seed), "--cpu-budget", "15"]
    try:
        res = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
        d = json.loads(res.stdout.strip().splitlines()[-1])
    except Exception as exc:  # report, never fail the GPU line
        return dict(value=None, unit=UNIT, cores=1, kind="oracle", sample=f"failed: {exc}")
    return dict(value=round(d["pairs"] / d["seconds"], 1), unit=UNIT, cores=1, kind="oracle",
                sample=f"{d['layers']} whole {args.config} layers (all routed blocks, both stages) "
                       f"in {d['seconds']:.1f} s, numpy float64, 1 BLAS thread")


def run_reference(args):
    """The CPU oracle timed on the same workload and metric (the reference arm)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return
    from synth import WORKLOADS, make_layer

    wl = WORKLOADS[args.config]
    li = make_layer(wl, args.seed, layer=0)
    cache = {}
    # calibrate: blocks per step so that warmup + steps stay within ~120 s
    t0 = time.perf_counter()
    oracle_layer_sample(wl, li, 1, 0, cache)
    t_first = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle_layer_sample(wl, li, 4, 1, cache)
    per_block = max((time.perf_counter() - t0) / 4, 1e-5)
    budget = 120.0 / max(1, args.steps + args.warmup)
    bps = int(max(1, min(1 << 20, budget / per_block)))
    for i in range(args.warmup):
        oracle_layer_sample(wl, li, bps, i, cache)
    t0 = time.perf_counter()
    pairs = 0
    for i in range(args.steps):
        pairs += oracle_layer_sample(wl, li, bps, args.warmup + i, cache)
    dt = time.perf_counter() - t0
    value = pairs / dt
    nthreads = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS") or str(os.cpu_count())
    out = dict(impl="reference", metric=METRIC, value=round(value, 1), unit=UNIT, n_gpus=world,
               steps=args.steps, warmup=args.warmup, ms_per_step=round(dt * 1e3 / args.steps, 4),
               higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
               data="synthetic",
               config=dict(workload=f"{args.config}: {wl.note}", blocks_per_step=bps,
                           routing_s=round(t_first, 4)),
               cpu_baseline=dict(value=round(value, 1), unit=UNIT, cores=int(nthreads),
                                 kind="oracle",
                                 sample=f"{bps} routed blocks of one {args.config} layer per step"),
               e2e=dict(value=round(value, 1), unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(out))


def main(argv=None):
    args = parse_args(argv)
    if args.cpu_worker:
        cpu_worker(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
