#!/usr/bin/env python
"""Throughput of causal shared-offset sparse attention, forward + backward.

One step = forward and backward (dQ, dK, dV, dalpha/dtheta) of a 16-layer
stack of interpolated shared-offset sparse attention over one batch:
B = 32 sequences of T = 1024 tokens, 8 query / 2 KV heads, head dim 64,
bf16 I/O, window W = 8, Fibonacci rungs (K = 15) scaled by the linear layer
schedule alpha_l = 0.5 + l/15, RoPE theta 1e4.  Every layer has its own
independently drawn Q, K, V, dO (N(0, 1), seeded), so each step streams
16 distinct layers' tensors (2.6 GB, far above the 129 MB L2: no L2 flush is
needed between steps).

The timed region replays the step captured as one CUDA graph (single rank;
multi-rank runs time the eager step with its all-reduce); a separate eager
pass with CUDA events around every library launch gives the per-kernel times
behind the roofline, and the eager step without those events is reported too.

Prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle on a
bounded sample of the same workload instead.  ``--mode decode`` measures the
integer-path decode step instead (one new token per sequence through the
16-layer stack against a T = 16384 cache); its JSON line names its own metric.

Launch: python bench.py [--gpus N --steps K --warmup W]; N > 1 under
torch.distributed.run (one rank per GPU, weak scaling: every rank runs its
own batch; the per-layer dtheta values are summed across ranks with one
all-reduce per step, as data-parallel training of theta would).
"""
from __future__ import annotations

import os

# The CPU oracle legs report a single core: keep BLAS / OpenMP pools at one
# thread (set before numpy is first imported).
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fwd+bwd sparse-attn tokens/s at T=1024 GQA bf16; HBM GB/s vs GB300 peak"
B, T, HQ, HKV, D = 32, 1024, 8, 2, 64
LAYERS = 16  # --layers changes it for profiling captures of a smaller case
ORDER = "training"  # --order: "training" (all forwards, then backwards last to first) or "layerwise"
FIB = [1, 2, 3, 5, 8, 13, 21, 34, 55, 89, 144, 233, 377, 610, 987]
ROPE = 1e4
SEED = 0
# unique bytes per token per layer, bf16: Q, O, dO, dQ (Hq heads) + K, V, dK, dV (Hkv heads)
UNIQUE_BYTES_PER_TOKEN = 2 * D * (4 * HQ + 4 * HKV)
# algorithmic bytes per token of each kernel (bf16, 8/2 heads): the method's
# tensors it must read or write once
KERNEL_BYTES_PER_TOKEN = {"fwd": 2 * D * (2 * HQ + 2 * HKV),   # Q, O, K, V
                          "bwd_q": 2 * D * (4 * HQ + 2 * HKV),  # Q, O, dO, dQ, K, V
                          "bwd_kv": 2 * D * (2 * HQ + 2 * HKV)}  # Q, dO, dK, dV
# algorithmic flop per (query head, key) pair, per kernel; D = 64
FLOP_PER_PAIR = {"fwd": 4 * D, "bwd_q": 6 * D, "bwd_kv": 4 * D}
FLOP_PER_RUNG_PAIR_DALPHA = 4 * D  # q.(k0 - k1) and dO.(v0 - v1)


def hbm_peak():
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        return json.load(open(pk))["hbm_gbs"], "MEASURED_PEAKS.json hbm_gbs (of measured)"
    return 6800.0, "fallback 6.8 TB/s (of fallback)"


SCHED_L = 16  # the schedules are defined over the 16-layer stack


def alphas(schedule: str):
    if schedule == "linear":
        return [0.5 + l / (SCHED_L - 1) for l in range(SCHED_L)]
    if schedule == "coprime":
        lin = [0.5 + l / (SCHED_L - 1) for l in range(SCHED_L)]
        return [lin[(7 * l) % SCHED_L] for l in range(SCHED_L)]
    if schedule == "fixed":
        return [1.0] * SCHED_L
    raise ValueError(schedule)


def layer_ids():
    """All 16 layers, or (profiling captures) LAYERS of them from layer 7 on."""
    return list(range(SCHED_L)) if LAYERS == SCHED_L else [(7 + j) % SCHED_L for j in range(LAYERS)]


def pair_counts(alpha: float, W: int, base=None):
    """(query, key) pairs per (b, query head) and how many are rung pairs.

    Counts the plain definition: window keys min(W, i) + 1 and a rung with
    ceil(alpha f) = c and alpha f > W reaching queries i >= c (f over the base
    list, Fibonacci by default)."""
    import math

    win = sum(min(W, i) + 1 for i in range(T))
    rung = 0
    for f in (FIB if base is None else base):
        d = alpha * f
        if d <= W:
            continue
        c = math.ceil(d)
        rung += max(0, T - c)
    return win + rung, rung


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) >= 9:
                rows.append(p)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in rows for j in range(4) if r[5 + j].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


def rank_seed(rank: int) -> int:
    """Input seed of a rank: every rank draws its own batch (weak scaling)."""
    import sfa_inputs as si

    return si.mix_seed(SEED, 1000 + rank)


def allreduce_dtheta(dadt_per_layer, out):
    """Sum the per-layer dL/dtheta over ranks (data-parallel theta): gathers
    element 1 of each layer's (dalpha, dtheta) pair into `out` and all-reduces
    it.  The only collective of the benchmark."""
    import torch.distributed as dist

    for l, d in enumerate(dadt_per_layer):
        out[l] = d[1]
    dist.all_reduce(out)
    return out


def kernel_traffic(kind: str):
    """Per-launch DRAM bytes of `kind` from the committed ncu summary, or None
    when there is none or the kernel source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", f"{kind}_traffic.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    src = os.path.join(ROOT, "static_offset_sparse_gb300", "csrc", vals.get("source", ""))
    if not os.path.isfile(src):
        return None
    if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != vals.get("source_sha256_16"):
        return None
    try:
        return float(vals["bytes_per_launch_full"])
    except (KeyError, ValueError):
        return None


class Layer:
    """One layer's device tensors and its prebuilt C-ABI descriptor."""

    def __init__(self, sfa, lib, x, alpha, W, dev, base=None):
        import ctypes as C
        import torch

        self.x = x
        self.alpha = alpha
        self.o = torch.empty_like(x["q"])
        self.lse = torch.empty((B, HQ, T), dtype=torch.float32, device=dev)
        self.dq = torch.empty_like(x["q"])
        self.dk = torch.empty_like(x["k"])
        self.dv = torch.empty_like(x["v"])
        self.dadt = torch.zeros((2,), dtype=torch.float64, device=dev)
        # the layer's rotated keys: one rotation per step serves forward and
        # backward (kept like a saved activation)
        self.k_rot = torch.empty_like(x["k"])
        self.desc = sfa.make_desc(x["q"], x["k"], W=W, alpha=alpha,
                                  base=FIB if base is None else base, rope_theta=ROPE,
                                  k_rot=self.k_rot)
        self.nws = max(1, sfa.workspace_size(self.desc, True, True),
                       sfa.workspace_size(self.desc, True, False))
        self.ws = torch.empty((self.nws,), dtype=torch.uint8, device=dev)
        P = lambda t: C.c_void_p(t.data_ptr())  # noqa: E731
        self.rargs = (C.byref(self.desc), P(x["k"]), P(self.k_rot))
        self.fargs = (C.byref(self.desc), P(x["q"]), P(x["k"]), P(x["v"]), P(self.o), P(self.lse),
                      P(self.ws), self.nws)
        self.bargs = (C.byref(self.desc), P(x["q"]), P(x["k"]), P(x["v"]), P(self.o), P(self.lse),
                      P(x["do"]), P(self.dq), P(self.dk), P(self.dv), P(self.dadt), P(self.ws),
                      self.nws)
        self.lib = lib

    def run_fwd(self, stream):
        rc = self.lib.sfa_rope_keys(*self.rargs, stream)
        rc = rc or self.lib.sfa_forward(*self.fargs, stream)
        if rc:
            raise RuntimeError(f"libsfa status {rc}")

    def run_bwd(self, stream):
        rc = self.lib.sfa_backward(*self.bargs, stream)
        if rc:
            raise RuntimeError(f"libsfa status {rc}")

    def run(self, stream):
        self.run_fwd(stream)
        self.run_bwd(stream)


def run_layers(layers, stream):
    """One training step's attention calls in a training step's order: every
    layer's forward (its keys rotated once, kept like a saved activation),
    then the backwards from the last layer to the first.  With ORDER ==
    "layerwise" each layer's backward follows its own forward instead (then
    the backward finds that layer's tensors still in L2)."""
    if ORDER == "layerwise":
        for L in layers:
            L.run(stream)
        return
    for L in layers:
        L.run_fwd(stream)
    for L in reversed(layers):
        L.run_bwd(stream)


def gpu_arm(args, rank, world, dev):
    import ctypes as C
    import torch
    import torch.distributed as dist

    import sfa_inputs as si
    import static_offset_sparse_gb300 as sfa
    from static_offset_sparse_gb300._lib import _lib

    lib = _lib()
    al = alphas(args.schedule)
    layers = []
    for l in layer_ids():
        x = si.make_qkvdo_device(B, T, HQ, HKV, D, "bf16", rank_seed(rank), dev, layer=l)
        layers.append(Layer(sfa, lib, x, al[l], args.W, dev))
    stream = torch.cuda.current_stream()
    sp = C.c_void_p(stream.cuda_stream)
    dtheta = torch.zeros((LAYERS,), dtype=torch.float64, device=dev)

    def step():
        run_layers(layers, sp)
        if world > 1:
            allreduce_dtheta([L.dadt for L in layers], dtheta)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert sfa.get_device_status() == 0
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(run, n):
        barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(n):
            run()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return ev0.elapsed_time(ev1) / n

    # 1) per-kernel breakdown for the roofline: library events around every
    #    launch (they add gaps, so this pass does not give the headline)
    n_k = min(args.steps, 20)
    sfa.timing_enable(True)
    sfa.timing_read()  # drop anything recorded before
    timed(step, n_k)
    kt = sfa.timing_read()
    sfa.timing_enable(False)
    # 2) eager step without events (one host call per layer and direction)
    ms_eager = timed(step, min(args.steps, 50))
    # 3) headline: the step as one CUDA graph (single rank; the multi-rank
    #    step keeps its all-reduce eager)
    run = step
    graphed = world == 1
    if graphed:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run_layers(layers, C.c_void_p(torch.cuda.current_stream().cuda_stream))
        run = graph.replay
        for _ in range(args.warmup):
            run()
        torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    clocks.start()
    ms = timed(run, args.steps)
    clk = clocks.stop()
    assert sfa.get_device_status() == 0
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    per_step_launches = sum(c for _, c in kt.values()) / n_k
    launches = int(round(per_step_launches * args.steps))
    kt = {k: (v[0] / n_k * args.steps, v[1] / n_k * args.steps) for k, v in kt.items()}

    # roofline of the dominant kernel (largest summed device time), HBM view:
    # algorithmic bytes per launch / mean launch time vs the measured copy peak
    dom = max(("fwd", "bwd_q", "bwd_kv"), key=lambda k: kt[k][0])
    per_launch_ms = kt[dom][0] / max(1, kt[dom][1])
    bytes_per_launch = KERNEL_BYTES_PER_TOKEN[dom] * B * T
    achieved = bytes_per_launch / (per_launch_ms * 1e-3) / 1e9
    peak, src = hbm_peak()
    flops = 0.0
    for L in layers:
        pairs, rung_pairs = pair_counts(L.alpha, args.W)
        f = pairs * FLOP_PER_PAIR[dom] + (rung_pairs * FLOP_PER_RUNG_PAIR_DALPHA if dom == "bwd_q" else 0)
        flops += f * B * HQ
    useful_tflops = flops / len(layers) / (per_launch_ms * 1e-3) / 1e12
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": kernel_traffic(dom),
                "peak_source": src, "algorithmic_bytes_per_launch": bytes_per_launch,
                "per_launch_ms": round(per_launch_ms, 4),
                "useful_tflops": round(useful_tflops, 2),
                "kernel_ms_per_step": {k: round(v[0] / args.steps, 4) for k, v in kt.items() if v[1]},
                "kernel_times": f"CUDA events around each launch, eager pass of {n_k} steps"}
    roofline["step_modes"] = {"headline": "CUDA graph of the 16-layer step" if graphed else "eager",
                              "eager_ms_per_step": round(ms_eager, 4)}
    return layers, ms, clk, launches, roofline


def e2e_arm(layers, steps, warmup, world, dev):
    """Same step through the C ABI with host buffers: every step copies each
    layer's Q, K, V, dO from pinned host memory and reads dQ, dK, dV and
    (dalpha, dtheta) back, inside the timed region.  Copies and compute run
    on three streams (host to device, compute, device to host) ordered by
    per-layer events, so one layer's copies overlap another layer's kernels;
    a layer's buffers are refilled only after its previous outputs were read
    back, and recomputed only after its inputs arrived.  The host's own time
    to issue a step (copies, events and the C-ABI calls) is reported beside
    it: when it exceeds the link's time, the host bounds the step."""
    import ctypes as C
    import torch
    import torch.distributed as dist

    host_in = [{n: t.to("cpu").pin_memory() for n, t in L.x.items()} for L in layers]
    host_out = [{n: torch.empty(getattr(L, n).shape, dtype=getattr(L, n).dtype).pin_memory()
                 for n in ("dq", "dk", "dv", "dadt")} for L in layers]
    h2d = sum(t.numel() * t.element_size() for h in host_in for t in h.values())
    d2h = sum(t.numel() * t.element_size() for h in host_out for t in h.values())
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    sp = C.c_void_p(s_cmp.cuda_stream)
    n = len(layers)
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_done = [torch.cuda.Event() for _ in range(n)]
    ev_out = [torch.cuda.Event() for _ in range(n)]
    first = [True]

    def step(compute=True):
        for l, (L, hi) in enumerate(zip(layers, host_in)):
            with torch.cuda.stream(s_in):
                if not first[0]:
                    s_in.wait_event(ev_out[l])  # previous outputs read back, inputs consumed
                for nm, t in hi.items():
                    L.x[nm].copy_(t, non_blocking=True)
                ev_in[l].record(s_in)
        for l, L in enumerate(layers):
            s_cmp.wait_event(ev_in[l])
            if compute:
                L.run(sp)
            ev_done[l].record(s_cmp)
        for l, (L, ho) in enumerate(zip(layers, host_out)):
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[l])
                for nm, t in ho.items():
                    t.copy_(getattr(L, nm), non_blocking=True)
                ev_out[l].record(s_out)
        first[0] = False

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    t_issue = (time.perf_counter() - t0) / steps
    torch.cuda.synchronize()
    el = (time.perf_counter() - t0) / steps
    # the same copies with the kernels left out: the host link's own time for
    # a step's bytes, the floor of the end-to-end step
    t0 = time.perf_counter()
    for _ in range(3):
        step(compute=False)
    torch.cuda.synchronize()
    el_copy = (time.perf_counter() - t0) / 3
    if world > 1:
        t = torch.tensor([el, el_copy, t_issue], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        el, el_copy, t_issue = float(t[0].item()), float(t[1].item()), float(t[2].item())
    # what the step waits for: the link (within 10% of the copies alone), the
    # host issuing the work (within 10% of its issue time), or neither
    bound = ("host link" if el <= 1.1 * el_copy else
             "host issue" if el <= 1.1 * t_issue else "unexplained: neither link nor issue")
    return {"value": round(world * B * T / el, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(el * 1e3, 3), "steps": steps,
            "copies_only_ms_per_step": round(el_copy * 1e3, 3),
            "host_issue_ms_per_step": round(t_issue * 1e3, 3),
            "host_link_gbs": round((h2d + d2h) / el_copy / 1e9, 1),
            "bound": bound,
            "overlap": "host-to-device, compute and device-to-host streams, per-layer events "
                       "(copies_only_ms_per_step: the same copies without the kernels; "
                       "host_issue_ms_per_step: the host's time to issue a step)"}


def oracle_step_sample(schedule: str, W: int, nb: int, layer: int):
    """One oracle fwd+bwd of `layer` for the first nb sequences (both KV heads)."""
    import oracle as o
    import sfa_inputs as si

    a = alphas(schedule)[layer]
    x = si.make_qkvdo(nb, T, HQ, HKV, D, "bf16", rank_seed(0), layer=layer)
    slots = o.interp_slots(FIB, a, W)
    t0 = time.perf_counter()
    o.forward(x["q"], x["k"], x["v"], slots, ROPE)
    o.backward(x["q"], x["k"], x["v"], x["do"], slots, ROPE, alpha=a)
    return time.perf_counter() - t0


def cpu_model() -> str:
    """The host CPU's model name from /proc/cpuinfo (x86 'model name', Arm
    implementer/part codes), else the platform's processor string."""
    import platform

    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        info = []
    for line in info:
        if line.lower().startswith("model name"):
            return line.split(":", 1)[1].strip()
    imp = [l.split(":", 1)[1].strip() for l in info if l.startswith("CPU implementer")]
    part = [l.split(":", 1)[1].strip() for l in info if l.startswith("CPU part")]
    if imp and part:
        return f"{platform.machine()} (CPU implementer {imp[0]}, part {part[0]})"
    return platform.processor() or platform.machine()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_unit(job):
    """Pool worker: one oracle (layer, sequence) unit; returns its seconds."""
    schedule, W, layer = job
    return oracle_step_sample(schedule, W, 1, layer)


def cpu_baseline(schedule: str, W: int, budget_s: float = 10.0):
    """The oracle as it stands on this host, on a bounded sample of the
    workload, scaled to the 16-layer step (tokens / (16 x seconds per
    layer-sequence)).

    Single thread: one sequence of one layer at a time, cycling through the 16
    layers' alphas, until ~budget_s of CPU work.  All cores: one process per
    host core (spawned: this process may hold a CUDA context), each running
    whole (layer, sequence) units, each process's numpy on one thread; after
    one warm-up unit per process, a batch of 4 units per process is timed by
    the wall clock."""
    spent, n = 0.0, 0
    while spent < budget_s and n < 16 * 32:
        spent += oracle_step_sample(schedule, W, 1, n % SCHED_L)
        n += 1
    tok_s = n * T / (spent * SCHED_L)
    out = {"value": round(tok_s, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
           "cpu_model": cpu_model(),
           "sample": f"fp64 numpy oracle, {n} (layer, sequence) units of {T} tokens cycling over the "
                     f"16 layers' alphas, W={W}, fwd+bwd incl. dtheta, single thread; {spent:.1f} s; "
                     "scaled to the 16-layer step"}
    cores = host_cores()
    if cores > 1:
        import multiprocessing as mp

        ctx = mp.get_context("spawn")
        with ctx.Pool(cores) as pool:
            pool.map(_oracle_unit, [(schedule, W, l % SCHED_L) for l in range(cores)], chunksize=1)
            units = 4 * cores
            t0 = time.perf_counter()
            pool.map(_oracle_unit, [(schedule, W, l % SCHED_L) for l in range(units)], chunksize=1)
            wall = time.perf_counter() - t0
        out["all_cores"] = {
            "value": round(units * T / (wall * SCHED_L), 3), "unit": "tokens/s", "cores": cores,
            "kind": "oracle", "cpu_model": out["cpu_model"],
            "sample": f"fp64 numpy oracle, {units} (layer, sequence) units over {cores} spawned "
                      f"processes (one thread each), wall {wall:.2f} s after one warm-up unit per "
                      "process; scaled to the 16-layer step"}
    return out


def reference_arm(args):
    """--impl reference: the fp64 oracle timed on this host, each step one
    sequence of one layer (bounded sample).  ms_per_step is that sample's own
    time, so steps x ms_per_step is the time this arm actually ran; value is
    the throughput scaled to the workload (B sequences x 16 layers per step),
    with the scale stated in sample_scale."""
    for _ in range(args.warmup):
        oracle_step_sample(args.schedule, args.W, 1, 7)
    ts = [oracle_step_sample(args.schedule, args.W, 1, 7) for _ in range(args.steps)]
    sec = sum(ts) / len(ts)
    val = T / (sec * LAYERS)
    cb = {"value": round(val, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
          "cpu_model": cpu_model(),
          "sample": f"fp64 numpy oracle, one {T}-token sequence of layer 7 per step, W={args.W}, "
                    "fwd+bwd incl. dtheta, single thread; scaled to 16 layers"}
    return {"metric": METRIC, "impl": "reference", "value": round(val, 3), "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "sample_scale": {"per_step": f"1 sequence x 1 layer of the workload's {B} sequences x "
                                         f"{LAYERS} layers",
                             "factor": B * LAYERS,
                             "workload_ms_per_step": round(sec * 1e3 * B * LAYERS, 1)},
            "config": config(args), "cpu_baseline": cb,
            "e2e": {"value": round(val, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ---- decode mode (--mode decode): one new token per sequence -------------
DEC_T = 16384  # cache capacity: the longest integer-path sequence of the configs
DEC_METRIC = ("decode tokens/s: one query per sequence through a 16-layer staggered integer "
              "stack (W=8, Fibonacci K=15, alpha_l rounded), cache T=16384, GQA 8/2 bf16")


def dec_distances(alpha: float, W: int):
    """Integer-path key set of one layer: {0..W} and round-half-even(alpha f)."""
    return sorted(set(range(W + 1)) | {round(alpha * f) for f in FIB})


DEC_STEPS_MAX = 1024  # positions advance one per step; starts leave room for this many


def dec_positions(Bd: int):
    """First positions of the Bd sequences: seeded, uniform in [T/2, T - 1024)."""
    import sfa_inputs as si

    u = si.uniform(si.mix_seed(9, Bd), Bd)
    span = DEC_T // 2 - DEC_STEPS_MAX
    return [DEC_T // 2 + int(x * span) for x in u]


class DecLayer:
    """One layer's caches, query rows and prebuilt decode descriptor."""

    def __init__(self, sfa, lib, l, alpha, W, Bd, pos_dev, dev):
        import ctypes as C
        import sfa_inputs as si

        def gen(tid, shape):
            n = 1
            for x in shape:
                n *= x
            return si.normal_device(si.mix_seed(7, l, tid), n, dev).view(*shape).to(__import__("torch").bfloat16)

        self.q = gen(1, (Bd, HQ, D)).contiguous()
        self.k = gen(2, (Bd, HKV, DEC_T, D)).contiguous()
        self.v = gen(3, (Bd, HKV, DEC_T, D)).contiguous()
        self.o = self.q.new_empty(self.q.shape)
        self.lse = self.q.new_empty((Bd, HQ), dtype=__import__("torch").float32)
        self.dist = dec_distances(alpha, W)
        self.desc = sfa.make_desc(self.q, self.k, dist=self.dist, rope_theta=1e4)
        self.lib, self.pos = lib, pos_dev  # [steps, Bd]: row r = positions of step r
        self.pre = [C.byref(self.desc)] + [C.c_void_p(t.data_ptr()) for t in (self.q, self.k, self.v)]
        self.posp = [C.c_void_p(pos_dev[r].data_ptr()) for r in range(pos_dev.shape[0])]
        self.post = [C.c_void_p(self.o.data_ptr()), C.c_void_p(self.lse.data_ptr())]

    def run(self, sp, r):
        self.run_ptr(sp, self.posp[r])

    def run_ptr(self, sp, posp):
        rc = self.lib.sfa_decode_int(*self.pre, posp, *self.post, sp)
        if rc:
            raise RuntimeError(f"sfa_decode_int failed: {rc}")


def dec_bytes_per_step(layers, Bd):
    """HBM bytes one 16-layer decode step must move: every gathered K and V
    row (bf16, 128 B) of every (sequence, KV head), the query rows in and the
    output rows and LSE out."""
    tot = 0
    for L in layers:
        tot += Bd * HKV * len(L.dist) * 2 * D * 2 + Bd * HQ * D * 2 * 2 + Bd * HQ * 4
    return tot


def decode_arm(args, dev):
    import ctypes as C
    import torch

    import static_offset_sparse_gb300 as sfa
    from static_offset_sparse_gb300._lib import _lib

    Bd = args.decode_batch
    n_e2e = min(args.steps, 50)
    n_total = args.warmup + args.steps + n_e2e + 1
    if n_total > DEC_STEPS_MAX:
        raise SystemExit(f"--mode decode: at most {DEC_STEPS_MAX} steps in all")
    pos0 = torch.tensor(dec_positions(Bd), dtype=torch.int32)
    pos_dev = (pos0[None, :] + torch.arange(n_total, dtype=torch.int32)[:, None]).to(dev).contiguous()
    al = alphas(args.schedule)
    layers = [DecLayer(sfa, _lib(), l, al[l], args.W, Bd, pos_dev, dev) for l in layer_ids()]
    stream = torch.cuda.current_stream()
    sp = C.c_void_p(stream.cuda_stream)

    ctr = [0]

    def step():  # every sequence advances one position per step
        r = ctr[0]
        ctr[0] += 1
        for L in layers:
            L.run(sp, r)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert sfa.get_device_status() == 0
    sfa.timing_enable(True)
    sfa.timing_read()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    kt = sfa.timing_read()
    sfa.timing_enable(False)
    ms_eager = ev0.elapsed_time(ev1) / args.steps
    per_launch_eager = kt["decode"][0] / max(1, kt["decode"][1])
    eager_launches = int(sum(c for _, c in kt.values()))

    # The same step as one CUDA graph (how a decode loop amortises launch
    # cost): advance every position by one, then the 16 decode calls.
    pos_cur = pos_dev[ctr[0]].clone()
    cur_p = C.c_void_p(pos_cur.data_ptr())
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm the capture path (torch requires it)
        pos_cur.add_(0)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cs = C.c_void_p(torch.cuda.current_stream().cuda_stream)
        pos_cur.add_(1)
        for L in layers:
            L.run_ptr(cs, cur_p)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    clocks.start()
    ev0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert sfa.get_device_status() == 0
    ms = ev0.elapsed_time(ev1) / args.steps
    per_launch_ms = ms / len(layers)
    nbytes = dec_bytes_per_step(layers, Bd)
    peak, src = hbm_peak()
    achieved = nbytes / len(layers) / (per_launch_ms * 1e-3) / 1e9
    # end to end: each step copies every layer's query rows in from pinned host
    # memory and its output rows and LSE back
    hq = [L.q.to("cpu").pin_memory() for L in layers]
    ho = [(torch.empty(L.o.shape, dtype=L.o.dtype).pin_memory(),
           torch.empty(L.lse.shape, dtype=L.lse.dtype).pin_memory()) for L in layers]

    def step_e2e():
        r = ctr[0]
        ctr[0] += 1
        for L, a, (bo, bl) in zip(layers, hq, ho):
            L.q.copy_(a, non_blocking=True)
            L.run(sp, r)
            bo.copy_(L.o, non_blocking=True)
            bl.copy_(L.lse, non_blocking=True)

    step_e2e()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n_e2e - 1):
        step_e2e()
    torch.cuda.synchronize()
    el = (time.perf_counter() - t0) / (n_e2e - 1)
    keys = sorted({len(L.dist) for L in layers})
    out = {"metric": DEC_METRIC, "value": round(Bd / (ms * 1e-3), 1), "unit": "tokens/s",
           "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic: seeded N(0,1) caches and query rows per layer",
           "config": {"workload": f"integer decode, {len(layers)} layers (alpha_l {args.schedule}, "
                                  f"rounded), W={args.W}: B={Bd} sequences starting at positions in "
                                  f"[{DEC_T // 2}, {DEC_T - DEC_STEPS_MAX}), one position further each "
                                  f"step, cache T={DEC_T}, Hq={HQ} Hkv={HKV} "
                                  f"D={D}, RoPE 1e4, {keys[0]}-{keys[-1]} keys per query",
                      "global_batch": Bd, "seq_len": DEC_T, "layers": len(layers),
                      "parallelism": "dp1",
                      "l2": "caches 4.3 GB exceed L2; positions advance each step, so a step's "
                            "rung rows are new while most window rows were read the step before"},
           "roofline": {"bound": "hbm", "kernel": "decode", "achieved": round(achieved, 1),
                        "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                        "traffic": None, "peak_source": src,
                        "algorithmic_bytes_per_launch": nbytes // len(layers),
                        "per_launch_ms": round(per_launch_ms, 4),
                        "note": "per-launch time = graph step / layers (includes the position "
                                "advance); the step is latency-bound, not bandwidth-bound"},
           "eager": {"value": round(Bd / (ms_eager * 1e-3), 1), "unit": "tokens/s",
                     "ms_per_step": round(ms_eager, 4), "per_launch_ms": round(per_launch_eager, 4),
                     "gpu_launches": eager_launches,
                     "note": "one host call per layer and step (ctypes), no graph"},
           "gpu_launches": len(layers) * args.steps, "clocks": clk,
           "e2e": {"value": round(Bd / el, 1), "unit": "tokens/s",
                   "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hq),
                   "d2h_bytes_per_step": sum(a.numel() * a.element_size() + b.numel() * b.element_size()
                                             for a, b in ho),
                   "ms_per_step": round(el * 1e3, 3), "steps": n_e2e}}
    if args.cpu_budget > 0:
        out["cpu_baseline"] = dec_cpu_baseline(args, min(args.cpu_budget, 10.0))
    return out


def dec_cpu_baseline(args, budget_s: float):
    """The oracle decode as it stands, timed on this host: one sequence of
    layer 7 (seeded host cache of the workload's shape) per sample, until
    ~budget_s of oracle work; scaled to the 16-layer step."""
    import oracle
    import sfa_inputs as si

    l = 7
    pos_first = dec_positions(args.decode_batch)[0]
    dist = dec_distances(alphas(args.schedule)[l], args.W)
    q = si.make_tensor((1, HQ, D), "bf16", si.mix_seed(7, l, 1))
    k = si.make_tensor((1, HKV, DEC_T, D), "bf16", si.mix_seed(7, l, 2))
    v = si.make_tensor((1, HKV, DEC_T, D), "bf16", si.mix_seed(7, l, 3))
    spent, n = 0.0, 0
    while spent < budget_s and n < 400:
        t0 = time.perf_counter()
        oracle.decode(q, k, v, [pos_first + n % DEC_STEPS_MAX], dist, 1e4)
        spent += time.perf_counter() - t0
        n += 1
    tok_s = n / (spent * LAYERS)
    return {"value": round(tok_s, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"fp64 numpy oracle decode, {n} single-sequence steps of layer {l} "
                      f"({len(dist)} keys, RoPE, cache T={DEC_T}), single thread; {spent:.2f} s of "
                      f"oracle work; scaled to the {LAYERS}-layer step"}


def dec_reference_arm(args):
    """--impl reference --mode decode: the oracle decode timed on this host."""
    cb = dec_cpu_baseline(args, 10.0)
    return {"metric": DEC_METRIC, "impl": "reference", "value": cb["value"], "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(args.decode_batch / cb["value"] * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"integer decode, cache T={DEC_T}, W={args.W}"}, "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ---- configs mode (--mode configs): the pages' five configurations ---------
def configs_arm(args, dev):
    """Device time of one fwd(+bwd) call of each configuration (the pages'
    setups; synthetic N(0, 1) inputs, seeded), CUDA events over K calls after
    3 warm-ups.  One JSON object per configuration."""
    import torch

    import sfa_inputs as si
    import static_offset_sparse_gb300 as sfa

    pow2 = [1 << j for j in range(11)]

    def int_set(alpha, W):
        return sorted(set(range(W + 1)) | {round(alpha * f) for f in FIB})

    def int_set_p2():  # window 0..8 and the powers of two (alpha = 1: exact rows)
        return sorted(set(range(9)) | set(pow2))

    def chris():
        S = sfa.offsets_christoffel(128, 1024, True)
        return S

    def chris_signed():  # bidirectional: the offsets and their negatives
        S = sfa.offsets_christoffel(128, 1024, True)
        return sorted(set(S) | {-x for x in S})

    cases = [  # name, B, T, Hq, Hkv, dtype, kind, params, backward
        ("1: fp32 interp, alpha=1", 1, 1024, 8, 2, "f32", "interp", (FIB, 1.0, 8), True),
        ("2: bf16 interp, one layer, alpha=0.9667", 32, 1024, 8, 2, "bf16", "interp", (FIB, 0.5 + 7 / 15, 8), True),
        ("3: bf16 pow2 K=11, alpha=1", 32, 1024, 8, 2, "bf16", "interp", (pow2, 1.0, 8), True),
        ("3: bf16 pow2 K=11, alpha=1, integer path", 32, 1024, 8, 2, "bf16", "int", (int_set_p2(),), True),
        ("4: bf16 integer forward, T=2048, alpha=1", 4, 2048, 8, 2, "bf16", "int", (int_set(1.0, 8),), False),
        ("4: bf16 integer forward, T=16384, alpha=1.5", 4, 16384, 8, 2, "bf16", "int", (int_set(1.5, 8),), False),
        ("5: bf16 Christoffel 128/1024, 4/4 heads", 16, 2048, 4, 4, "bf16", "int", (chris(),), True),
        ("5 with 8/2 heads (G = 4)", 16, 2048, 8, 2, "bf16", "int", (chris(),), True),
        ("2 with 16/2 heads (G = 8)", 16, 1024, 16, 2, "bf16", "interp", (FIB, 0.5 + 7 / 15, 8), True),
        ("5 with 8/1 heads (G = 8)", 16, 2048, 8, 1, "bf16", "int", (chris(),), True),
        ("signed (bidirectional) Christoffel 128/1024, 4/4 heads", 16, 2048, 4, 4, "bf16", "int",
         (chris_signed(),), True),
    ]
    # per-rung cost: one config-2 layer (alpha = 0.97, W = 8) with the Fibonacci list
    # cut to its first n entries (the first five are window distances, so n - 5 rungs);
    # selected with --only "2 rung sweep", not part of the default list
    sweep = [(f"2 rung sweep: {max(n - 5, 0)} rungs", 32, 1024, 8, 2, "bf16", "interp",
              (FIB[:n], 0.97, 8), True) for n in (5, 6, 8, 10, 12, 15)]
    # config 4 over its whole grid: the integer forward at T in {2k, 4k, 8k, 16k}
    # and alpha in {0.5, 1, 1.5} (rounded offsets, W = 8); selected with --only "4 grid"
    grid4 = [(f"4 grid: T={Tg}, alpha={ag}", 4, Tg, 8, 2, "bf16", "int", (int_set(ag, 8),), False)
             for Tg in (2048, 4096, 8192, 16384) for ag in (0.5, 1.0, 1.5)]
    if args.only and args.only.startswith("2 rung sweep"):
        cases = sweep
    elif args.only and args.only.startswith("4 grid"):
        cases = grid4
    elif args.only:
        cases = [c for c in cases if c[0].startswith(args.only)]
    out = []
    for name, Bc, Tc, Hq, Hkv, dt, kind, par, bwd in cases:
        x = si.make_qkvdo_device(Bc, Tc, Hq, Hkv, D, dt, SEED, dev, layer=7)
        if kind == "interp":
            base, alpha, W = par
            f = lambda: sfa.forward(x["q"], x["k"], x["v"], W=W, alpha=alpha, base=base)  # noqa: E731
            b = lambda O, L: sfa.backward(x["q"], x["k"], x["v"], O, L, x["do"], W=W,  # noqa: E731
                                          alpha=alpha, base=base)
            keys = round(pair_counts(alpha, W)[0] / T, 2) if base is FIB else None  # mean over T=1024
        else:
            dist = par[0]
            f = lambda: sfa.forward_int(x["q"], x["k"], x["v"], dist=dist)  # noqa: E731
            b = lambda O, L: sfa.backward_int(x["q"], x["k"], x["v"], O, L, x["do"], dist=dist)  # noqa: E731
            keys = len(dist)

        def call():
            O, L = f()
            if bwd:
                b(O, L)

        for _ in range(3):
            call()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = max(3, min(args.steps, 20))
        ev0.record()
        for _ in range(n):
            call()
        ev1.record()
        torch.cuda.synchronize()
        assert sfa.get_device_status() == 0
        ms = ev0.elapsed_time(ev1) / n
        # per-kernel device time: one more timed pass with the library's launch events
        sfa.timing_enable(True)
        for _ in range(n):
            call()
        torch.cuda.synchronize()
        rec = sfa.timing_read()
        sfa.timing_enable(False)
        kernels = {k: round(t / n * 1e3, 2) for k, (t, c) in rec.items() if c}
        band = kind == "int" and dt == "bf16" and sfa.band_plan(par[0], Tc, Hq // Hkv)[0] > 0
        if band:
            path = "band (tensor cores)"
        elif dt == "bf16" and Hq // Hkv in (4, 8, 16) and not (kind == "int" and min(par[0]) < 0):
            path = "rung (tensor cores)"
        else:
            path = "SIMT"
        out.append({"config": name, "B": Bc, "T": Tc, "heads": f"{Hq}/{Hkv}", "dtype": dt,
                    "direction": "fwd+bwd" if bwd else "fwd", "path": path,
                    "ms_per_call": round(ms, 4), "tokens_per_s": round(Bc * Tc / (ms * 1e-3), 1),
                    "keys_per_query": keys, "kernel_us_per_call": kernels})
        del x
        torch.cuda.empty_cache()
    return out


def grid_arm(args, dev, staggered_pow2=False):
    """The 16-layer step of the interpolated configuration over its whole grid:
    W in {6, 8, 10, 12} x {linear, coprime} alpha schedules (staggered_pow2:
    the power-of-two base list K = 11 instead, W = 8, both schedules).  Each
    point builds its 16 layers (own seeded inputs, rotated keys once per
    layer), captures the step as one CUDA graph and times K replays with CUDA
    events after the warm-ups; one JSON object per point."""
    import ctypes as C
    import torch

    import sfa_inputs as si
    import static_offset_sparse_gb300 as sfa
    from static_offset_sparse_gb300._lib import _lib

    lib = _lib()
    peak, src = hbm_peak()
    out = []
    base = [1 << j for j in range(11)] if staggered_pow2 else None
    for schedule in ("linear", "coprime"):
        al = alphas(schedule)
        for W in ((8,) if staggered_pow2 else (6, 8, 10, 12)):
            layers = [Layer(sfa, lib, si.make_qkvdo_device(B, T, HQ, HKV, D, "bf16", rank_seed(0), dev,
                                                           layer=l), al[l], W, dev, base)
                      for l in layer_ids()]
            stream = torch.cuda.current_stream()
            sp = C.c_void_p(stream.cuda_stream)
            for _ in range(args.warmup):
                run_layers(layers, sp)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                run_layers(layers, C.c_void_p(torch.cuda.current_stream().cuda_stream))
            for _ in range(args.warmup):
                graph.replay()
            torch.cuda.synchronize()
            n = max(3, min(args.steps, 50))
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for _ in range(n):
                graph.replay()
            ev1.record(stream)
            torch.cuda.synchronize()
            assert sfa.get_device_status() == 0
            ms = ev0.elapsed_time(ev1) / n
            hbm = UNIQUE_BYTES_PER_TOKEN * B * T * len(layers) / (ms * 1e-3) / 1e9
            keys = sum(pair_counts(L.alpha, W, base)[0] for L in layers) / len(layers) / T
            name = (f"3 staggered: pow2 K=11, {schedule}, W={W}" if staggered_pow2
                    else f"2 grid: {schedule}, W={W}")
            out.append({"config": name, "B": B, "T": T, "heads": f"{HQ}/{HKV}",
                        "layers": len(layers), "dtype": "bf16", "direction": "fwd+bwd+dtheta",
                        "ms_per_step": round(ms, 4), "tokens_per_s": round(B * T / (ms * 1e-3), 1),
                        "hbm_frac": round(hbm / peak, 4), "hbm_peak_source": src,
                        "keys_per_query": round(keys, 2), "timing": f"CUDA graph of the step, {n} replays"})
            del layers, graph
            torch.cuda.empty_cache()
    return out


def config(args):
    return {"workload": f"interp {args.schedule} schedule, W={args.W}: B={B} T={T} Hq={HQ} Hkv={HKV} "
                        f"D={D}, {LAYERS} layers, Fibonacci K=15, RoPE 1e4, fwd+bwd+dtheta",
            "global_batch": B * args.gpus, "seq_len": T, "layers": LAYERS, "W": args.W,
            "schedule": args.schedule, "parallelism": f"dp{args.gpus}",
            "order": ("every forward, then the backwards from the last layer to the first"
                      if args.order == "training" else "each layer's backward right after its forward"),
            "l2": "inputs exceed L2 (16 distinct layers, 2.6 GB per step); no flush"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--W", type=int, default=8)
    ap.add_argument("--schedule", default="linear", choices=["linear", "coprime", "fixed"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--layers", type=int, default=16, help="profiling captures only")
    ap.add_argument("--order", default="training", choices=["training", "layerwise"],
                    help="order of the step's calls: training (every forward, then the "
                         "backwards last to first) or layerwise (each layer's backward right "
                         "after its forward)")
    ap.add_argument("--only", default="", help="configs mode: run the configurations whose name "
                    "starts with this (e.g. '5:'; '2 grid' runs only the W x schedule grid, '3 staggered' "
                    "only the 16-layer power-of-two step, '4 grid' the integer forward over T x alpha)")
    ap.add_argument("--mode", default="train", choices=["train", "decode", "configs"],
                    help="train: the fwd+bwd step (default); decode: one token per sequence; "
                         "configs: one line per configuration of the pages")
    ap.add_argument("--decode-batch", type=int, default=32)
    args = ap.parse_args()
    global LAYERS, ORDER
    LAYERS = args.layers
    ORDER = args.order
    args.warmup = max(3, args.warmup)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))

    if args.impl == "reference":
        if rank == 0:
            arm = dec_reference_arm if args.mode == "decode" else reference_arm
            print(json.dumps(arm(args)), flush=True)
        return

    import torch

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    from static_offset_sparse_gb300._lib import LIB_PATH

    if not os.path.exists(LIB_PATH):
        raise SystemExit("libsfa.so is not built: run __graft_entry__.build() first")
    if args.mode == "decode":  # one process per GPU, independent replicas
        if rank == 0:
            print(json.dumps(decode_arm(args, dev)), flush=True)
        return
    if args.mode == "configs":
        if rank == 0:
            if not args.only or args.only.startswith("2 grid"):
                for line in grid_arm(args, dev):
                    print(json.dumps(line), flush=True)
            if not args.only or args.only.startswith("3 staggered"):
                for line in grid_arm(args, dev, staggered_pow2=True):
                    print(json.dumps(line), flush=True)
            if args.only not in ("2 grid", "3 staggered"):
                for line in configs_arm(args, dev):
                    print(json.dumps(line), flush=True)
        return
    layers, ms, clk, launches, roofline = gpu_arm(args, rank, world, dev)
    value = world * B * T / (ms * 1e-3)
    hbm = UNIQUE_BYTES_PER_TOKEN * B * T * LAYERS / (ms * 1e-3) / 1e9
    peak, peak_src = hbm_peak()
    out = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic: seeded N(0,1) Q, K, V, dO per layer", "config": config(args),
           "roofline": roofline,
           "hbm": {"unique_bytes_per_token_layer": UNIQUE_BYTES_PER_TOKEN,
                   "achieved_gbs": round(hbm, 1), "peak_gbs": peak, "peak_source": peak_src,
                   "frac": round(hbm / peak, 4)},
           "gpu_launches": launches, "clocks": clk}
    if not args.no_e2e:
        out["e2e"] = e2e_arm(layers, min(args.steps, 20), args.warmup, world, dev)
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        out["cpu_baseline"] = cpu_baseline(args.schedule, args.W, args.cpu_budget)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
