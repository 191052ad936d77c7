#!/usr/bin/env python3
"""Throughput of the W1.58A8 BitLinear hot path on one GB300 (or N replicas).

Default workload (one step = one decode layer): all seven BitLinear projections
of one Qwen3-shaped 0.6B layer at M=1 token (q 1024->2048, k/v 1024->1024,
o 2048->1024, gate/up 1024->3072, down 3072->1024), each with its own seeded
input, norm weight and ternary weights, run as ONE grouped launch
(bitnet_bitlinear_forward_group).  Steps rotate through a pool of distinct
layers whose I2_S weights total more than twice the L2 cache, so every step
streams its weights from HBM.  Metric: weight-stream GB/s = algorithmic bytes
(packed weights + scale + x + norm weight + y) per step / time.  The same line
carries a `prefill` object, the other half of the metric, timed in the same run:
int8-TOPS of the Qwen3-shaped 28-layer stack at 32768 tokens and of one
compute-bound projection (M=16384, K=4096, N=16384), each against the bf16 dense
peak and HBM, with sampled rows checked against the oracle (--no-prefill skips it).

Other workloads (--workload): q_proj_m8 (M=8, K=1024, N=2048), proj (one
projection, --m/--k/--n), gemma3_prefill
(seven Gemma3-shaped projections at M=32768 with 1% x20 outlier features),
qwen3_prefill_stack (28 layers x 7 projections at M=32768), sweep (K, N in
{1024,4096,8192,16384} x M in {1,16,128,2048,16384}), glu_proj (the down
projection BitLinear(act(gate) * up), --m/--k/--n/--act), qk_proj (a q/k projection
with its QK head norm, --m/--k/--n/--head-dim).  --io f16|bf16 runs the
prefill workloads with 16-bit x and y (bitnet_bitlinear_forward_typed).

--impl reference times the CPU oracle (test infrastructure, plain C) on the
host cores on a bounded sample of the same workload.

Launch: python bench.py [--gpus N --steps K --warmup W]; for N > 1 under
torchrun, one replica per GPU (the projection shards by token rows and needs
no exchange; this benchmark runs independent replicas, weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BitLinear int8-TOPS (prefill) and weight-stream GB/s (M=1) vs GB300 roofline"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ------------------------------------------------------------------ helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "bitlinear_rmsnorm_token_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(profile_md, sha):
    """dram bytes per launch recorded by an ncu capture of this exact kernel
    source (a line 'traffic_bytes_per_launch: <int> source_sha: <sha>'), else None."""
    path = os.path.join(ROOT, "profiles", profile_md)
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)\s+source_sha:\s*([0-9a-f]+)", text)
    if m and m.group(2) == sha:
        return int(m.group(1))
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples with wall-clock timestamps."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.flush()

    def summary(self, t0, t1):
        rows = []
        try:
            with open(self.out.name) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                        frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                        rows.append((ts + frac, float(parts[1]), float(parts[2]), parts[5:9]))
                    except (ValueError, IndexError):
                        continue
        finally:
            os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        window = "timed"
        if not inside:
            inside, window = rows, "whole run"
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


def dist_setup(gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = os.environ.get("BENCH_DIST_BACKEND", "nccl")
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def reduce_max(value, world):
    """Max of a float over ranks (gloo or nccl)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value, world):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(ms_local, units_local, world):
    """Whole-job figures over replicas: the slowest rank's time and the units
    every rank processed.  Returns (ms_max, units_total, units_total / s)."""
    ms = reduce_max(float(ms_local), world)
    units = reduce_sum(float(units_local), world)
    return ms, units, units / (ms * 1e-3)


# --------------------------------------------------------- decode workload

def decode_config(world):
    """The workload the default line (and the reference arm) measures."""
    from bitlinear_rmsnorm_token_gb300 import workloads as wl

    shapes = wl.QWEN3_0P6B_LAYER
    return {"workload": "qwen3_0p6b_decode_layer_M1_7proj", "tokens": 1,
            "projections": [f"{p.name} {p.K}->{p.N}" for p in shapes],
            "bytes_per_step": decode_layer_bytes(shapes, 1),
            "l2": "inputs larger than L2: GPU steps rotate through a weight pool > 2x L2 (no flush)",
            "parallelism": f"replicas x{world}"}


def decode_layer_bytes(layer_shapes, M=1):
    """Algorithmic bytes of one step: I2_S weights + scale, x, norm weight, y."""
    return sum(p.N * p.K // 4 + 4 + M * p.K * 4 + p.K * 4 + M * p.N * 4 for p in layer_shapes)


def build_decode_pool(torch, bn, wl, n_layers, device, M=1):
    """n_layers distinct Qwen3-shaped layers: weights packed on the device from
    seeded latents; x / norm weights seeded.  Inputs for one layer are views of
    one contiguous buffer (one host<->device copy per step in the e2e loop)."""
    shapes = wl.QWEN3_0P6B_LAYER
    kx = sum(p.K for p in shapes)
    ny = sum(p.N for p in shapes)
    layers = []
    for layer in range(n_layers):
        xbuf = torch.empty((M * kx,), dtype=torch.float32, device=device)
        ybuf = torch.zeros((M * ny,), dtype=torch.float32, device=device)
        items = []
        ox = oy = 0
        for i, p in enumerate(shapes):
            seed_w = wl.seed_for(1, layer, i, wl.T_W)
            w = wl.gen_device((p.N, p.K), seed_w, device, std=0.02)
            packed, ws = bn.pack_i2s(w)
            del w
            x = wl.gen_x(M, p.K, wl.seed_for(1, layer, i, wl.T_X))
            g = wl.gen_norm_w(p.K, wl.seed_for(1, layer, i, wl.T_G))
            xv = xbuf[ox:ox + M * p.K].view(M, p.K)
            xv.copy_(torch.from_numpy(x))
            yv = ybuf[oy:oy + M * p.N].view(M, p.N)
            ox += M * p.K
            oy += M * p.N
            items.append((xv, torch.from_numpy(g).to(device), packed, ws, p.N, yv))
        layers.append({"items": items, "desc": bn.make_group(items), "xbuf": xbuf, "ybuf": ybuf})
    return layers


def check_decode_layer(oracle, layer, M=1):
    """Oracle check of one pool layer (run after timing): every projection's y."""
    worst = 0.0
    for (xv, g, packed, ws, N, yv) in layer["items"]:
        x = xv.cpu().numpy()
        ref = oracle.bitlinear_forward(x, g.cpu().numpy(), packed.cpu().numpy(), ws, N)
        y = yv.cpu().numpy()
        rel = np.linalg.norm(y - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
        worst = max(worst, float(rel.max()))
    return worst


def run_decode(args, rank, world, local):
    import torch

    import bitlinear_rmsnorm_token_gb300 as bn
    from bitlinear_rmsnorm_token_gb300 import workloads as wl

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    bn.lib()
    M = 1
    shapes = wl.QWEN3_0P6B_LAYER
    step_bytes = decode_layer_bytes(shapes, M)
    weight_bytes = sum(p.N * p.K // 4 + 4 for p in shapes)
    n_layers = max(8, int(np.ceil(2.0 * L2_BYTES / weight_bytes)))  # pool > 2x L2
    pool = build_decode_pool(torch, bn, wl, n_layers, device, M)
    flags = bn.FLAG_WEIGHTS_STATIC
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize()

    # one graph holds `chunk` consecutive steps; replays continue the rotation
    chunk = n_layers * max(1, 512 // n_layers)
    with torch.cuda.stream(stream):
        for i in range(n_layers):  # eager first calls (load the module, set up the device)
            bn.bitlinear_forward_group(pool[i]["desc"], M, wl.EPS, flags, stream=stream)
    stream.synchronize()
    graphs = {}

    def graph_of(n):
        """A CUDA graph of n consecutive steps of the rotation (n <= chunk)."""
        if n not in graphs:
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_, stream=stream):
                for i in range(n):
                    bn.bitlinear_forward_group(pool[i % n_layers]["desc"], M, wl.EPS, flags, stream=stream)
            graphs[n] = g_
        return graphs[n]

    def run_steps(n):
        """Exactly n steps: whole graphs of `chunk` steps, then one of the rest."""
        with torch.cuda.stream(stream):
            for _ in range(n // chunk):
                graph_of(chunk).replay()
            if n % chunk:
                graph_of(n % chunk).replay()

    # Timed region: exactly `steps` steps between two events, repeated in
    # batches of `batch` until the timed phase has lasted `min_wall_s` (so that
    # the clock samples are taken under this load); the per-step time is the
    # median repeat's.  Each repeat
    # starts with one graph holding an untimed pre-roll of `preroll` steps and
    # then the first timed steps.  The start event is recorded inside that graph
    # on a side branch that waits for the last pre-roll step, so it fires when
    # that step completes while the first timed step keeps its programmatic
    # launch overlap with it (as every step has in a long run): the region is
    # exactly `steps` step-to-step intervals of the steady state.  The rest of
    # the steps follow as whole graphs; the end event follows the last step.
    preroll = min(chunk, 64)
    batch, min_wall_s = 8, 0.6
    first_n = min(args.steps, chunk)
    side = torch.cuda.Stream(device)

    def first_graph(ev0):
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_, stream=stream):
            for i in range(preroll):
                bn.bitlinear_forward_group(pool[i % n_layers]["desc"], M, wl.EPS, flags, stream=stream)
            fork = torch.cuda.Event()
            fork.record(stream)
            side.wait_event(fork)
            ev0.record(side)
            for i in range(first_n):
                bn.bitlinear_forward_group(pool[(preroll + i) % n_layers]["desc"], M, wl.EPS, flags, stream=stream)
            stream.wait_stream(side)
        return g_

    try:
        starts = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(batch)]
        firsts = [first_graph(e) for e in starts]
        start_event = "recorded inside the first graph on a branch after the last pre-roll step"
    except (TypeError, RuntimeError):
        # no event nodes in graphs: record the start event between the pre-roll
        # graph and the timed steps instead (the first timed step then loses its
        # overlap with the pre-roll)
        torch.cuda.synchronize()
        starts, firsts = [torch.cuda.Event(enable_timing=True) for _ in range(batch)], None
        first_n = 0
        start_event = "recorded on the stream between the pre-roll graph and the first timed step"
    rest = args.steps - first_n
    graph_of(preroll)
    graph_of(chunk)
    if rest % chunk:
        graph_of(rest % chunk)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.5)
    run_steps(args.warmup)  # exactly `warmup` untimed steps
    stream.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(batch)]
    rep_ms = []
    t0 = time.time()
    with torch.cuda.stream(stream):
        while True:
            for r in range(batch):
                if firsts is not None:
                    firsts[r].replay()
                else:
                    graph_of(preroll).replay()
                    starts[r].record(stream)
                run_steps(rest)
                ends[r].record(stream)
            ends[-1].synchronize()
            rep_ms += [starts[r].elapsed_time(ends[r]) for r in range(batch)]
            if time.time() - t0 >= min_wall_s:
                break
    t1 = time.time()
    torch.cuda.synchronize()
    barrier(world)
    sampler.stop()
    ms_local = float(np.median(rep_ms))
    ms, _, value = aggregate(ms_local, float(step_bytes) * args.steps, world)
    value /= 1e9
    clocks = sampler.summary(t0, t1)

    # parity of the timed configuration: every projection of two pool layers
    import oracle

    worst = 0.0
    for li in (0, n_layers - 1):
        worst = max(worst, check_decode_layer(oracle, pool[li], M))
    dev_status = bn.last_device_status()

    # e2e through the public API with host buffers: per step, H2D of the
    # layer's activations from pinned memory, the grouped call, D2H of y.
    # The per-step sequence is captured in a CUDA graph (one rotation through
    # the weight pool) and replayed; the copies are nodes of the graph and
    # happen on every replayed step.  Headline form: pipelined as a serving
    # loop would run it -- inputs on one copy stream, the grouped calls in
    # order on the compute stream, results on another copy stream, events for
    # the true dependencies (step i's call after step i's input copy, step i's
    # result copy after step i's call), so one step's copies overlap its
    # neighbours' calls.  Every layer of the rotation has its own device
    # buffers, so no copy can overwrite data a pending call still reads.
    # Also reported: the same three calls in one stream (serial) and issued
    # eagerly from Python.
    kx = pool[0]["xbuf"].numel()
    ny = pool[0]["ybuf"].numel()
    xh = torch.empty((n_layers, kx), dtype=torch.float32).pin_memory()
    for i in range(n_layers):
        xh[i].copy_(pool[i]["xbuf"].cpu())
    yh = torch.empty((n_layers, ny), dtype=torch.float32).pin_memory()

    def e2e_step(i):
        L = pool[i % n_layers]
        L["xbuf"].copy_(xh[i % n_layers], non_blocking=True)
        bn.bitlinear_forward_group(L["desc"], M, wl.EPS, flags, stream=stream)
        yh[i % n_layers].copy_(L["ybuf"], non_blocking=True)

    s_in = torch.cuda.Stream(device)
    s_out = torch.cuda.Stream(device)

    def e2e_rotation_pipelined():
        start = torch.cuda.Event()
        start.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        for i in range(n_layers):
            L = pool[i]
            with torch.cuda.stream(s_in):
                L["xbuf"].copy_(xh[i], non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
            stream.wait_event(ev_in)
            bn.bitlinear_forward_group(L["desc"], M, wl.EPS, flags, stream=stream)
            ev_k = torch.cuda.Event()
            ev_k.record(stream)
            s_out.wait_event(ev_k)
            with torch.cuda.stream(s_out):
                yh[i].copy_(L["ybuf"], non_blocking=True)
        done = torch.cuda.Event()
        done.record(s_out)
        stream.wait_event(done)

    def e2e_rotation_serial():
        for i in range(n_layers):
            e2e_step(i)

    def timed_graph(rotation):
        with torch.cuda.stream(stream):
            rotation()
        torch.cuda.synchronize()
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_, stream=stream):
            rotation()
        reps = max(1, -(-min(args.steps, 2000) // n_layers))
        with torch.cuda.stream(stream):
            for _ in range(2):
                g_.replay()
        stream.synchronize()
        barrier(world)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(reps):
                g_.replay()
            b.record(stream)
        b.synchronize()
        return aggregate(a.elapsed_time(b), float(step_bytes) * reps * n_layers, world)[2], reps * n_layers

    e2e_value, e2e_steps = timed_graph(e2e_rotation_pipelined)
    e2e_serial, _ = timed_graph(e2e_rotation_serial)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # the same loop issued eagerly from Python, for reference
    eager_steps = min(args.steps, 1000)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(eager_steps):
            e2e_step(i)
        e1.record(stream)
    e1.synchronize()
    _, _, e2e_eager = aggregate(e0.elapsed_time(e1), float(step_bytes) * eager_steps, world)

    # cold: L2 flushed before each launch (a write of 2x L2), the layer timed
    # alone between events (the flush is still running when the layer and its
    # events are enqueued, so no host gap falls inside)
    flush = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.float32, device=device)
    cold = []
    with torch.cuda.stream(stream):
        for i in range(21):
            flush.fill_(float(i))
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            bn.bitlinear_forward_group(pool[i % n_layers]["desc"], M, wl.EPS, flags, stream=stream)
            b.record(stream)
            b.synchronize()
            cold.append(a.elapsed_time(b))
    del flush
    cold_ms = float(np.median(cold[1:]))

    hbm, _, _, peak_kind = peaks()
    per_launch_ms = ms_local / args.steps
    achieved = step_bytes / (per_launch_ms * 1e-3) / 1e9
    sha = source_sha("gemv.cu", "rowquant.cuh", "common.cuh")
    traffic = profiled_traffic("decode_group_qwen3_layer.md", sha)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8 x ternary -> int32, fp32 I/O", "data": "synthetic",
        "config": decode_config(world),
        "setup": {"weight_pool_layers": n_layers, "weight_pool_bytes": n_layers * weight_bytes,
                  "launch": "one grouped kernel per step, CUDA graph replay, programmatic dependent launch"},
        "timing": {"repeats": len(rep_ms), "ms_per_repeat_min": round(min(rep_ms), 6),
                   "ms_per_repeat_median": round(ms_local, 6), "ms_per_repeat_max": round(max(rep_ms), 6),
                   "timed_phase_s": round(t1 - t0, 3),
                   "statistic": "median repeat; each repeat times exactly `steps` steps between two events; "
                                f"repeats run in batches of {batch} until the timed phase has lasted "
                                f"{min_wall_s} s, so that the clock samples fall under this load",
                   "preroll_steps": preroll, "start_event": start_event},
        "roofline": {"bound": "hbm", "kernel": "k_decode (grouped BitLinear GEMV)", "achieved": round(achieved, 2),
                     "peak": hbm, "peak_kind": f"{peak_kind} HBM copy GB/s", "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": step_bytes},
        "e2e": {"value": round(e2e_value / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": kx * 4, "d2h_bytes_per_step": ny * 4, "steps": e2e_steps,
                "api": "per step: H2D of x from pinned memory, bitnet_bitlinear_forward_group, D2H of y; "
                       "pipelined over three streams (input copies, grouped calls in order, result copies) with "
                       "events for step i's dependencies, captured in a CUDA graph and replayed",
                "serial_value": round(e2e_serial / 1e9, 2),
                "serial_api": "the same three calls in one stream, captured in a CUDA graph",
                "eager_value": round(e2e_eager / 1e9, 2),
                "eager_api": "the same three calls issued from Python every step, one stream"},
        "cold_l2": {"us_per_layer": round(cold_ms * 1e3, 3), "GBps": round(step_bytes / (cold_ms * 1e-3) / 1e9, 2),
                    "method": "L2 flushed by a 2x L2 write before each launch; median of 20 launches"},
        "gpu_launches": args.steps,  # per timed region: one grouped launch per step
        "clocks": clocks,
        "parity": {"oracle_worst_row_rel_l2": worst, "device_status": bn.status_string(dev_status)},
    }
    del pool, graphs, firsts
    torch.cuda.empty_cache()
    if not args.no_prefill:
        # the prefill half of the metric, timed in the same run: the Qwen3-shaped
        # 28-layer stack at 32768 tokens (fp32 I/O) and one compute-bound shape
        out["prefill"] = {
            "qwen3_0p6b_stack_M32768": measure_prefill(args, world, local, "qwen3_prefill_stack", "f32",
                                                       steps=min(args.steps, 10), warmup=2),
            "proj_M16384_K4096_N16384": measure_point(args, world, local, 16384, 4096, 16384),
        }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline_decode(args, single_thread=True)
    return out


def cpu_baseline_decode(args, budget_s=None, max_steps=None, warmup=0, single_thread=False):
    """The oracle, as it stands, on the host cores: whole decode layers (7
    projections at M=1, packed on the host by the oracle).  `warmup` untimed
    layers, then timed layers until `max_steps` or ~budget_s, whichever first."""
    import oracle
    from bitlinear_rmsnorm_token_gb300 import workloads as wl

    budget_s = args.cpu_seconds if budget_s is None else budget_s
    shapes = wl.QWEN3_0P6B_LAYER
    step_bytes = decode_layer_bytes(shapes, 1)
    layers = []
    for layer in range(2):
        items = []
        for i, p in enumerate(shapes):
            x, g, w = wl.gen_projection(1, layer, i, 1, p.K, p.N)
            packed, ws = oracle.pack_i2s(w)
            items.append((x, g, packed, ws, p.N))
        layers.append(items)

    def one_layer(n):
        for (x, g, packed, ws, N) in layers[n % 2]:
            oracle.bitlinear_forward(x, g, packed, ws, N)

    for n in range(warmup):
        one_layer(n)
    n = 0
    t0 = time.perf_counter()
    while max_steps is None or n < max_steps:
        one_layer(n)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    # the oracle's contraction shares its (row, column) pairs among the threads,
    # so the one token row of a decode layer spreads over every host core
    cores = oracle.num_threads()
    out = {"value": round(step_bytes * n / dt / 1e9, 4), "unit": "GB/s", "cores": cores,
           "kind": "oracle", "steps": n, "seconds": dt,
           "sample": f"{n} decode layers (7 projections each, M=1) in {dt:.1f} s on {cores} threads"}
    if single_thread:
        # the same with the thread count set to one (a short sample)
        cores = oracle.num_threads()
        oracle.set_num_threads(1)
        try:
            n1, t1 = 0, time.perf_counter()
            while n1 < 2 or time.perf_counter() - t1 < min(3.0, budget_s):
                one_layer(n1)
                n1 += 1
            d1 = time.perf_counter() - t1
        finally:
            oracle.set_num_threads(cores)
        out["single_thread"] = {"value": round(step_bytes * n1 / d1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                                "sample": f"{n1} decode layers in {d1:.1f} s"}
    return out


# ----------------------------------------------------- other workloads

def time_region(torch, stream, fn, steps, warmup):
    for _ in range(warmup):
        fn()
    stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / steps


def run_q_proj_m8(args, rank, world, local):
    import torch

    import bitlinear_rmsnorm_token_gb300 as bn
    from bitlinear_rmsnorm_token_gb300 import workloads as wl

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    M, K, N = 8, 1024, 2048
    pool = []
    nl = int(np.ceil(2.0 * L2_BYTES / (N * K / 4)))
    for l in range(nl):
        x, g, w = wl.gen_projection(0, l, 0, M, K, N)
        packed, ws = bn.pack_i2s(torch.from_numpy(w).to(device))
        pool.append((torch.from_numpy(x).to(device), torch.from_numpy(g).to(device), packed, ws,
                     torch.empty((M, N), dtype=torch.float32, device=device)))
    stream = torch.cuda.Stream(device)
    it = [0]

    def step():
        x, g, packed, ws, y = pool[it[0] % nl]
        it[0] += 1
        bn.bitlinear_forward(x, g, packed, ws, N, wl.EPS, y, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(nl):
            step()
    stream.synchronize()
    g_ = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_, stream=stream):
        for _ in range(nl):
            step()
    reps = max(1, args.steps // nl)
    with torch.cuda.stream(stream):
        ms = time_region(torch, stream, g_.replay, reps, max(3, args.warmup // nl)) / nl
    step_bytes = N * K // 4 + 4 + M * K * 4 + K * 4 + M * N * 4
    return {"metric": METRIC, "value": round(step_bytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "n_gpus": world,
            "steps": reps * nl, "ms_per_step": ms, "us_per_projection": ms * 1e3,
            "tops": 2.0 * M * N * K / (ms * 1e-3) / 1e12,
            "config": {"workload": "q_proj_M8_K1024_N2048", "launch": "CUDA graph, weight pool > 2x L2"}}


def noalloc_fits(bn, M, K, N):
    """True when the no-alloc entry point's fixed array holds the codes, the
    scales and the largest K-split workspace any plan could ask for (fp32
    partial sums and one ticket per 128x64 tile), so that it runs the same plan
    as bitnet_bitlinear_forward."""
    r256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    code_bytes = M * K * (1 if M <= 8 else 2)
    ws_bound = r256(M * N * 4) + 4 * (-(-M // 128)) * (-(-N // 64))
    return r256(code_bytes) + r256(4 * M) + ws_bound <= bn.NOALLOC_SCRATCH_BYTES


def run_proj(args, rank, world, local):
    """One projection of M tokens, K -> N (--m, --k, --n), cycling through
    distinct weight tensors totalling more than twice the L2.  Where the no-alloc
    entry point's fixed scratch holds the plan's temporaries, the cycle is one
    CUDA graph of that entry point (kernel time, not launch time); otherwise
    bitnet_bitlinear_forward is called eagerly (such shapes run >= 80 us)."""
    import torch

    import bitlinear_rmsnorm_token_gb300 as bn
    from bitlinear_rmsnorm_token_gb300 import workloads as wl

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    M, K, N = args.m, args.k, args.n
    wb = N * K // 4
    nw = min(1024, max(2, int(np.ceil(2.0 * L2_BYTES / wb))))
    ws_list = []
    for i in range(nw):
        w = wl.gen_device((N, K), wl.seed_for(5, K, N, i), device, std=0.02)
        ws_list.append(bn.pack_i2s(w))
        del w
    g = torch.from_numpy(wl.gen_norm_w(K, seed=K)).to(device)
    x = wl.gen_device((M, K), wl.seed_for(5, M, K, N), device)
    y = torch.empty((M, N), dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device)
    graphed = noalloc_fits(bn, M, K, N)
    fwd = bn.bitlinear_forward_noalloc if graphed else bn.bitlinear_forward

    def cycle():
        for packed, sc in ws_list:
            fwd(x, g, packed, sc, N, wl.EPS, y, stream=stream)

    with torch.cuda.stream(stream):
        cycle()
    stream.synchronize()
    reps = max(1, args.steps // nw)
    if graphed:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            cycle()
        with torch.cuda.stream(stream):
            ms = time_region(torch, stream, graph.replay, reps, max(1, min(args.warmup, 3))) / nw
    else:
        with torch.cuda.stream(stream):
            ms = time_region(torch, stream, cycle, reps, max(1, min(args.warmup, 3))) / nw
    b = wb + 4 + M * K * 4 + K * 4 + M * N * 4
    hbm, bf16, _, _ = peaks()
    return {"metric": METRIC, "value": round(b / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "n_gpus": world,
            "steps": reps * nw, "ms_per_step": ms, "us_per_projection": ms * 1e3,
            "tops": 2.0 * M * N * K / (ms * 1e-3) / 1e12, "hbm_frac": b / (ms * 1e-3) / 1e9 / hbm,
            "config": {"workload": f"proj_M{M}_K{K}_N{N}", "weights_cycled": nw,
                       "launch": "CUDA graph of bitnet_bitlinear_forward_noalloc" if graphed
                       else "eager bitnet_bitlinear_forward, one stream"}}


def run_glu_proj(args, rank, world, local):
    """The down projection y = BitLinear(act(gate) * up) (--m, --k, --n, --act): few
    tokens as a CUDA graph cycling distinct weight tensors totalling more than twice
    the L2, many tokens eagerly (the norm launch computes the activation as it loads
    the rows; pool memory for the intermediates)."""
    import torch

    import bitlinear_rmsnorm_token_gb300 as bn
    import oracle
    from bitlinear_rmsnorm_token_gb300 import workloads as wl

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    M, K, N, act = args.m, args.k, args.n, args.act
    wb = N * K // 4
    nw = min(1024, max(2, int(np.ceil(2.0 * L2_BYTES / wb)))) if M <= 8 else 1
    ws_list = []
    for i in range(nw):
        w = wl.gen_device((N, K), wl.seed_for(6, K, N, i), device, std=0.02)
        ws_list.append(bn.pack_i2s(w))
        del w
    g = torch.from_numpy(wl.gen_norm_w(K, seed=K)).to(device)
    gate = wl.gen_device((M, K), wl.seed_for(6, M, K, 1), device) * 2.0
    up = wl.gen_device((M, K), wl.seed_for(6, M, K, 2), device)
    y = torch.empty((M, N), dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device)

    def cycle():
        for packed, sc in ws_list:
            bn.bitlinear_forward_glu(gate, up, act, g, packed, sc, N, wl.EPS, y, stream=stream)

    with torch.cuda.stream(stream):
        cycle()
    stream.synchronize()
    if M <= 8:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            cycle()
        reps = max(1, args.steps // nw)
        with torch.cuda.stream(stream):
            ms = time_region(torch, stream, graph.replay, reps, max(1, min(args.warmup, 3))) / nw
        launch = "CUDA graph of bitnet_bitlinear_forward_glu"
    else:
        reps = max(1, args.steps)
        with torch.cuda.stream(stream):
            ms = time_region(torch, stream, cycle, reps, max(1, min(args.warmup, 3)))
        launch = "bitnet_bitlinear_forward_glu, eager"
    rows = np.arange(M) if M <= 64 else np.random.default_rng(0).choice(M, 32, replace=False)
    packed, sc = ws_list[-1]
    ref = oracle.bitlinear_forward_glu(gate[rows].cpu().numpy(), up[rows].cpu().numpy(), act, g.cpu().numpy(),
                                       packed.cpu().numpy(), sc, N)
    yy = y[rows].cpu().numpy()
    worst = float((np.linalg.norm(yy - ref, axis=1) / np.linalg.norm(ref, axis=1)).max())
    b = wb + 4 + 2 * M * K * 4 + K * 4 + M * N * 4
    hbm, bf16, _, _ = peaks()
    return {"metric": METRIC, "value": round(b / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "n_gpus": world,
            "steps": reps * nw, "ms_per_step": ms, "us_per_projection": ms * 1e3,
            "tops": 2.0 * M * N * K / (ms * 1e-3) / 1e12, "hbm_frac": b / (ms * 1e-3) / 1e9 / hbm,
            "tensor_frac": 2.0 * M * N * K / (ms * 1e-3) / 1e12 / bf16,
            "config": {"workload": f"down_glu_M{M}_K{K}_N{N}_act{act}", "weights_cycled": nw, "launch": launch,
                       "bytes_per_step": b},
            "parity": {"oracle_worst_row_rel_l2": worst}}


def run_qk_proj(args, rank, world, local):
    """The q/k projection with its QK head norm (--m/--k/--n/--head-dim; default
    the Qwen3 q projection at 32768 tokens, heads of 128): the projection alone
    and chained with the head norm (several weight sets, inputs larger than L2),
    and the head norm alone on y in place, replayed from a CUDA graph."""
    import torch

    import bitlinear_rmsnorm_token_gb300 as bn
    import oracle
    from bitlinear_rmsnorm_token_gb300 import workloads as wl

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    M, K, N, hd = args.m, args.k, args.n, args.head_dim
    stream = torch.cuda.Stream(device)
    x = wl.gen_device((M, K), wl.seed_for(6, M, K, N), device)
    g = torch.from_numpy(wl.gen_norm_w(K, seed=K)).to(device)
    hw = torch.from_numpy(wl.gen_norm_w(hd, seed=hd)).to(device)
    sets = []
    for i in range(4):
        w = wl.gen_device((N, K), wl.seed_for(6, K, N, i), device, std=0.02)
        sets.append(bn.pack_i2s(w))
        del w
    y = torch.empty((M, N), dtype=torch.float32, device=device)

    def fwd():
        for packed, ws in sets:
            bn.bitlinear_forward(x, g, packed, ws, N, wl.EPS, y, stream=stream)

    def fwd_qk():
        for packed, ws in sets:
            bn.bitlinear_forward_qk(x, g, packed, ws, N, hd, hw, wl.EPS, y, stream=stream)

    with torch.cuda.stream(stream):
        ms_f = time_region(torch, stream, fwd, 5, 2) / len(sets)
        ms_qk = time_region(torch, stream, fwd_qk, 5, 2) / len(sets)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(8):
                bn.head_rmsnorm(y, hd, hw, wl.EPS, out=y, stream=stream)
        ms_h = time_region(torch, stream, graph.replay, 5, 2) / 8
    hbm, _, _, _ = peaks()
    hb = M * N * 8 + hd * 4
    rows = np.random.default_rng(0).choice(M, min(M, 16), replace=False)
    fwd_qk()
    packed, ws = sets[-1]
    ref = oracle.bitlinear_forward_qk(x[rows].cpu().numpy(), g.cpu().numpy(), packed.cpu().numpy(), ws, N, hd,
                                      hw.cpu().numpy())
    yy = y[rows].cpu().numpy()
    worst = float((np.linalg.norm(yy - ref, axis=1) / np.linalg.norm(ref, axis=1)).max())
    return {"metric": METRIC, "value": round(2.0 * M * N * K / (ms_qk * 1e-3) / 1e12, 2), "unit": "TOPS",
            "n_gpus": world, "ms_per_step": ms_qk, "us_projection": ms_f * 1e3, "us_projection_qk": ms_qk * 1e3,
            "us_head_norm_alone": ms_h * 1e3, "head_norm_GBps": hb / (ms_h * 1e-3) / 1e9,
            "head_norm_hbm_frac": hb / (ms_h * 1e-3) / 1e9 / hbm,
            "config": {"workload": f"qk_proj_M{M}_K{K}_N{N}_hd{hd}", "weights_cycled": len(sets),
                       "launch": "eager projections; head norm alone: CUDA graph"},
            "parity": {"oracle_worst_row_rel_l2": worst}}


def prefill_projection_step(torch, bn, wl, shapes, M, device, config, layer, outlier_frac, stream,
                            io_dtype=None):
    """Buffers for one layer's projections at M tokens (x drawn on the device;
    with io_dtype, x rounded to that 16-bit type and y allocated in it)."""
    items = []
    for i, p in enumerate(shapes):
        x = wl.gen_device((M, p.K), wl.seed_for(config, layer, i, wl.T_X), device)
        if outlier_frac > 0:
            cols = torch.from_numpy(wl.gen_device_outlier_cols(p.K, wl.seed_for(config, layer, i, wl.T_OUTLIER),
                                                               outlier_frac)).to(device)
            x[:, cols] *= 20.0
        g = torch.from_numpy(wl.gen_norm_w(p.K, wl.seed_for(config, layer, i, wl.T_G))).to(device)
        w = wl.gen_device((p.N, p.K), wl.seed_for(config, layer, i, wl.T_W), device, std=0.02)
        packed, ws = bn.pack_i2s(w)
        del w
        if io_dtype is not None:
            x = x.to(io_dtype)
        y = torch.empty((M, p.N), dtype=io_dtype or torch.float32, device=device)
        items.append((p, x, g, packed, ws, y))
    return items


def sampled_row_parity(oracle, bn, x, g, packed, ws, N, y, rows, y_dtype=0):
    """Oracle check of sampled rows: y under the row contract (worst relative
    L2 distance), and the int8 codes of the same rows from the norm launch
    against the oracle's (count and size of any differences)."""
    xr = x[rows]
    ref = oracle.bitlinear_forward_typed(xr.float().cpu().numpy(), g.cpu().numpy(), packed.cpu().numpy(), ws, N,
                                         y_dtype=y_dtype)
    yy = y[rows].float().cpu().numpy()
    worst = float((np.linalg.norm(yy - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)).max())
    flips = 0
    if y_dtype == 0:
        codes, _, _ = bn.rmsnorm_quant_a8(xr.contiguous(), g)
        q_o, _, _ = oracle.quant_a8(oracle.rmsnorm(xr.cpu().numpy(), g.cpu().numpy()))
        d = np.abs(codes.cpu().numpy().astype(np.int32) - q_o.astype(np.int32))
        flips = int(np.sum(d != 0))
        assert d.max(initial=0) <= 1, "an int8 code differs from the oracle's by more than one"
    return worst, flips


def measure_prefill(args, world, local, which, io_name="f32", steps=None, warmup=None):
    """One step = every projection of the workload at M = 32768 tokens, issued
    eagerly on one stream (each call one norm launch and one contraction)."""
    import torch

    import bitlinear_rmsnorm_token_gb300 as bn
    import oracle
    from bitlinear_rmsnorm_token_gb300 import workloads as wl

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    steps = max(1, args.steps if steps is None else steps)
    warmup = max(1, min(args.warmup, 3) if warmup is None else warmup)
    M = 32768
    if which == "gemma3_prefill":
        shapes, n_layers, frac, cfg = wl.GEMMA3_270M_LAYER, 1, 0.01, 2
    else:
        shapes, n_layers, frac, cfg = wl.QWEN3_0P6B_LAYER, wl.QWEN3_0P6B_LAYERS, 0.0, 3
    stream = torch.cuda.Stream(device)
    io = {"f32": None, "f16": torch.float16, "bf16": torch.bfloat16}[io_name]
    io_bytes = 4 if io is None else 2
    layers = [prefill_projection_step(torch, bn, wl, shapes, M, device, cfg, l, frac, stream, io)
              for l in range(n_layers)]
    torch.cuda.synchronize()

    def step():
        for items in layers:
            for (p, x, g, packed, ws, y) in items:
                if io is None:
                    bn.bitlinear_forward(x, g, packed, ws, p.N, wl.EPS, y, stream=stream)
                else:
                    bn.bitlinear_forward_typed(x, g, packed, ws, p.N, wl.EPS, y, stream=stream)

    with torch.cuda.stream(stream):
        ms = time_region(torch, stream, step, steps, warmup)
    flops = sum(2.0 * M * p.N * p.K for p in shapes) * n_layers
    alg_bytes = sum(M * p.K * io_bytes + p.K * 4 + p.N * p.K / 4 + 4 + M * p.N * io_bytes for p in shapes) * n_layers
    # sampled-row parity of the first and last projection
    worst, flips = 0.0, 0
    rows = np.random.default_rng(0).choice(M, 32, replace=False)
    for (p, x, g, packed, ws, y) in (layers[0][0], layers[-1][-1]):
        w_, f_ = sampled_row_parity(oracle, bn, x, g, packed, ws, p.N, y, rows,
                                    {"f32": 0, "f16": 1, "bf16": 2}[io_name])
        worst, flips = max(worst, w_), flips + f_
    del layers
    torch.cuda.empty_cache()
    ms_all, _, ops_per_s = aggregate(ms * steps, flops * steps, world)
    ms = ms_all / steps
    hbm, bf16, bf16_s, kind = peaks()
    return {"value": round(ops_per_s / 1e12, 2), "unit": "TOPS", "ms_per_step": ms, "steps": steps,
            "warmup": warmup, "alg_GBps": alg_bytes * world / (ms * 1e-3) / 1e9,
            "tensor_frac": round(ops_per_s / 1e12 / bf16, 4),
            "tensor_frac_sustained": round(ops_per_s / 1e12 / bf16_s, 4),
            "hbm_frac": round(alg_bytes * world / (ms * 1e-3) / 1e9 / hbm, 4),
            "peaks": f"{kind}: bf16 dense {bf16} TFLOP/s burst, {bf16_s} sustained; HBM {hbm} GB/s",
            "config": {"workload": which, "tokens": M, "layers": n_layers, "io": io_name,
                       "projections": [f"{p.name} {p.K}->{p.N}" for p in shapes],
                       "launch": "eager, one stream; inputs larger than L2"},
            "parity": {"oracle_worst_row_rel_l2": worst, "rows_checked": 2 * len(rows), "codes_off_by_one": flips}}


def measure_point(args, world, local, M, K, N, steps=5, warmup=2):
    """One projection shape, cycling through distinct weight tensors (inputs
    larger than L2 through x and y), eager calls of bitnet_bitlinear_forward."""
    import torch

    import bitlinear_rmsnorm_token_gb300 as bn
    import oracle
    from bitlinear_rmsnorm_token_gb300 import workloads as wl

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    sets = []
    for i in range(4):
        w = wl.gen_device((N, K), wl.seed_for(4, K, N, i), device, std=0.02)
        sets.append(bn.pack_i2s(w))
        del w
    g = torch.from_numpy(wl.gen_norm_w(K, seed=K)).to(device)
    x = wl.gen_device((M, K), wl.seed_for(4, M, K, N), device)
    y = torch.empty((M, N), dtype=torch.float32, device=device)

    def cycle():
        for packed, sc in sets:
            bn.bitlinear_forward(x, g, packed, sc, N, wl.EPS, y, stream=stream)

    with torch.cuda.stream(stream):
        ms = time_region(torch, stream, cycle, steps, warmup) / len(sets)
    rows = np.random.default_rng(1).choice(M, 8, replace=False)
    packed, sc = sets[-1]
    worst, flips = sampled_row_parity(oracle, bn, x, g, packed, sc, N, y, rows)
    n_sets = len(sets)
    del sets, x, y
    torch.cuda.empty_cache()
    ms_all, _, ops_per_s = aggregate(ms * steps, 2.0 * M * N * K * steps, world)
    ms = ms_all / steps
    b = N * K / 4 + 4 + M * K * 4 + K * 4 + M * N * 4
    hbm, bf16, bf16_s, kind = peaks()
    return {"value": round(ops_per_s / 1e12, 2), "unit": "TOPS", "us_per_projection": ms * 1e3,
            "tensor_frac": round(ops_per_s / 1e12 / bf16, 4),
            "tensor_frac_sustained": round(ops_per_s / 1e12 / bf16_s, 4),
            "hbm_frac": round(b * world / (ms * 1e-3) / 1e9 / hbm, 4),
            "config": {"workload": f"proj_M{M}_K{K}_N{N}", "weights_cycled": n_sets,
                       "launch": "eager bitnet_bitlinear_forward, one stream"},
            "parity": {"oracle_worst_row_rel_l2": worst, "rows_checked": len(rows), "codes_off_by_one": flips}}


def run_prefill(args, rank, world, local, which):
    r = measure_prefill(args, world, local, which, args.io)
    out = {"metric": METRIC, "n_gpus": world}
    out.update(r)
    return out


def run_sweep(args, rank, world, local):
    """K, N in {1024, 4096, 8192, 16384} x M in {1, 16, 128, 2048, 16384}.  Each
    point cycles through enough distinct weight tensors to exceed twice the L2
    (at most 1024), one projection call per tensor.  Where every temporary of
    the allocating path's plan fits the no-alloc entry point's fixed scratch,
    the whole cycle is one CUDA graph of that entry point (kernel time, not
    Python launch time); otherwise calls are issued eagerly through
    bitnet_bitlinear_forward (those points run >= 80 us per call)."""
    import torch

    import bitlinear_rmsnorm_token_gb300 as bn
    from bitlinear_rmsnorm_token_gb300 import workloads as wl

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    hbm, bf16, _, _ = peaks()
    rows = []
    for K in wl.SWEEP_KN:
        for N in wl.SWEEP_KN:
            wb = N * K // 4
            nw = min(1024, max(1, int(np.ceil(2.0 * L2_BYTES / wb))))
            ws_list = []
            for i in range(nw):
                w = wl.gen_device((N, K), wl.seed_for(4, K, N, i), device, std=0.02)
                ws_list.append(bn.pack_i2s(w))
                del w
            g = torch.from_numpy(wl.gen_norm_w(K, seed=K)).to(device)
            for M in wl.SWEEP_M:
                x = wl.gen_device((M, K), wl.seed_for(4, M, K, N), device)
                y = torch.empty((M, N), dtype=torch.float32, device=device)
                graphed = noalloc_fits(bn, M, K, N)
                fwd = bn.bitlinear_forward_noalloc if graphed else bn.bitlinear_forward

                def cycle():
                    for packed, sc in ws_list:
                        fwd(x, g, packed, sc, N, wl.EPS, y, stream=stream)

                with torch.cuda.stream(stream):
                    cycle()  # warm-up (also checks every call)
                stream.synchronize()
                if graphed:
                    graph = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(graph, stream=stream):
                        cycle()
                    with torch.cuda.stream(stream):
                        ms = time_region(torch, stream, graph.replay, 3, 1) / nw
                    del graph
                else:
                    with torch.cuda.stream(stream):
                        ms = time_region(torch, stream, cycle, 1, 1) / nw
                b = wb + 4 + M * K * 4 + K * 4 + M * N * 4
                rows.append({"M": M, "K": K, "N": N, "us": ms * 1e3, "GBps": b / (ms * 1e-3) / 1e9,
                             "TOPS": 2.0 * M * N * K / (ms * 1e-3) / 1e12,
                             "hbm_frac": b / (ms * 1e-3) / 1e9 / hbm,
                             "tensor_frac": 2.0 * M * N * K / (ms * 1e-3) / 1e12 / bf16,
                             "weights_cycled": nw, "launch": "cuda graph" if graphed else "eager"})
                del x, y
            del ws_list
            torch.cuda.empty_cache()
    return {"metric": METRIC, "workload": "sweep", "rows": rows}


# ------------------------------------------------------------ reference

def run_reference(args, rank, world):
    """The oracle on the host cores, rank 0 only (other ranks do no work).  A
    step is one whole decode layer; W warm-up layers (at most 3: one oracle
    layer takes milliseconds) then up to K timed ones, bounded by --cpu-seconds."""
    if rank != 0:
        return None
    import oracle

    oracle.build()
    warm = min(args.warmup, 3)
    cb = cpu_baseline_decode(args, budget_s=None, max_steps=args.steps, warmup=warm)
    value = cb["value"]
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": cb["steps"], "steps_requested": args.steps, "warmup": warm,
            "ms_per_step": cb["seconds"] / max(1, cb["steps"]) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8 x ternary -> int64, fp32",
            "data": "synthetic",
            "config": decode_config(world),
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300000)
    ap.add_argument("--warmup", type=int, default=20000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_decode_layer",
                    choices=["qwen3_decode_layer", "q_proj_m8", "gemma3_prefill", "qwen3_prefill_stack", "sweep",
                             "proj", "glu_proj", "qk_proj"])
    ap.add_argument("--m", type=int, default=16, help="--workload proj: tokens")
    ap.add_argument("--k", type=int, default=16384, help="--workload proj: input features")
    ap.add_argument("--n", type=int, default=16384, help="--workload proj: output features")
    ap.add_argument("--act", type=int, default=1, help="--workload glu_proj: 1 SiLU, 2 tanh GELU")
    ap.add_argument("--head-dim", type=int, default=128, help="--workload qk_proj: values per head")
    ap.add_argument("--io", choices=["f32", "f16", "bf16"], default="f32",
                    help="prefill workloads: element type of x and y (bitnet_bitlinear_forward_typed)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="default workload: skip the prefill block")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    args.steps_ref = args.steps

    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    elif args.workload == "qwen3_decode_layer":
        out = run_decode(args, rank, world, local)
    elif args.workload == "q_proj_m8":
        out = run_q_proj_m8(args, rank, world, local)
    elif args.workload == "sweep":
        out = run_sweep(args, rank, world, local)
    elif args.workload == "proj":
        out = run_proj(args, rank, world, local)
    elif args.workload == "glu_proj":
        out = run_glu_proj(args, rank, world, local)
    elif args.workload == "qk_proj":
        out = run_qk_proj(args, rank, world, local)
    else:
        out = run_prefill(args, rank, world, local, args.workload)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
