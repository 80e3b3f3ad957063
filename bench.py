"""Benchmark: full-model decode weight sweep through the W4A16 GEMV.

Workload (one step): the M=1 decode weight sweep of a 35-layer, hidden-1536
model: per layer q 2048x1536, k 256x1536, v 256x1536, o 1536x2048, gate and up
Fx1536, down 1536xF (F = 6144 for layers 0-14, 12288 for 15-34), 4-bit codes in
groups of 32 with bf16 steps, bf16 activations, fp32 outputs. q|k|v and gate|up
read the same input and run as one fused call each (140 calls per sweep), in
per-layer dependency order, replayed as one CUDA graph. Inputs are seeded
synthetic data (SplitMix64 codes, |N(0,1)|*0.02+1e-4 steps, N(0,1) x).

Metric: GB/s of the sweep (algorithmic bytes: packed codes + steps + x + y,
divided by the device time of one sweep) and ms per sweep.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the plain CPU oracle (the reference arm of this build)
on a bounded sample of the same workload on the host cores.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

HIDDEN = 1536
LAYERS = 35
METRIC = "W4A16 GEMV GB/s & % of HBM roofline; ms per full-model decode weight sweep"
WORKLOAD = ("decode weight sweep, M=1: 35 layers, hidden 1536, q 2048/k 256/v 256/o 1536x2048/"
            "gate,up Fx1536/down 1536xF, F=6144 (layers 0-14) or 12288 (15-34); W4A16 g32")
PROJ = ("q", "k", "v", "o", "gate", "up", "down")


def ffn(layer: int) -> int:
    return 6144 if layer < 15 else 12288


def layer_shapes(layer: int):
    """(name, N, K) of the 7 projections of a layer, in decode order."""
    F = ffn(layer)
    return [("q", 2048, HIDDEN), ("k", 256, HIDDEN), ("v", 256, HIDDEN), ("o", HIDDEN, 2048),
            ("gate", F, HIDDEN), ("up", F, HIDDEN), ("down", HIDDEN, F)]


def seed_of(layer: int, proj: str) -> int:
    return 1 + 7 * layer + PROJ.index(proj)


def fused_stages(layer: int):
    """The 4 fused calls of a layer: (name, [member projections], N, K)."""
    F = ffn(layer)
    return [("qkv", ["q", "k", "v"], 2560, HIDDEN), ("o", ["o"], HIDDEN, 2048),
            ("gateup", ["gate", "up"], 2 * F, HIDDEN), ("down", ["down"], HIDDEN, F)]


def stage_bytes(N: int, K: int, M: int = 1) -> int:
    """Algorithmic bytes of one call: codes + steps + x + y."""
    return N * K // 2 + N * (K // 32) * 2 + M * K * 2 + M * N * 4


def sweep_bytes(M: int = 1) -> int:
    return sum(stage_bytes(N, K, M) for l in range(LAYERS) for _, _, N, K in fused_stages(l))


def sweep_weight_bytes() -> int:
    return sum(N * K // 2 + N * (K // 32) * 2 for l in range(LAYERS) for _, _, N, K in fused_stages(l))


# ----------------------------------------------------------------- data ----

class Sweep:
    """Device-resident sweep: per fused stage views qw/sc/x (inputs) and y
    (output). All inputs live in one contiguous device arena (stage by stage,
    each piece 256-byte aligned) and all outputs in another, so that the end-to-end
    step can move them with a few large copies; with keep_host a pinned host
    arena mirrors the input arena byte for byte."""

    ALIGN = 256

    def __init__(self, device, keep_host: bool, m: int = 1):
        import torch
        plan, off = [], 0

        def take(nbytes):
            nonlocal off
            o = off
            off += (nbytes + self.ALIGN - 1) // self.ALIGN * self.ALIGN
            return o

        for l in range(LAYERS):
            for name, members, N, K in fused_stages(l):
                o_q = take(N * K // 2)
                o_s = take(N * (K // 32) * 2)
                o_x = take(m * K * 2)
                plan.append((l, name, members, N, K, o_q, o_s, o_x))
        self.in_bytes = off
        self.arena = torch.empty(off, dtype=torch.uint8, device=device)
        ytot = sum(m * N for (_, _, _, N, _, _, _, _) in plan)
        self.y_arena = torch.empty(ytot, dtype=torch.float32, device=device)
        self.stages = []
        yo = 0
        for (l, name, members, N, K, o_q, o_s, o_x) in plan:
            qw = self.arena[o_q:o_q + N * K // 2].view(torch.int32).view(N, K // 8)
            sc = self.arena[o_s:o_s + N * (K // 32) * 2].view(torch.int16).view(N, K // 32)
            x = self.arena[o_x:o_x + m * K * 2].view(torch.int16).view(m, K)
            r = 0
            sc_host = np.empty((N, K // 32), dtype=np.uint16)
            for p in members:
                n_p = next(n for nm, n, _ in layer_shapes(l) if nm == p)
                synth.gen_qweight_torch(seed_of(l, p), n_p, K, device, out=qw[r:r + n_p])
                sc_host[r:r + n_p] = synth.gen_scales(seed_of(l, p), n_p, K)
                r += n_p
            sc.copy_(torch.from_numpy(sc_host.view(np.int16)))
            x.copy_(torch.from_numpy(synth.gen_x(seed_of(l, members[0]), m, K).view(np.int16)))
            y = self.y_arena[yo:yo + m * N].view(m, N)
            yo += m * N
            self.stages.append({"layer": l, "name": name, "N": N, "K": K, "qw": qw, "sc": sc, "x": x,
                                "y": y, "in_end": o_x + m * K * 2})
        if keep_host:
            self.arena_h = torch.empty(off, dtype=torch.uint8, pin_memory=True)
            self.arena_h.copy_(self.arena)
            self.y_h = torch.empty(ytot, dtype=torch.float32, pin_memory=True)

    def run(self, w4, stream=None):
        for st in self.stages:
            w4.w4a16_gemv(st["x"], st["qw"], st["sc"], out=st["y"], stream=stream)

    def chunks(self, n: int):
        """Split the stages into n runs of about equal input bytes: [(first, last+1, byte_end)]."""
        out, first, target = [], 0, self.in_bytes / n
        for i, st in enumerate(self.stages):
            if st["in_end"] >= target * (len(out) + 1) or i == len(self.stages) - 1:
                out.append((first, i + 1, st["in_end"]))
                first = i + 1
        return out


# --------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi samples during the timed region (SM clock and throttle reasons)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.reader = None

    def start(self):
        # nvidia-smi's samples come back through a pipe that a reader thread
        # drains as they arrive (no file, and the pipe never fills).
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.reader = threading.Thread(target=lambda: self.lines.extend(self.proc.stdout), daemon=True)
        self.reader.start()

    def count(self) -> int:
        """Samples received so far (None-safe when nvidia-smi is missing)."""
        return len(self.lines) if self.proc is not None else -1

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in list(self.lines):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------- reference ----

_ORACLE_INPUTS = {}


def _stage_inputs(l, members, K):
    """Host copies of one fused stage's x, codes and steps (cached across calls)."""
    key = (l, tuple(members))
    if key not in _ORACLE_INPUTS:
        x = synth.gen_x(seed_of(l, members[0]), 1, K)
        qws, scs = [], []
        for p in members:
            n_p = next(n for nm, n, _ in layer_shapes(l) if nm == p)
            qws.append(synth.gen_qweight(seed_of(l, p), n_p, K))
            scs.append(synth.gen_scales(seed_of(l, p), n_p, K))
        _ORACLE_INPUTS[key] = (x, np.concatenate(qws), np.concatenate(scs))
    return _ORACLE_INPUTS[key]


def oracle_sample(budget_s: float = 12.0, max_stages: int = 16 * LAYERS):
    """Time the fp64 CPU oracle over sweep stages, in sweep order, until ~budget_s of work.

    Stages are taken in the sweep's own order (layer 0 q|k|v, o, gate|up, down,
    layer 1, ...), at most max_stages of them, wrapping around the sweep if the
    budget is not used up. Returns (GB/s of algorithmic sweep bytes, description
    of the sample, seconds of oracle time).
    """
    import oracle
    order = [(l, st) for l in range(LAYERS) for st in fused_stages(l)]
    done_bytes, t_total, stages = 0, 0.0, 0
    while t_total < budget_s and stages < max_stages:
        l, (name, members, N, K) = order[stages % len(order)]
        x, qw, sc = _stage_inputs(l, members, K)
        t0 = time.perf_counter()
        oracle.gemm(x, qw, sc)
        t_total += time.perf_counter() - t0
        done_bytes += stage_bytes(N, K)
        stages += 1
    desc = (f"{stages} fused stages taken in sweep order, wrapping after all {len(order)} "
            f"({stages / len(order):.2f} sweeps, {done_bytes / 1e6:.1f} MB)")
    return done_bytes / t_total / 1e9, desc, t_total


def oracle_sample_all_cores(budget_s: float = 12.0):
    """The same oracle over the same stages, one worker thread per host core.

    The oracle's C routine runs outside the interpreter lock (ctypes), so the
    workers compute stages concurrently; each takes the next stage in sweep
    order until ~budget_s of wall time has passed. Inputs are drawn before the
    clock starts. Returns (GB/s of algorithmic bytes per wall second, threads,
    description)."""
    import oracle
    order = [(l, st) for l in range(LAYERS) for st in fused_stages(l)]
    inputs = [_stage_inputs(l, members, K) for l, (name, members, N, K) in order]
    threads = max(1, os.cpu_count() or 1)
    lock = threading.Lock()
    state = {"next": 0, "bytes": 0, "stages": 0}
    t0 = time.perf_counter()

    def worker():
        while time.perf_counter() - t0 < budget_s:
            with lock:
                i = state["next"]
                state["next"] += 1
            l, (name, members, N, K) = order[i % len(order)]
            x, qw, sc = inputs[i % len(order)]
            oracle.gemm(x, qw, sc)
            with lock:
                state["bytes"] += stage_bytes(N, K)
                state["stages"] += 1

    pool = [threading.Thread(target=worker) for _ in range(threads)]
    for t in pool:
        t.start()
    for t in pool:
        t.join()
    wall = time.perf_counter() - t0
    desc = (f"{state['stages']} fused stages in sweep order over {threads} threads "
            f"({state['bytes'] / 1e6:.1f} MB in {wall:.1f} s wall)")
    return state["bytes"] / wall / 1e9, threads, desc


def run_reference(args, rank, world):
    if rank != 0:
        return
    vals = []
    desc = ""
    for i in range(args.warmup + args.steps):
        gbs, desc, secs = oracle_sample(budget_s=4.0)
        if i >= args.warmup:
            vals.append(gbs)
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sweep_bytes() / (v * 1e9) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sweep_bytes": sweep_bytes()},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": desc + " per step; ms_per_step extrapolated to the full sweep"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- ours ----

def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def measure_rows(w4, dev, stream, sweep=None):
    """Per-row measurements beside the sweep (device time, CUDA events on the
    launching stream; decode calls replayed from a CUDA graph with programmatic
    dependent launch like the sweep; inputs larger than L2 or rotated through
    more than L2's worth of copies).

    Returns a dict keyed by row with us per call and GB/s (or TFLOP/s)."""
    import torch
    res = {}

    def graph_time(fn, reps=20):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps * 1e3  # us per replay

    def dev16(a):
        return torch.from_numpy(a.view(np.int16)).to(dev)

    # Single GEMV 2048x2048, M=1: 64 weight copies (154 MB) rotated.
    N, K, copies = 2048, 2048, 64
    qs = [synth.gen_qweight_torch(7000 + c, N, K, dev) for c in range(copies)]
    sc = dev16(synth.gen_scales(0, N, K))
    x = dev16(synth.gen_x(0, 1, K))
    y = torch.empty((1, N), dtype=torch.float32, device=dev)
    us = graph_time(lambda: [w4.w4a16_gemv(x, q, sc, out=y, stream=stream) for q in qs]) / copies
    b = stage_bytes(N, K)
    res["gemv_2048x2048_m1"] = {"us": us, "GBps": b / us / 1e3, "bytes": b}
    # The same with Hadamard-rotated weights (blocks of 256): x H formed by the
    # decode kernel while it stages x.
    us = graph_time(lambda: [w4.w4a16_gemv_hadamard(x, q, sc, 256, out=y, stream=stream) for q in qs]) / copies
    res["gemv_hadamard_2048x2048_b256"] = {"us": us, "GBps": b / us / 1e3, "bytes": b}
    del qs

    # Vocabulary projection 262144x1536 with the fused argmax (226 MB).
    N, K = 262144, 1536
    q = synth.gen_qweight_torch(1000, N, K, dev)
    sc = dev16(synth.gen_scales(1000, N, K))
    x = dev16(synth.gen_x(1000, 1, K))
    y = torch.empty((1, N), dtype=torch.float32, device=dev)
    am = torch.empty((1,), dtype=torch.int32, device=dev)
    us = graph_time(lambda: w4.w4a16_gemv_argmax(x, q, sc, out=y, argmax=am, stream=stream), reps=10)
    b = stage_bytes(N, K) + 4
    res["vocab_argmax_262144x1536"] = {"us": us, "GBps": b / us / 1e3, "bytes": b}
    # The same projection for 8 x-rows (8 sequences), a pick per x-row.
    x8 = dev16(synth.gen_x(1001, 8, K))
    y8 = torch.empty((8, N), dtype=torch.float32, device=dev)
    am8 = torch.empty((8,), dtype=torch.int32, device=dev)
    us = graph_time(lambda: w4.w4a16_gemv_argmax(x8, q, sc, out=y8, argmax=am8, stream=stream), reps=10)
    b = stage_bytes(N, K, 8) + 4 * 8
    res["vocab_argmax_262144x1536_m8"] = {"us": us, "GBps": b / us / 1e3, "bytes": b}
    del x8, y8, am8

    if sweep is not None:
        # One token's weight reads: the 140-call sweep then the vocabulary
        # projection with the greedy pick, in one graph (1184 MiB).
        def token():
            sweep.run(w4, stream)
            w4.w4a16_gemv_argmax(x, q, sc, out=y, argmax=am, stream=stream)
        us = graph_time(token, reps=10)
        b = sweep_bytes() + stage_bytes(N, K) + 4
        res["sweep_plus_vocab"] = {"us": us, "ms": us / 1e3, "GBps": b / us / 1e3, "bytes": b}

        # The same sweep unfused: q, k, v and gate, up as separate calls on row
        # slices of the fused matrices (245 calls per sweep instead of 140).
        calls = []
        for st in sweep.stages:
            members = next(m for nm, m, _, _ in fused_stages(st["layer"]) if nm == st["name"])
            r = 0
            for p in members:
                n_p = next(n for nm, n, _ in layer_shapes(st["layer"]) if nm == p)
                calls.append((st["x"], st["qw"][r:r + n_p], st["sc"][r:r + n_p], st["y"][:, r:r + n_p]))
                r += n_p

        def unfused():
            for (xx, qq, ss, yy) in calls:
                w4.w4a16_gemv(xx, qq, ss, out=yy, stream=stream)
        us = graph_time(unfused, reps=10)
        b = sum(stage_bytes(qq.shape[0], xx.shape[1]) for (xx, qq, ss, yy) in calls)
        res["sweep_unfused_245"] = {"us": us, "ms": us / 1e3, "GBps": b / us / 1e3, "bytes": b,
                                    "calls": len(calls)}

        # Every call of the sweep with Hadamard-rotated weights (blocks of 512,
        # as a model whose linear weights are all rotated would run).
        def rotated():
            for st in sweep.stages:
                w4.w4a16_gemv_hadamard(st["x"], st["qw"], st["sc"], 512, out=st["y"], stream=stream)
        us = graph_time(rotated, reps=10)
        b = sweep_bytes()
        res["sweep_hadamard_b512"] = {"us": us, "ms": us / 1e3, "GBps": b / us / 1e3, "bytes": b}

    # The LM head as the fastgemma card stores it: Hadamard-rotated, group 256,
    # with the activation's transform (blocks of 512) and the greedy pick.
    sc256 = dev16(synth.gen_scales(1000, N, K, 256))
    us = graph_time(lambda: w4.w4a16_gemv_hadamard(x, q, sc256, 512, group=256, out=y, argmax=am,
                                                   stream=stream), reps=10)
    b = N * K // 2 + N * (K // 256) * 2 + 2 * K + 4 * N + 4
    res["vocab_hadamard_g256_b512_argmax"] = {"us": us, "GBps": b / us / 1e3, "bytes": b}

    # Device-resident step plumbing on the tied 262144 x 1536 group-256 table
    # (embedding and LM head share it): the greedy LM head with and without a
    # forced token (a forced step reads no weight), the next-step prologue
    # (history, position, the token's embedding row) and, with the sweep, whole
    # token steps in both modes.
    forced = torch.full((1,), -1, dtype=torch.int32, device=dev)
    pos = torch.zeros((1,), dtype=torch.int32, device=dev)
    hist = torch.zeros((1 << 20,), dtype=torch.int32, device=dev)
    xn = torch.empty((1, K), dtype=torch.bfloat16, device=dev)

    def head():
        w4.w4a16_gemv_argmax_forced(x, q, sc256, forced, group=256, out=y, argmax=am, stream=stream)

    def prologue():
        w4.w4_decode_prologue(am, pos, q, sc256, group=256, x_next=xn, tokens=hist, stream=stream)

    b = N * K // 2 + N * (K // 256) * 2 + 2 * K + 4 * N + 4
    us = graph_time(head, reps=10)
    res["lm_head_g256_greedy"] = {"us": us, "GBps": b / us / 1e3, "bytes": b}
    forced.fill_(7)
    us = graph_time(lambda: [head() for _ in range(20)], reps=10) / 20
    res["lm_head_g256_forced_skip"] = {"us": us, "bytes_read": 4}
    us = graph_time(lambda: [prologue() for _ in range(50)], reps=10) / 50
    pos.zero_()
    res["decode_prologue_1536_g256"] = {"us": us, "bytes": K // 2 + (K // 256) * 2 + 2 * K + 16}
    if sweep is not None:
        forced.fill_(-1)
        us = graph_time(lambda: (sweep.run(w4, stream), head(), prologue()), reps=10)
        res["token_step_greedy"] = {"us": us, "ms": us / 1e3}
        forced.fill_(7)
        us = graph_time(lambda: (sweep.run(w4, stream), head(), prologue()), reps=10)
        res["token_step_forced"] = {"us": us, "ms": us / 1e3}
        pos.zero_()
    del q, sc, sc256, hist

    # M=8 decode sweep: the sweep's shapes with 8 x-rows per call.
    sw8 = Sweep(dev, keep_host=False, m=8)
    us = graph_time(lambda: sw8.run(w4, stream), reps=10)
    b = sweep_bytes(8)
    res["sweep_m8"] = {"us": us, "ms": us / 1e3, "GBps": b / us / 1e3, "bytes": b}
    del sw8

    # 4-bit row gather: 8 ids from the 262144 x 8960 per-layer table (1.32 GB).
    N, K = 262144, 8960
    qt = synth.gen_qweight_torch(2001, N, K, dev)
    st = dev16(synth.gen_scales(2001, N, K))
    ids = torch.from_numpy(synth.gen_ids(2002, 8, N).astype(np.int32)).to(dev)
    out = torch.empty((8, K), dtype=torch.bfloat16, device=dev)
    us = graph_time(lambda: w4.w4_embed_gather(ids, qt, st, out=out, stream=stream))
    b = 8 * (K // 2 + K // 16 + 2 * K)
    res["gather_8x8960"] = {"us": us, "GBps": b / us / 1e3, "bytes": b}
    ids = torch.from_numpy(synth.gen_ids(2003, 4096, N).astype(np.int32)).to(dev)
    out = torch.empty((4096, K), dtype=torch.bfloat16, device=dev)
    us = graph_time(lambda: w4.w4_embed_gather(ids, qt, st, out=out, stream=stream))
    b = 4096 * (K // 2 + K // 16 + 2 * K)
    res["gather_4096x8960"] = {"us": us, "GBps": b / us / 1e3, "bytes": b}
    del qt, st

    # Decode attention over a one-head key/value cache (8 query heads): the
    # full-length layer at 131072 slots x 512 (256 MiB of keys and values per
    # call, larger than L2) and the sliding layer's 512-slot ring x 256 (512 KB,
    # rotated through 512 copies).
    hbm = measured_peaks()[0]
    H, T, D = 8, 131072, 512
    q = dev16(synth.gen_attn_q(404, H, D))
    kh, vh = synth.gen_attn_kv(404, T, D)
    k, v = dev16(kh), dev16(vh)
    del kh, vh
    out = torch.empty((H, D), dtype=torch.float32, device=dev)
    us = graph_time(lambda: w4.w4_attn_decode(q, k, v, scale=D ** -0.5, out=out, stream=stream))
    b = 2 * T * D * 2 + H * D * 2 + H * D * 4
    res["attn_full_131072x512"] = {"us": us, "GBps": b / us / 1e3, "bytes": b,
                                   "frac_of_copy_peak": b / us / 1e3 / hbm}
    del k, v
    H, T, D, copies, qpos = 8, 512, 256, 512, 70000
    q = dev16(synth.gen_attn_q(405, H, D))
    kh, vh = synth.gen_attn_kv(405, T, D)
    k1, v1 = dev16(kh), dev16(vh)
    ks = [k1.clone() for _ in range(copies)]
    vs = [v1.clone() for _ in range(copies)]
    kp = torch.from_numpy(synth.ring_positions(qpos, T)).to(dev)
    us = graph_time(lambda: [w4.w4_attn_decode(q, ks[c], vs[c], kp, qpos=qpos, window=T, scale=D ** -0.5,
                                               out=out, stream=stream) for c in range(copies)], reps=5) / copies
    b = 2 * T * D * 2 + H * D * 2 + H * D * 4 + T * 4
    res["attn_ring_512x256"] = {"us": us, "GBps": b / us / 1e3, "bytes": b}
    # The sliding layer's append at a device position (ring slot of *pos).
    kn = k1[0].clone()
    vn = v1[0].clone()
    posd = torch.full((1,), 70001, dtype=torch.int32, device=dev)
    us = graph_time(lambda: [w4.w4_kv_append(ks[c], vs[c], kn, vn, posd, kpos=kp, stream=stream)
                             for c in range(64)], reps=10) / 64
    res["kv_append_ring_512x256"] = {"us": us, "bytes": 4 * D * 2 + 8}
    del ks, vs, k1, v1

    # Prefill GEMM, 1024 tokens, tensor-core bound: 8 weight copies rotated.
    peak_tf = measured_bf16_peak()
    for N, K in ((6144, 1536), (1536, 6144)):
        M = 1024
        qs = [synth.gen_qweight_torch(3000 + r, N, K, dev) for r in range(8)]
        sc = dev16(synth.gen_scales(3000, N, K))
        x = dev16(synth.gen_x(3002, M, K))
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        with torch.cuda.stream(stream):
            for r in range(3):
                w4.w4a16_gemm(x, qs[r], sc, out=y, stream=stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for r in range(40):
                w4.w4a16_gemm(x, qs[r % 8], sc, out=y, stream=stream)
            e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / 40 * 1e3
        tf = 2.0 * M * N * K / us / 1e6
        res[f"prefill_{M}x{N}x{K}"] = {"us": us, "TFLOPs": tf, "roofline": {
            "bound": "tensor", "achieved": tf, "peak": peak_tf[0], "unit": "TFLOP/s", "frac": tf / peak_tf[0],
            "peak_source": peak_tf[1]}}
        del qs
    torch.cuda.empty_cache()
    return res


def measured_bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), "measured bf16 burst (MEASURED_PEAKS.json bf16_tflops)"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback bf16 burst"


def captured_traffic():
    """DRAM bytes (read + write) of one sweep from the committed ncu capture, or
    None when the decode kernel's sources changed after that capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "w4_decode_sweep_m1_35layers_traffic.json")) as f:
            rec = json.load(f)
        h = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != rec["sources_sha256"]:
            return None
        return int(rec["dram_bytes_read"]) + int(rec["dram_bytes_write"])
    except (OSError, KeyError, ValueError):
        return None


def max_over_ranks(t_ms: float, world: int, device) -> float:
    """The slowest rank's time (all_reduce MAX over the default process group when
    world > 1): the job's time, as every rank sees it."""
    if world <= 1:
        return t_ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([t_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(t_ms: float, nbytes: int, world: int) -> float:
    """Whole-job GB/s: every rank moved nbytes in the slowest rank's time."""
    return world * nbytes / (t_ms * 1e-3) / 1e9


def run_ours(args, rank, world):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    __graft_entry__.build()
    import bit_weight_only_w4a16_gb300 as w4

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w4.init()
    stream = torch.cuda.Stream(device=dev)

    sweep = Sweep(dev, keep_host=True)
    nbytes = sweep_bytes()
    ncalls = len(sweep.stages)

    # Capture the sweep once; every step replays the graph.
    with torch.cuda.stream(stream):
        sweep.run(w4, stream)  # warm the library (and any lazy set-up) outside capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        sweep.run(w4, stream)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(3, args.warmup)):
        with torch.cuda.stream(stream):
            g.replay()
    torch.cuda.synchronize()

    # The timed block of K steps is repeated (each block timed on its own with
    # events) until the clock sampler holds >= 10 samples under load, so that
    # the clock record stands on its own; the line reports the median block.
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    block_ms = []
    t_wall = time.time()
    while True:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(args.steps):
                g.replay()
            ev1.record(stream)
        torch.cuda.synchronize()
        block_ms.append(ev0.elapsed_time(ev1) / args.steps)
        n_clk = clocks.count()
        if n_clk < 0 or n_clk >= 10 or time.time() - t_wall > 20.0:
            break
    barrier()
    clk = clocks.stop()
    t_ms = max_over_ranks(statistics.median(block_ms), world, dev)
    value = job_rate(t_ms, nbytes, world)

    # In-run read ceiling: the plain-sum probe over a 4 GiB buffer.
    probe_buf = torch.empty(1 << 30, dtype=torch.int32, device=dev)
    probe_buf.fill_(1)
    with torch.cuda.stream(stream):
        for _ in range(3):
            w4.hbm_read_probe(probe_buf, stream=stream)
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for _ in range(10):
            w4.hbm_read_probe(probe_buf, stream=stream)
        p1.record(stream)
    torch.cuda.synchronize()
    probe_gbs = probe_buf.numel() * 4 / (p0.elapsed_time(p1) / 10 * 1e-3) / 1e9
    del probe_buf
    torch.cuda.empty_cache()

    rows = measure_rows(w4, dev, stream, sweep) if args.rows else None

    # End to end through the public call with host buffers: every step copies
    # the sweep's packed weights, steps and x from pinned host memory and reads
    # every y back. Copies of stage s+1 overlap the GEMV of stage s.
    e2e = None
    if args.e2e:
        # One copy stream: two or four streams measured no faster (the pinned
        # host-to-device path tops out near 230 GB/s on this machine either way).
        ncopy = 1
        cstreams = [torch.cuda.Stream(device=dev) for _ in range(ncopy)]
        h2d = sweep.in_bytes
        d2h = sweep.y_h.numel() * 4
        chunks = sweep.chunks(8)

        def e2e_step():
            # Inputs: a few large host-to-device copies of the pinned arena (one
            # per run of stages, alternating over the copy streams); each run's
            # GEMVs start as soon as its copy lands, overlapping later copies.
            # Outputs: one device-to-host copy.
            ready, prev = [], 0
            for i, (_, _, end) in enumerate(chunks):
                cs = cstreams[i % ncopy]
                with torch.cuda.stream(cs):
                    sweep.arena[prev:end].copy_(sweep.arena_h[prev:end], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(cs)
                    ready.append(e)
                prev = end
            with torch.cuda.stream(stream):
                for (first, last, _), e in zip(chunks, ready):
                    stream.wait_event(e)
                    for st in sweep.stages[first:last]:
                        w4.w4a16_gemv(st["x"], st["qw"], st["sc"], out=st["y"], stream=stream)
                sweep.y_h.copy_(sweep.y_arena, non_blocking=True)
            for cs in cstreams:
                cs.wait_stream(stream)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        # Three timed blocks; the median block is reported (the host link is
        # shared with other jobs on the machine, and one block of ~50 ms can
        # catch a burst of their traffic), every block's time beside it.
        e2e_steps = max(2, min(args.steps, 10))
        blocks = []
        for _ in range(3):
            q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            q0.record(stream)
            for cs in cstreams:
                cs.wait_stream(stream)  # every copy of the timed steps starts after q0
            for _ in range(e2e_steps):
                e2e_step()
            for cs in cstreams:
                stream.wait_stream(cs)
            q1.record(stream)
            torch.cuda.synchronize()
            blocks.append(max_over_ranks(q0.elapsed_time(q1) / e2e_steps, world, dev))
        te = sorted(blocks)[1]
        e2e = {"value": job_rate(te, nbytes, world), "unit": "GB/s", "ms_per_step": te,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "blocks_ms_per_step": blocks, "steps_per_block": e2e_steps}

    cpu = cpu_all = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, desc, secs = oracle_sample()
        cpu = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": desc + f", {secs:.1f} s single-threaded fp64"}
        gbs_all, nthr, desc_all = oracle_sample_all_cores()
        cpu_all = {"value": gbs_all, "unit": "GB/s", "cores": nthr, "kind": "oracle", "sample": desc_all}

    peak, peak_src = measured_peaks()
    achieved = nbytes / (t_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": t_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 x int4 -> f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "calls_per_sweep": ncalls, "fused": "q|k|v and gate|up",
                   "launch": "one CUDA graph per sweep, programmatic dependent launch",
                   "num_sms": torch.cuda.get_device_properties(dev).multi_processor_count,
                   "sweep_bytes": nbytes, "weight_bytes": sweep_weight_bytes(),
                   "l2": "inputs larger than L2 (1.02 GB per sweep vs 129 MB)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": captured_traffic(),
                     "traffic_unit": "bytes per sweep (140 launches), ncu dram__bytes_read.sum + "
                                     "dram__bytes_write.sum; null if the kernel changed since",
                     "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "kernel": "w4_decode_slab_kernel (q|k|v, gate|up, down) and w4_decode_m1_kernel (o 1536x2048): all 140 launches of the sweep"},
        "probe": {"hbm_read_probe_gbs": probe_gbs, "sweep_frac_of_probe": achieved / probe_gbs},
        "rows": rows,
        "gpu_launches": ncalls * args.steps * len(block_ms),
        "timed_blocks": {"blocks": len(block_ms), "steps_per_block": args.steps,
                         "ms_per_step_each": block_ms, "reported": "median block (max over ranks)"},
        "clocks": clk,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_ncu_case(case: str):
    """One small fixed case for an ncu capture: no timing, no output but "ok".

    sweep         : the 140 calls of one M=1 decode weight sweep, launched eagerly once.
    decode_shapes : w4a16_gemv, M=1, twice on each of (24576,1536) (1536,12288)
                    (2560,1536) (1536,2048) (1536,6144), writing a 256 MB buffer
                    between calls.
    m8_shapes     : (24576,1536) (1536,12288) (2560,1536) with M=8.
    vocab         : w4a16_gemv_argmax twice on the 262144 x 1536 vocabulary projection.
    m8_vocab      : the same with M=8 x-rows.
    m8_ragged     : w4a16_gemv, M=8, twice on 4096 x 1056 (K not a multiple of 128:
                    the 32-bit-load M <= 8 form).
    Every case ends with hbm_read_probe over 1 GiB (the in-capture read ceiling).
    gather_probe  : w4_embed_gather of 8 ids from the 262144 x 8960 table and
                    hbm_read_probe over 1 GiB, twice each.
    attn          : w4_attn_decode twice over a 131072-slot x 512 cache (8 heads).
    hadamard      : w4a16_gemv_hadamard (blocks of 512, group 256, argmax) twice on
                    the 262144 x 1536 vocabulary projection.
    prefill:NxK   : w4a16_gemm twice with M=1024 tokens on an N x K weight.
    """
    import torch
    import __graft_entry__
    __graft_entry__.build()
    import bit_weight_only_w4a16_gb300 as w4
    torch.cuda.set_device(0)
    w4.init()
    dev = torch.device("cuda", 0)

    def problem(seed, M, N, K):
        x = torch.from_numpy(synth.gen_x(seed + 2, M, K).view(np.int16)).to(dev)
        q = synth.gen_qweight_torch(seed, N, K, dev)
        sc = torch.from_numpy(synth.gen_scales(seed, N, K).view(np.int16)).to(dev)
        return x, q, sc

    if case == "sweep":
        # The 140 calls of one M=1 decode weight sweep, launched eagerly once (ncu's
        # launch list of graph-replayed nodes failed to launch the shared-memory
        # slot kernel; eager launches profile normally).
        sweep = Sweep(dev, keep_host=False)
        s = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(s):
            sweep.run(w4, s)
        torch.cuda.synchronize()
    elif case == "hadamard":
        N, K = 262144, 1536
        q = synth.gen_qweight_torch(1000, N, K, dev)
        sc = torch.from_numpy(synth.gen_scales(1000, N, K, 256).view(np.int16)).to(dev)
        x = torch.from_numpy(synth.gen_x(1000, 1, K).view(np.int16)).to(dev)
        for _ in range(2):
            w4.w4a16_gemv_hadamard(x, q, sc, 512, group=256, argmax=True)
    elif case == "step":
        # One device-resident decode step of a sliding layer, twice: append into
        # the 512-slot ring x 256 at the device position, attention at it, the
        # group-256 LM head (262144 x 1536) with the forced-token form (not
        # forced, then forced), the prologue.
        H, T, D, N, K = 8, 512, 256, 262144, 1536
        q = torch.from_numpy(synth.gen_attn_q(405, H, D).view(np.int16)).to(dev)
        kh, vh = synth.gen_attn_kv(405, T, D)
        k = torch.from_numpy(kh.view(np.int16)).to(dev)
        v = torch.from_numpy(vh.view(np.int16)).to(dev)
        kp = torch.from_numpy(synth.ring_positions(70000, T)).to(dev)
        pos = torch.full((1,), 70001, dtype=torch.int32, device=dev)
        lq = synth.gen_qweight_torch(1000, N, K, dev)
        ls = torch.from_numpy(synth.gen_scales(1000, N, K, 256).view(np.int16)).to(dev)
        x = torch.from_numpy(synth.gen_x(1000, 1, K).view(np.int16)).to(dev)
        forced = torch.full((1,), -1, dtype=torch.int32, device=dev)
        for rep in range(2):
            forced.fill_(-1 if rep == 0 else 7)
            w4.w4_kv_append(k, v, k[0].clone(), v[0].clone(), pos, kpos=kp)
            w4.w4_attn_decode(q, k, v, kp, qpos=pos, window=T, scale=D ** -0.5)
            _, tok = w4.w4a16_gemv_argmax_forced(x, lq, ls, forced, group=256)
            w4.w4_decode_prologue(tok, pos, lq, ls, group=256)
            torch.cuda.synchronize()
    elif case == "attn":
        H, T, D = 8, 131072, 512
        q = torch.from_numpy(synth.gen_attn_q(404, H, D).view(np.int16)).to(dev)
        kh, vh = synth.gen_attn_kv(404, T, D)
        k = torch.from_numpy(kh.view(np.int16)).to(dev)
        v = torch.from_numpy(vh.view(np.int16)).to(dev)
        for _ in range(2):
            w4.w4_attn_decode(q, k, v, scale=D ** -0.5)
    elif case in ("vocab", "m8_vocab"):
        x, q, sc = problem(1000, 1 if case == "vocab" else 8, 262144, 1536)
        for _ in range(2):
            w4.w4a16_gemv_argmax(x, q, sc)
    elif case == "m8_ragged":
        x, q, sc = problem(210, 8, 4096, 1056)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        for rep in range(2):
            flush.fill_(rep)
            w4.w4a16_gemv(x, q, sc)
    elif case == "m8_shapes":
        data = [problem(200 + i, 8, N, K) for i, (N, K) in enumerate([(24576, 1536), (1536, 12288), (2560, 1536)])]
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        for rep in range(2):
            for x, q, sc in data:
                flush.fill_(rep)
                w4.w4a16_gemv(x, q, sc)
    elif case == "gather_probe":
        N, K = 262144, 8960
        qt = synth.gen_qweight_torch(2001, N, K, dev)
        st = torch.from_numpy(synth.gen_scales(2001, N, K).view(np.int16)).to(dev)
        ids = torch.from_numpy(synth.gen_ids(2002, 8, N).astype(np.int32)).to(dev)
        buf = torch.ones(1 << 28, dtype=torch.int32, device=dev)
        for _ in range(2):
            w4.w4_embed_gather(ids, qt, st)
            w4.hbm_read_probe(buf)
    elif case == "decode_shapes":
        data = [problem(100 + i, 1, N, K) for i, (N, K) in
                enumerate([(24576, 1536), (1536, 12288), (2560, 1536), (1536, 2048), (1536, 6144)])]
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        for rep in range(2):
            for x, q, sc in data:
                flush.fill_(rep)
                w4.w4a16_gemv(x, q, sc)
    elif case.startswith("prefill:"):
        N, K = (int(v) for v in case.split(":")[1].split("x"))
        x, q, sc = problem(3000, 1024, N, K)
        for _ in range(2):
            w4.w4a16_gemm(x, q, sc)
    else:
        raise SystemExit(f"unknown --ncu-case {case}")
    probe = torch.ones(1 << 28, dtype=torch.int32, device=dev)
    w4.hbm_read_probe(probe)
    torch.cuda.synchronize()
    print("ok")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rows", dest="rows", action="store_false",
                    help="skip the per-row measurements (single GEMV, vocabulary argmax, M=8 sweep, "
                         "gather, prefill)")
    ap.add_argument("--ncu-case", default=None,
                    help="run one small fixed case for an ncu capture instead of the bench: "
                         "sweep | decode_shapes | m8_shapes | vocab | gather_probe | attn | hadamard | step | prefill:NxK")
    args = ap.parse_args()
    if args.ncu_case:
        run_ncu_case(args.ncu_case)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
