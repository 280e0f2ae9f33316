#!/usr/bin/env python
"""WKV7 forward + checkpointed backward throughput on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the whole path on one batch of the 36M "debug" training
shape (B=12, T=1024, H=6, D=64, bf16 inputs, fp32 state, chunk 32): wkv7_forward
(y, checkpoints, hT) with a workspace, then wkv7_backward_from_forward (dr, dw, dk,
dv, da, db, dh0) on the operators that forward left in it (--path operators, the
default; --path operators-reform has wkv7_backward form them again, --path two-phase
and --path single time the other backward paths).  other_configs adds the step time and
step roofline fractions of the other training workloads.  Inputs are
seeded synthetic draws (wkv7_inputs.py).  Under torchrun each rank runs its own
independent batch (weak scaling, no collective on the data path); rank 0 prints
one JSON line.

--impl reference times the fp64 CPU oracle on this host's cores instead, on a
bounded sample of the same workload, in the same unit.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import wkv7_inputs as gen  # noqa: E402

METRIC = "WKV7 fwd+bwd tokens/s at B12 T1024 H6 D64; % of FP32/HBM roofline"
WORKLOAD = "debug_b12_t1024_h6"
N_SETS = 4  # input/output sets rotated between steps so a step never finds its inputs in L2
FALLBACK_HBM_GBS = 6400.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle CPU-baseline budget")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--workload", default=WORKLOAD, choices=sorted(gen.WORKLOADS),
                   help="default: the debug training shape (the headline line); others for extra measurements")
    p.add_argument("--decode-batch", type=int, default=0,
                   help="decode workload only: number of sequences (default: the workload's 256)")
    p.add_argument("--path", choices=list(PATHS), default="operators",
                   help="operators: chunk-operator forward with a workspace, then the backward on the operators "
                        "it left there (the default); operators-reform: the backward forms them again "
                        "(wkv7_backward with a workspace, no sa); two-phase: forward saving sa, two-phase "
                        "backward reading it; single: single-pass backward without a workspace")
    p.add_argument("--graph", choices=["on", "off"], default="on",
                   help="time the step as CUDA-graph replays (one graph per input set) instead of eager calls")
    p.add_argument("--no-other-configs", action="store_true",
                   help="skip the step times of the other training workloads (other_configs in the line)")
    return p.parse_args()


# ------------------------------------------------------------------------------ workload math

def byte_counts(wl, in_bytes: int):
    """Minimum HBM bytes the method must move (forward, backward), per step."""
    N = wl.B * wl.T * wl.H * wl.D
    C = math.ceil(wl.T / wl.chunk)
    S = wl.B * wl.H * wl.D * wl.D * 4
    h0 = S if wl.h0_std else 0
    dhT = S if wl.dhT_std else 0
    fwd = 6 * N * in_bytes + h0 + 4 * N + C * S + S
    bwd = 6 * N * in_bytes + 4 * N + (C - 1) * S + h0 + dhT + 6 * 4 * N + S
    return fwd, bwd


def literal_flops(wl):
    return 8 * wl.D * wl.D * wl.B * wl.T * wl.H


def derived_flops(wl):
    """FLOPs of forward + backward as the recurrences are written: ~28 D^2 per head-token."""
    return 28 * wl.D * wl.D * wl.B * wl.T * wl.H


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured", d
    return FALLBACK_HBM_GBS, "fallback", {}


def workload_config(wl) -> dict:
    """The `config` object of both arms' lines: the workload alone (how the step runs is in `path`)."""
    fwd_b, bwd_b = byte_counts(wl, 2 if wl.dtype == "bf16" else 4)
    return {"workload": wl.name, "B": wl.B, "T": wl.T, "H": wl.H, "D": wl.D, "chunk": wl.chunk, "inputs": wl.dtype,
            "state": "fp32", "l2": f"{N_SETS} rotating input/output sets "
                                   f"({N_SETS * (fwd_b + bwd_b) / 1e9:.2f} GB touched per rotation > 126 MB L2)"}


# ------------------------------------------------------------------------------ ranks

def max_over_ranks(value: float, device) -> float:
    """The largest `value` over all ranks of the default process group (the slowest replica
    sets the job's time); `value` itself when no group is initialised."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(per_rank_tokens: int, world: int, elapsed_ms_max: float) -> float:
    """Whole-job throughput: every rank processes its own batch (weak scaling)."""
    return world * per_rank_tokens / (elapsed_ms_max / 1e3)


# ------------------------------------------------------------------------------ clocks

class ClockSampler:
    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,"
                   "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
                   "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                   "clocks_event_reasons.sw_power_cap", "--format=csv,noheader,nounits", "-lms", "100"]
            if self.uuid:
                cmd[1:1] = ["-i", self.uuid]
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            c = [x.strip() for x in line.split(",")]
            if len(c) < 9:
                continue
            try:
                sms.append(float(c[1]))
                mx = float(c[2])
            except ValueError:
                continue
            for n, v in zip(names, c[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sms)}


# ------------------------------------------------------------------------------ oracle (CPU)

def oracle_pass(wl, heads, xs_by_b):
    """fp64 oracle forward + checkpointed backward over the given (b, h) heads."""
    import oracle
    for b, h in heads:
        x, dy = xs_by_b[b]
        sl = {n: x[n][None, :, h:h + 1] for n in "rwkvab"}
        _, ck, _ = oracle.forward(*(sl[n] for n in "rwkvab"), None, chunk=wl.chunk)
        oracle.backward(*(sl[n] for n in "rwkvab"), None, ck, dy[None, :, h:h + 1], None,
                        chunk=wl.chunk, mode="ckpt")


_POOL_INPUTS = {}


def _pool_init(name: str):
    """Worker start-up (outside any timed region): draw this workload's inputs once."""
    wl = gen.WORKLOADS[name]
    for b in range(wl.B):
        _POOL_INPUTS[b] = (gen.token_inputs(wl, b), gen.dy_init(wl, b))
    import oracle
    oracle.default()


def _pool_head(task):
    name, b, h = task
    oracle_pass(gen.WORKLOADS[name], [(b, h)], _POOL_INPUTS)
    return 1


def oracle_pool(wl):
    """A spawned process pool (no inherited CUDA state) with one worker per core, up to one per head."""
    import multiprocessing as mp
    n = max(1, min(os.cpu_count() or 1, wl.B * wl.H))
    return mp.get_context("spawn").Pool(n, initializer=_pool_init, initargs=(wl.name,)), n


def pool_pass(pool, wl, heads):
    pool.map(_pool_head, [(wl.name, b, h) for b, h in heads], chunksize=1)


def cpu_baseline(wl, seconds: float):
    """The oracle on the host's cores: all heads of the workload over a spawned pool (one head per task),
    plus the same single-threaded, both for a bounded time."""
    xs = {b: (gen.token_inputs(wl, b), gen.dy_init(wl, b)) for b in range(wl.B)}
    heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
    oracle_pass(wl, heads[:1], xs)  # build + warm
    done, t0 = 0, time.perf_counter()
    while True:
        oracle_pass(wl, heads, xs)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    single = {"value": done * wl.B * wl.T / el, "cores": 1, "passes": done}
    what = (f"all {len(heads)} heads of {wl.name} (B{wl.B} T{wl.T} H{wl.H} D{wl.D}), fp64 forward + "
            f"checkpoint-recompute backward in the oracle's C")
    try:
        pool, n = oracle_pool(wl)
    except Exception as e:  # no process pool on this host: the single-threaded figure stands alone
        return {"value": single["value"], "unit": "tokens/s", "cores": 1, "kind": "oracle",
                "sample": f"{what}, {done} pass(es), single-threaded (process pool unavailable: {e})"}
    with pool:
        pool_pass(pool, wl, heads)  # warm every worker
        pdone, t0 = 0, time.perf_counter()
        while True:
            pool_pass(pool, wl, heads)
            pdone += 1
            pel = time.perf_counter() - t0
            if pel >= seconds / 2:
                break
    return {"value": pdone * wl.B * wl.T / pel, "unit": "tokens/s", "cores": n, "kind": "oracle",
            "sample": f"{what}, {pdone} pass(es) over {n} single-threaded worker processes (one head per task; "
                      f"os.cpu_count() = {os.cpu_count()})",
            "single_thread": single}


def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = gen.WORKLOADS[args.workload]
    if wl.decode:
        print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the training workloads only"}))
        return
    # bounded sample: per step as many heads as there are workers (at most all of them), so a step is one
    # round of the pool whatever the core count; the value is scaled to whole-batch tokens/s
    pool, n = oracle_pool(wl)
    heads = [(b, h) for b in range(wl.B) for h in range(wl.H)][:n]
    frac = len(heads) / (wl.B * wl.H)
    with pool:
        for _ in range(args.warmup):
            pool_pass(pool, wl, heads)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            pool_pass(pool, wl, heads)
        el = time.perf_counter() - t0
    value = args.steps * frac * wl.B * wl.T / el
    sample = (f"{len(heads)} of {wl.B * wl.H} heads of {wl.name} per step (fp64 forward + checkpoint-recompute "
              f"backward in the oracle's C, one head per single-threaded worker process, {n} workers); value "
              f"scaled to whole-batch tokens/s")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, wkv7_inputs.py)",
            "config": workload_config(wl),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": n, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ GPU arm

def decode_bytes(wl, in_bytes: int):
    """Minimum HBM bytes of one decode step: state read + write, six inputs, y."""
    n = wl.B * wl.H * wl.D
    return 2 * wl.B * wl.H * wl.D * wl.D * 4 + 6 * n * in_bytes + 4 * n


def run_decode(args, rank, world, local_rank):
    """7B decode: every step advances all B sequences by one token through all 32 x 64 heads, in place."""
    import torch
    import linear_rnn_lm_wkv7_b300 as wkv7

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = gen.WORKLOADS[args.workload]
    if args.decode_batch > 0:
        import dataclasses
        wl = dataclasses.replace(wl, B=args.decode_batch)
    B, H, D = wl.B, wl.H, wl.D
    rows = [gen.token_inputs(wl, b) for b in range(B)]
    host_in = {n: torch.from_numpy(np.stack([rw[n][0] for rw in rows])).to(torch.bfloat16) for n in "rwkvab"}
    ins = {n: t.to(dev) for n, t in host_in.items()}
    g = torch.Generator(device=dev)
    g.manual_seed(wl.seed)
    state = torch.randn((B, H, D, D), generator=g, device=dev) * wl.h0_std   # 8.6 GB, > L2: no flush needed
    y = torch.empty((B, H, D), device=dev)
    stream = torch.cuda.current_stream()

    def step():
        wkv7.decode(state, *(ins[n] for n in "rwkvab"), y=y)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    with ClockSampler(uuid) as clk:
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    clocks = clk.summary()
    ms = max_over_ranks(e0.elapsed_time(e1), dev) / args.steps
    # end to end: inputs from pinned host memory, y back to the host; the state stays resident
    pin_in = {n: t.pin_memory() for n, t in host_in.items()}
    pin_y = torch.empty((B, H, D), pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in pin_in.values())
    d2h = pin_y.numel() * 4

    def e2e_step():
        for n in "rwkvab":
            ins[n].copy_(pin_in[n], non_blocking=True)
        step()
        pin_y.copy_(y, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(max(1, args.e2e_steps)):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev) / max(1, args.e2e_steps)

    # The same step as one call per layer (H = 64 heads each, separate per-layer states and inputs),
    # the calls captured once in a CUDA graph and replayed: how a model's decode loop would issue them.
    nbytes = decode_bytes(wl, 2)
    per_layer = None
    if H > 64 and H % 64 == 0:
        nl, err, lms = H // 64, None, 0.0
        try:
            lst = [state[:, 64 * l:64 * (l + 1)].contiguous() for l in range(nl)]
            lin = [{n: ins[n][:, 64 * l:64 * (l + 1)].contiguous() for n in "rwkvab"} for l in range(nl)]
            ly = [torch.empty((B, 64, D), device=dev) for _ in range(nl)]

            def layers():
                for l in range(nl):
                    wkv7.decode(lst[l], *(lin[l][n] for n in "rwkvab"), y=ly[l])

            side = torch.cuda.Stream(dev)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                for _ in range(3):
                    layers()
            stream.wait_stream(side)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                layers()
            for _ in range(3):
                graph.replay()
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            lms = e0.elapsed_time(e1) / args.steps
            del lst, lin, ly, graph
        except Exception as e:  # reported in the line; every rank still joins the max below
            err = f"{type(e).__name__}: {e}"[:300]
        lms = max_over_ranks(lms, dev)
        per_layer = {"layers": nl, "heads_per_layer": 64, "error": err} if err else {
            "layers": nl, "heads_per_layer": 64, "launch": f"{nl} wkv7_decode calls per step in one CUDA graph",
            "ms_per_step": lms, "value": world * B / (lms / 1e3), "unit": "tokens/s",
            "achieved_gbs": nbytes / (lms / 1e3) / 1e9}
    if rank != 0:
        return
    hbm, peak_kind, _ = measured_peaks()
    achieved = nbytes / (ms / 1e3) / 1e9
    line = {
        "metric": "WKV7 decode tokens/s (7B state: 32 layers x 64 heads x 64x64 fp32 per sequence)",
        "value": world * B / (ms / 1e3), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded: inputs wkv7_inputs.py, state torch.randn)",
        "config": {"workload": wl.name, "B": B, "H": H, "D": D, "inputs": "bf16", "state": "fp32, in place",
                   "l2": f"state {B * H * D * D * 4 / 1e9:.1f} GB > 126 MB L2"},
        "roofline": {"bound": "hbm", "kernel": "wkv7_decode", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": None, "algorithmic_bytes": nbytes, "avg_launch_ms": ms},
        "clocks": clocks, "gpu_launches": args.steps,
        "e2e": {"value": world * B / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
    }
    if per_layer is not None:
        line["per_layer_graph"] = per_layer
    print(json.dumps(line), flush=True)


PATHS = {
    # forward call, backward call and the kernels each launches (counted per step for gpu_launches)
    "operators": {"forward": "wkv7_forward with a workspace, no sa: chunk-operator prep + chain",
                  "backward": "wkv7_backward_from_forward on the forward's workspace: E_c kernel + walk (with "
                              "whole-head chain CTAs, past 74 heads on 148 SMs: the walk forming E_c itself, no E_c "
                              "kernel) + matrix column kernel + token-by-token companion (exits at once without "
                              "flagged chunks)",
                  "backward_call": "wkv7_backward_from_forward",
                  # two 32-row chain CTAs per head while 2 x heads fit the SMs, else whole heads
                  "launches": lambda heads, sms: 2 + (4 if 2 * heads <= sms else 3)},
    "operators-reform": {"forward": "wkv7_forward with a workspace, no sa: chunk-operator prep + chain",
                         "backward": "wkv7_backward with a workspace, no sa: operator prep + walk + matrix column "
                                     "kernel + token-by-token companion",
                         "launches": 2 + 4},
    "two-phase": {"forward": "wkv7_forward saving sa: 16-token sub-chunks (one wave) or token by token",
                  "backward": "wkv7_backward with sa and a workspace: sub-chunk walk + column passes",
                  "launches": 1 + 2},
    "single": {"forward": "wkv7_forward saving sa: 16-token sub-chunks (one wave) or token by token",
               "backward": "wkv7_backward without a workspace: single pass (rebuilds states dividing by w)",
               "launches": 1 + 1},
}


def make_runner(wkv7, torch, dev, wl, path, n_sets):
    """Input/output sets on the device and the step (forward then backward) of one path."""
    B, T, H, D = wl.B, wl.T, wl.H, wl.D
    C = wkv7.num_chunks(T, wl.chunk)
    x = gen.full(wl)
    host_in = {n: torch.from_numpy(x[n]).to(torch.bfloat16 if wl.dtype == "bf16" else torch.float32)
               for n in "rwkvab"}
    host = {"in": host_in, "dy": torch.from_numpy(x["dy"]),
            "h0": None if x["h0"] is None else torch.from_numpy(x["h0"]),
            "dhT": None if x["dhT"] is None else torch.from_numpy(x["dhT"])}
    del x
    operators = path.startswith("operators")
    saved = not operators
    ws_bytes = 0
    if path == "operators":
        ws_bytes = wkv7.forward_workspace_size(B, T, H, D, wl.chunk)
    elif path == "operators-reform":
        ws_bytes = max(wkv7.forward_workspace_size(B, T, H, D, wl.chunk), wkv7.backward_workspace_size(B, T, H, D, wl.chunk))
    elif path == "two-phase":
        ws_bytes = wkv7.backward_workspace_size(B, T, H, D, wl.chunk)

    def make_set():
        s = {n: host_in[n].to(dev) for n in "rwkvab"}
        s["dy"] = host["dy"].to(dev)
        s["h0"] = None if host["h0"] is None else host["h0"].to(dev)
        s["dhT"] = None if host["dhT"] is None else host["dhT"].to(dev)
        s["y"] = torch.empty((B, T, H, D), device=dev)
        s["ck"] = torch.empty((B, H, C, D, D), device=dev)
        s["hT"] = torch.empty((B, H, D, D), device=dev)
        s["sa"] = torch.empty((B, T, H, D), device=dev) if saved else None
        s["ws"] = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
        s["g"] = [torch.empty((B, T, H, D), device=dev) for _ in range(6)] + [torch.empty((B, H, D, D), device=dev)]
        return s

    sets = [make_set() for _ in range(n_sets)]

    def fwd_call(s):
        ins = [s[n] for n in "rwkvab"]
        out = (s["y"], s["ck"], s["hT"]) + ((s["sa"],) if saved else ())
        wkv7.forward(*ins, s["h0"], chunk=wl.chunk, out=out, save_sa=saved,
                     workspace=s["ws"] if operators else None)

    def bwd_call(s):
        ins = [s[n] for n in "rwkvab"]
        if path == "operators":
            wkv7.backward_from_forward(*ins, s["h0"], s["ck"], s["dy"], s["dhT"], workspace=s["ws"], out=s["g"])
        else:
            wkv7.backward(*ins, s["h0"], s["ck"], s["dy"], s["dhT"], chunk=wl.chunk, sa=s["sa"],
                          workspace=s["ws"] if path != "single" else None, out=s["g"])

    def step(s, stream=None, ev=None):
        if ev is not None:
            ev[0].record(stream)
        fwd_call(s)
        if ev is not None:
            ev[1].record(stream)
        bwd_call(s)
        if ev is not None:
            ev[2].record(stream)

    step.calls = (fwd_call, bwd_call)
    return sets, step, host


def capture_graphs(torch, dev, stream, sets, *fns):
    """One CUDA graph per input set for each of `fns` (called in order on the set while warming up)."""
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for s_ in sets:
            for fn in fns:
                fn(s_)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    out = []
    for fn in fns:
        graphs = []
        for s_ in sets:
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_):
                fn(s_)
            graphs.append(g_)
        out.append(graphs)
    return out[0] if len(fns) == 1 else out


def other_configs(wkv7, torch, dev, args, peaks, hbm, sms):
    """Step time and step roofline fractions of the other training workloads (CUDA-graph replays)."""
    out = {}
    stream = torch.cuda.current_stream()
    for name, wl in gen.WORKLOADS.items():
        if wl.decode or name == args.workload or name.startswith("oracle"):
            continue
        try:
            sets, step, _ = make_runner(wkv7, torch, dev, wl, args.path, 2)
            graphs = capture_graphs(torch, dev, stream, sets, step)
            for i in range(3):
                graphs[i % 2].replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n = 10
            e0.record(stream)
            for i in range(n):
                graphs[i % 2].replay()
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / n
            fwd_b, bwd_b = byte_counts(wl, 2 if wl.dtype == "bf16" else 4)
            roof_s = max((fwd_b + bwd_b) / (hbm * 1e9), literal_flops(wl) / (fp32_peak_tflops(peaks, sms) * 1e12))
            roof_d = max((fwd_b + bwd_b) / (hbm * 1e9), derived_flops(wl) / (fp32_peak_tflops(peaks, sms) * 1e12))
            out[name] = {"B": wl.B, "T": wl.T, "H": wl.H, "ms_per_step": ms, "tokens_per_s": wl.B * wl.T / (ms / 1e3),
                         "roofline_step_frac": roof_s / (ms / 1e3), "roofline_step_derived_frac": roof_d / (ms / 1e3),
                         "launch": "CUDA graph replay (2 input sets)"}
            del sets, graphs
            torch.cuda.empty_cache()
        except Exception as e:  # reported in the line
            out[name] = {"error": f"{type(e).__name__}: {str(e)[:200]}"}
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    import linear_rnn_lm_wkv7_b300 as wkv7

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = gen.WORKLOADS[args.workload]
    if wl.decode:
        return run_decode(args, rank, world, local_rank)
    B, T, H, D = wl.B, wl.T, wl.H, wl.D
    sets, step, host = make_runner(wkv7, torch, dev, wl, args.path, N_SETS)
    stream = torch.cuda.current_stream()

    for i in range(max(3, args.warmup)):
        step(sets[i % N_SETS])
    torch.cuda.synchronize()

    dist = world > 1
    if dist:
        import torch.distributed as tdist
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    # eager calls, CUDA events around each call (the per-call split)
    with ClockSampler(uuid) as clk:
        if dist:
            tdist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(args.steps):
            step(sets[i % N_SETS], stream, evs[i])
        stop.record(stream)
        torch.cuda.synchronize()
        if dist:
            tdist.barrier()
    elapsed_ms = start.elapsed_time(stop)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
    calls_timing = "eager calls, CUDA events around each"

    # The same steps replayed from CUDA graphs (one per input set, captured once): the launches no
    # longer wait on the host.  The per-call split above stays the eager one.
    launch = "eager"
    if args.graph == "on":
        try:
            graphs = capture_graphs(torch, dev, stream, sets, step)
            for i in range(max(3, args.warmup)):
                graphs[i % N_SETS].replay()
            torch.cuda.synchronize()
            with ClockSampler(uuid) as clk:
                if dist:
                    tdist.barrier()
                torch.cuda.synchronize()
                start.record(stream)
                for i in range(args.steps):
                    graphs[i % N_SETS].replay()
                stop.record(stream)
                torch.cuda.synchronize()
                if dist:
                    tdist.barrier()
            elapsed_ms = start.elapsed_time(stop)
            launch = f"CUDA graph replay ({N_SETS} graphs, one per input set)"
            del graphs
            # the per-call split from one graph per call and input set, CUDA events between the replays
            # (the host enqueues far ahead of the device, so no launch gap falls inside a call's time)
            gf, gb = capture_graphs(torch, dev, stream, sets, *step.calls)
            for i in range(max(3, args.warmup)):
                gf[i % N_SETS].replay()
                gb[i % N_SETS].replay()
            torch.cuda.synchronize()
            for i in range(args.steps):
                evs[i][0].record(stream)
                gf[i % N_SETS].replay()
                evs[i][1].record(stream)
                gb[i % N_SETS].replay()
                evs[i][2].record(stream)
            torch.cuda.synchronize()
            fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
            bwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
            calls_timing = "CUDA graph replay per call (one graph per call and input set), CUDA events between"
            del gf, gb
        except Exception as e:  # capture refused: the eager timing stands, and the line says why
            launch = f"eager (graph capture failed: {type(e).__name__}: {str(e)[:160]})"
    clocks = clk.summary()
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    tokens_per_s = job_tokens_per_s(B * T * args.steps, world, elapsed_ms)

    # ---- end to end through the public API with host buffers (pinned), copies inside the timed region
    e2e = None
    if args.e2e_steps > 0:
        host_in, host_dy = host["in"], host["dy"]
        pin_in = {n: host_in[n].pin_memory() for n in "rwkvab"}
        pin_dy = host_dy.pin_memory()
        pin_y = torch.empty((B, T, H, D), pin_memory=True)
        pin_g = [torch.empty((B, T, H, D), pin_memory=True) for _ in range(6)] + \
                [torch.empty((B, H, D, D), pin_memory=True)]
        h2d = sum(t.numel() * t.element_size() for t in pin_in.values()) + pin_dy.numel() * 4
        d2h = pin_y.numel() * 4 + sum(t.numel() * 4 for t in pin_g)
        pin_st = {n: t.pin_memory() for n, t in (("h0", host["h0"]), ("dhT", host["dhT"])) if t is not None}
        h2d += sum(t.numel() * 4 for t in pin_st.values())

        # Pipelined across steps like an input pipeline: step i's host->device copies, compute and
        # device->host copies run on three streams, two device buffer sets alternate, so the copies of
        # step i+1 overlap the compute of step i.  Every step still copies all its inputs in and all
        # its outputs (y and the seven gradients) back.
        s_h2d, s_comp, s_d2h = (torch.cuda.Stream(dev) for _ in range(3))
        pin_out = [[pin_y, pin_g], [torch.empty_like(pin_y).pin_memory(), [torch.empty_like(g).pin_memory() for g in pin_g]]]
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]

        def e2e_step(i):
            kq = i % 2
            sb = sets[kq]
            with torch.cuda.stream(s_h2d):
                if used[kq]:
                    s_h2d.wait_event(ev_out[kq])   # step i-2 has been read back: its buffers are free
                for n in "rwkvab":
                    sb[n].copy_(pin_in[n], non_blocking=True)
                sb["dy"].copy_(pin_dy, non_blocking=True)
                for n, t in pin_st.items():
                    sb[n].copy_(t, non_blocking=True)
                ev_in[kq].record(s_h2d)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev_in[kq])
                step(sb)
                ev_done[kq].record(s_comp)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_done[kq])
                hy, hg = pin_out[kq]
                hy.copy_(sb["y"], non_blocking=True)
                for h_, d_ in zip(hg, sb["g"]):
                    h_.copy_(d_, non_blocking=True)
                ev_out[kq].record(s_d2h)
            used[kq] = True

        def run_e2e(nsteps, first):
            for i in range(nsteps):
                e2e_step(first + i)
            for st in (s_h2d, s_comp, s_d2h):
                stream.wait_stream(st)

        run_e2e(2, 0)
        torch.cuda.synchronize()
        if dist:
            tdist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for st in (s_h2d, s_comp, s_d2h):
            st.wait_event(e0)
        run_e2e(args.e2e_steps, 2)
        e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1), dev)
        e2e = {"value": job_tokens_per_s(B * T * args.e2e_steps, world, ems), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    if rank != 0:
        return

    fwd_b, bwd_b = byte_counts(wl, 2 if wl.dtype == "bf16" else 4)
    hbm, peak_kind, peaks = measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    f_ms, b_ms = statistics.mean(fwd_ms), statistics.mean(bwd_ms)
    pth = PATHS[args.path]
    bwd_call = pth.get("backward_call", "wkv7_backward")
    dom = (bwd_call, bwd_b, b_ms) if b_ms >= f_ms else ("wkv7_forward", fwd_b, f_ms)
    achieved = dom[1] / (dom[2] / 1e3) / 1e9
    step_s = elapsed_ms / 1e3 / args.steps
    fp32 = fp32_peak_tflops(peaks, sms)
    roof_s = max((fwd_b + bwd_b) / (hbm * 1e9), literal_flops(wl) / (fp32 * 1e12))
    roof_d = max((fwd_b + bwd_b) / (hbm * 1e9), derived_flops(wl) / (fp32 * 1e12))
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded, wkv7_inputs.py)",
        "config": workload_config(wl),
        "path": {"name": args.path, "forward": pth["forward"], "backward": pth["backward"], "launch": launch,
                 "parallelism": f"replicas x{world} (independent batches, no collective)"},
        "roofline": {"bound": "hbm", "kernel": f"{dom[0]} ({args.path} path: the whole call, all its kernels)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": None,
                     "traffic_note": "DRAM bytes are not measured inside the run; ncu counts per kernel are in profiles/",
                     "algorithmic_bytes": dom[1], "avg_launch_ms": dom[2]},
        "roofline_step": {"definition": "max(HBM bytes / peak BW, 8*D^2 FLOP per head-token / FP32 peak) / step time",
                          "bytes": fwd_b + bwd_b, "roofline_ms": roof_s * 1e3, "frac": roof_s / step_s,
                          "fp32_peak_tflops": fp32},
        "roofline_step_derived": {"definition": "max(HBM bytes / peak BW, 28*D^2 FLOP per head-token / FP32 peak) "
                                                "/ step time", "flops": derived_flops(wl),
                                  "roofline_ms": roof_d * 1e3, "frac": roof_d / step_s},
        "calls_ms": {"wkv7_forward": f_ms, bwd_call: b_ms, "timing": calls_timing},
        "clocks": clocks,
        "gpu_launches": launches_per_step(pth, wl, sms) * args.steps,
        "e2e": e2e,
    }
    if world == 1 and not args.no_other_configs:
        line["other_configs"] = other_configs(wkv7, torch, dev, args, peaks, hbm, sms)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def launches_per_step(pth: dict, wl, sms: int) -> int:
    """This library's kernel launches in one step of a path at a workload."""
    n = pth["launches"]
    return n(wl.B * wl.H, sms) if callable(n) else n


def fp32_peak_tflops(peaks: dict, sms: int) -> float:
    """FP32 CUDA-core peak: SMs x 128 FMA lanes x 2 FLOP x max SM clock."""
    mhz = float(peaks.get("sm_max_mhz", 2032.0)) if peaks else 2032.0
    return sms * 128 * 2 * mhz * 1e6 / 1e12


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group(backend="nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as tdist
            tdist.destroy_process_group()


if __name__ == "__main__":
    main()
