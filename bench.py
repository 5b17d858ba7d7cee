#!/usr/bin/env python3
"""Benchmark of the routed MoE FFN forward on GB300.

Default (``--impl ours``): one step = one moe_forward (route -> shuffle -> tile
map -> Gate/Up grouped GEMM with fused gather + SwiGLU -> Down grouped GEMM ->
combine) over the skewed prefill workload T=16384, E=128, top-8, H=2048,
I=768, bf16, Zipf(1.1) routing, on every rank (independent replicas, weak
scaling).  The JSON line also carries:
  roofline      the Gate/Up grouped GEMM (the dominant kernel) timed live with
                CUDA events on the launching stream over the timed region;
  e2e           the same metric through the C ABI with host buffers, the
                host->device copy of x and the scores and the device->host read
                of y of every step inside the timed region, overlapped with the
                neighbouring steps' compute on separate copy streams;
  decode        the FP8 decode sweeps (per-tensor E=192 H=4096 I=192;
                blockwise E=128 H=2048 I=768 and H=4096 I=512; B=1..8), both
                the route-direct and the grouped path at every B, us/call from
                CUDA-graph replays with L2 flushed between replays (outside the
                timed events), and the HBM roofline fraction of the AUTO path;
  fp8_prefill   the grouped path with e4m3 operands (per-tensor, blockwise)
                at the prefill shape, against the FP8 dense peak measured live;
  cpu_baseline  the CPU oracle timed on this host on a bounded token sample.

``--impl reference`` times the CPU oracle (the reference of this library) on
the same workload and metric, each step a bounded token sample.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE fwd µs/call (B=1–8) & tokens/s (T=16K); % of HBM / tensor-core roofline"
UNIT = "tokens/s"
PREFILL = "prefill"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Route-MMA latencies on H20 from "perf: add small-batch route MMA for MoE" (Performance
# tables), B = 1..8: context only (other hardware).
H20_ROUTE_MMA_US = {
    "hunyuan": [13.243, 16.833, 22.773, 30.663, 35.983, 41.554, 47.259, 54.124],
    "qwen3a": [17.349, 29.863, 40.708, 52.732, 62.510, 73.040, 84.419, 94.352],
    "qwen3b": [19.779, 37.585, 52.295, 63.833, 85.218, 98.465, 111.362, 121.922],
}


# ----------------------------------------------------------------------------- helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def rank_seed(base: int, rank: int) -> int:
    """Each replica draws its own batch: the seed of rank r is base + 7919 r."""
    return base + 7919 * rank


def reduce_max(value: float, world: int) -> float:
    """Max of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(tokens_per_rank: int, world: int, steps: int, max_ms: float) -> float:
    """Whole-job tokens/s: every rank processes tokens_per_rank per step."""
    return tokens_per_rank * world * steps / (max_ms / 1000.0)


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_digest(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


GEMM_SOURCES = ["mixture_experts_layer_index_gb300/csrc/grouped_gemm.cu",
                "mixture_experts_layer_index_gb300/csrc/common.cuh"]


def committed_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    when the summary is missing or the kernel's source changed since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        ent = d[kernel]
    except (OSError, ValueError, KeyError):
        return None
    if ent.get("source_digest") != source_digest(GEMM_SOURCES):
        return None
    return ent.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.25)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {
            "sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "power_w_max": max(pw) if pw else None,
            "reasons": sorted(reasons),
            "samples": len(sm),
        }


def gpu_id_for_smi(torch, dev_index: int) -> str:
    try:
        u = torch.cuda.get_device_properties(dev_index).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis and vis.split(",")[dev_index].strip().isdigit():
            return vis.split(",")[dev_index].strip()
        return str(dev_index)


# ----------------------------------------------------------------------------- CPU oracle legs
def oracle_tokens_per_s(inp, wl, n_tokens: int, seed: int = 0):
    """Times the CPU oracle (as it stands) on n_tokens sampled tokens; -> (tokens/s, seconds)."""
    import numpy as np
    import torch

    from oracle import moe as O

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    x, w1, w2 = bits(inp["x"]), bits(inp["w1"]), bits(inp["w2"])
    scores = inp["scores"].numpy()
    rng = np.random.default_rng(seed)
    tokens = np.sort(rng.choice(wl.T, size=min(n_tokens, wl.T), replace=False))
    t0 = time.perf_counter()
    O.forward(x, scores, w1, w2, None, None, wl.k, wl.quant, tokens=tokens)
    dt = time.perf_counter() - t0
    return len(tokens) / dt, dt


def cpu_baseline(inp, wl, budget_s: float = 15.0):
    # Two-point calibration: the oracle routes and groups the whole batch whatever
    # the sample, so its time is a fixed part plus a per-sampled-token part.
    _, t_a = oracle_tokens_per_s(inp, wl, 64, seed=1)
    _, t_b = oracle_tokens_per_s(inp, wl, 512, seed=1)
    per_tok = max((t_b - t_a) / 448.0, 1e-6)
    fixed = max(t_a - 64 * per_tok, 0.0)
    n = int(min(wl.T, max(64, (budget_s - fixed) / per_tok)))
    v, dt = oracle_tokens_per_s(inp, wl, n, seed=2)
    return {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} of the {wl.T} tokens (all {wl.k} routes each, full routing/shuffle of the batch), "
                      f"numpy fp64 oracle, {dt:.1f} s",
            "seconds": dt}


# ----------------------------------------------------------------------------- ours
def workload_config(wl, l2_note):
    return {"workload": f"{wl.name}: T={wl.T} E={wl.E} top_k={wl.k} H={wl.H} I={wl.I} bf16, "
                        "Zipf(1.1)-skewed routing with 4 empty experts",
            "T": wl.T, "E": wl.E, "top_k": wl.k, "H": wl.H, "I": wl.I, "quant": wl.quant,
            "path": "grouped", "l2": l2_note}


def graph_replay_us(m, torch, p, args, flush, reps: int, warm: int = 20):
    """Median / p10 / p90 µs of one moe_forward captured in a CUDA graph, L2
    flushed (a write of 2.5x its size) before every replay, outside the events."""
    x, sc, w1, w2, s1, s2, y, ws = args
    s = torch.cuda.Stream()
    m.moe_forward(p, x, sc, w1, w2, s1, s2, y, ws, stream=s)  # eager warm-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        m.moe_forward(p, x, sc, w1, w2, s1, s2, y, ws, stream=s)
    times = []
    with torch.cuda.stream(s):
        for i in range(reps + warm):
            flush.fill_(float(i))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            g.replay()
            b.record(s)
            b.synchronize()
            if i >= warm:
                times.append(a.elapsed_time(b) * 1000.0)
    del g
    if m.moe_read_device_status(ws) != m.MOE_OK:
        raise RuntimeError("device status not OK after decode replays")
    t = sorted(times)
    return statistics.median(t), t[len(t) // 10], t[(9 * len(t)) // 10]


CHAIN_LAYERS = 16


def chain_replay_us(m, torch, p, layers, ws, flush, reps: int, warm: int = 10):
    """Median µs per call of a chain of distinct layers captured in one CUDA
    graph: layer l reads its own weights and router scores, and its input x is
    the previous layer's y.  The weights the chain touches exceed L2 and L2 is
    flushed before every replay (outside the events); the graph's own launch is
    spread over the layers, as in a model that replays all its layers at once."""
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for (x, sc, w1, w2, s1, s2, y) in layers:  # eager warm-up of every layer
            m.moe_forward(p, x, sc, w1, w2, s1, s2, y, ws, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for (x, sc, w1, w2, s1, s2, y) in layers:
            m.moe_forward(p, x, sc, w1, w2, s1, s2, y, ws, stream=s)
    times = []
    with torch.cuda.stream(s):
        for i in range(reps + warm):
            flush.fill_(float(i))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            g.replay()
            b.record(s)
            b.synchronize()
            if i >= warm:
                times.append(a.elapsed_time(b) * 1000.0 / len(layers))
    del g
    if m.moe_read_device_status(ws) != m.MOE_OK:
        raise RuntimeError("device status not OK after chain replays")
    return statistics.median(times)


def run_decode_sweep(m, torch, dev, peaks, reps: int):
    """Both paths at every B: the route-direct path and the grouped path (the
    crossover that sets the AUTO dispatch), reported for the path AUTO takes."""
    import workloads as W

    out = {}
    flush = torch.empty(int(2.5 * 129e6) // 4, dtype=torch.float32, device=dev)
    for name in W.DECODE_SWEEPS:
        base = W.workload(name, 1)
        w1, w2, s1, s2 = W.make_weights(base, device=dev)
        # the layer chain's weights: copies of the sweep's experts at distinct addresses
        chain_w = [(w1.clone(), w2.clone(), None if s1 is None else s1.clone(), None if s2 is None else s2.clone())
                   for _ in range(CHAIN_LAYERS)]
        per_b = []
        for B in range(1, 9):
            wl = W.workload(name, B)
            x = W.make_x(wl).to(dev)
            sc = W.make_scores(wl).to(dev)
            y = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
            res = {}
            U = None
            for pname, path in (("route_direct", m.MOE_PATH_ROUTE_DIRECT), ("grouped", m.MOE_PATH_GROUPED)):
                p = m.problem(wl.T, wl.E, wl.k, wl.H, wl.I, wl.quant, path)
                ws = torch.empty(m.moe_workspace_size(p), dtype=torch.uint8, device=dev)
                res[pname] = graph_replay_us(m, torch, p, (x, sc, w1, w2, s1, s2, y, ws), flush, reps)
                if U is None:
                    v = m.moe_forward_views(p, ws)
                    off = v.ids - ws.data_ptr()
                    U = int(torch.unique(ws[off:off + wl.T * wl.k * 4].view(torch.int32)).numel())
                del ws
            auto = m.moe_select_path(m.problem(wl.T, wl.E, wl.k, wl.H, wl.I, wl.quant))
            auto_name = "route_direct" if auto == m.MOE_PATH_ROUTE_DIRECT else "grouped"
            us, p10, p90 = res[auto_name]
            w1e = 2 * wl.I * wl.H + (0 if s1 is None else s1[0].numel() * 4)
            w2e = wl.H * wl.I + (0 if s2 is None else s2[0].numel() * 4)
            algo = U * (w1e + w2e) + wl.T * wl.H * 2 * 2 + wl.T * wl.E * 4
            # the chain of CHAIN_LAYERS distinct layers on the AUTO path (own scores per layer)
            pa = m.problem(wl.T, wl.E, wl.k, wl.H, wl.I, wl.quant)
            wsa = torch.empty(m.moe_workspace_size(pa), dtype=torch.uint8, device=dev)
            ys = [torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev) for _ in range(CHAIN_LAYERS)]
            layers, chain_algo = [], 0
            for li in range(CHAIN_LAYERS):
                scl = W.make_scores(dataclasses.replace(wl, seed=wl.seed * 1000 + li))
                Ul = int(torch.unique(torch.topk(scl, wl.k, dim=1).indices).numel())
                chain_algo += Ul * (w1e + w2e) + wl.T * wl.H * 2 * 2 + wl.T * wl.E * 4
                cw = chain_w[li]
                layers.append((x if li == 0 else ys[li - 1], scl.to(dev), cw[0], cw[1], cw[2], cw[3], ys[li]))
            chain_us = chain_replay_us(m, torch, pa, layers, wsa, flush, reps)
            del wsa, ys, layers
            per_b.append({"B": B, "auto_path": auto_name, "us": round(us, 3), "p10_us": round(p10, 3),
                          "p90_us": round(p90, 3),
                          "route_direct_us": round(res["route_direct"][0], 3),
                          "grouped_us": round(res["grouped"][0], 3),
                          "distinct_experts": U, "algo_bytes": algo,
                          "hbm_gbs": round(algo / (us * 1e-6) / 1e9, 1),
                          "hbm_frac": round(algo / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                          "chain_us": round(chain_us, 3),
                          "chain_hbm_frac": round(chain_algo / CHAIN_LAYERS / (chain_us * 1e-6) / 1e9
                                                  / peaks["hbm_gbs"], 4),
                          "h20_route_mma_us": H20_ROUTE_MMA_US[name][B - 1],
                          "tokens_per_s": round(B / (us * 1e-6), 1)})
        out[name] = {"E": base.E, "H": base.H, "I": base.I, "top_k": base.k, "quant": base.quant,
                     "timing": f"CUDA-graph replay, median of {reps} after 20 warm-up replays, "
                               "L2 flushed before each replay (outside the events)",
                     "chain_timing": f"chain_us: one CUDA graph of {CHAIN_LAYERS} layers with distinct "
                                     "weights and router scores, each layer's x the previous layer's y; "
                                     "graph time / layers, L2 flushed before each replay; AUTO path",
                     "by_batch": per_b}
        del w1, w2, s1, s2, chain_w
        torch.cuda.empty_cache()
    return out


def run_world16(m, torch, dev, peaks, reps: int):
    """The 16-expert top-8 bf16 layer (T=4096, E=16, H=I=1024, uniform routing):
    whole-call µs from CUDA-graph replays with L2 flushed before each replay
    (outside the events; the 96 MB of weights would otherwise stay in L2), then
    the Gate/Up and Down GEMMs' device times from a pass with every kernel
    bracketed by CUDA events."""
    import workloads as W

    wl = W.workload("world16")
    inp = W.make_inputs(wl)
    d = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    p = m.problem(wl.T, wl.E, wl.k, wl.H, wl.I, wl.quant)
    ws = torch.empty(m.moe_workspace_size(p), dtype=torch.uint8, device=dev)
    y = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(int(2.5 * 129e6) // 4, dtype=torch.float32, device=dev)
    us, p10, p90 = graph_replay_us(m, torch, p, (d["x"], d["scores"], d["w1"], d["w2"], None, None, y, ws), flush,
                                   reps)
    m.moe_profile_start()
    for _ in range(50):
        flush.fill_(1.0)
        m.moe_forward(p, d["x"], d["scores"], d["w1"], d["w2"], None, None, y, ws)
    torch.cuda.synchronize()
    stages = m.moe_profile_stop()
    if m.moe_read_device_status(ws) != m.MOE_OK:
        raise RuntimeError("device status not OK after the world16 steps")
    R = wl.T * wl.k
    peak = peaks["bf16_tflops_sustained"]

    def tf(name, flops):
        t, n = stages.get(name, (float("nan"), 0))
        return round(flops / (t / max(n, 1) / 1000.0) / 1e12, 1) if n else None

    gu, dn = tf("gateup_gemm", 4.0 * R * wl.H * wl.I), tf("down_gemm", 2.0 * R * wl.H * wl.I)
    return {"workload": f"world16: T={wl.T} E={wl.E} top_k={wl.k} H={wl.H} I={wl.I} bf16, uniform routing",
            "us_per_call": round(us, 2), "p10_us": round(p10, 2), "p90_us": round(p90, 2),
            "tokens_per_s": round(wl.T / (us * 1e-6), 1),
            "whole_call_tflops": round(6.0 * R * wl.H * wl.I / (us * 1e-6) / 1e12, 1),
            "gateup_tflops": gu, "down_tflops": dn,
            "gateup_frac_of_bf16_sustained": round(gu / peak, 4) if gu else None,
            "down_frac_of_bf16_sustained": round(dn / peak, 4) if dn else None,
            "stages_us": {k: round(1000.0 * t / max(n, 1), 1) for k, (t, n) in stages.items()},
            "timing": f"CUDA-graph replay, median of {reps}, L2 flushed before each replay (outside the events); "
                      "GEMM TFLOP/s from a pass with an event pair around every kernel"}


_ORACLE_1T = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
import numpy as np, torch
torch.set_num_threads(1)
import workloads as W
from oracle import moe as O
from tests._util import oracle_args
out = {}
cases = [("tiny", None)] + [(n, b) for n in W.DECODE_SWEEPS for b in (1, 8)]
weights = {}
for name, B in cases:
    wl = W.workload(name, B)
    if name not in weights:  # a decode sweep shares its weights across B
        weights = {name: W.make_weights(wl if B is None else W.workload(name, 1))}
    w1, w2, s1, s2 = weights[name]
    args = oracle_args({"x": W.make_x(wl), "scores": W.make_scores(wl), "w1": w1, "w2": w2,
                        "w1_scale": s1, "w2_scale": s2})
    best = float("inf")
    for _ in range(2):
        t0 = time.perf_counter()
        O.forward(*args, wl.k, wl.quant)
        best = min(best, time.perf_counter() - t0)
    out[wl.name] = {"us_per_call": round(best * 1e6, 1), "tokens_per_s": round(wl.T / best, 2)}
print(json.dumps(out))
"""


def oracle_single_thread():
    """The CPU oracle, single-threaded (BLAS and torch limited to one thread), on
    the tiny bf16 config and the decode sweeps' B=1 and B=8 calls: µs per call,
    best of 2, with the weights' e4m3 decoding inside the timed call."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, "-c", _ORACLE_1T, ROOT], env=env, capture_output=True, text=True,
                           timeout=600)
        if r.returncode != 0:
            return {"error": r.stderr.strip().splitlines()[-1] if r.stderr.strip() else f"exit {r.returncode}"}
        res = json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.TimeoutExpired, ValueError, OSError) as exc:
        return {"error": str(exc)}
    res["note"] = ("numpy fp64 oracle with one thread (OMP/OPENBLAS/MKL_NUM_THREADS=1, torch 1 thread), "
                   "best of 2 calls; a baseline, not the target")
    return res


def gather4_ab(steps: int = 30):
    """Same-box A/B of the two ways the bf16 Gate/Up GEMM gets its expert-sorted
    activation rows at the prefill shape: the default (the scatter kernel writes
    the sorted rows, the GEMM loads plain TMA tiles) against the fused gather
    (the GEMM gathers x rows itself with TMA tile::gather4, selected by
    MOE_GATEUP_A=gather4, which the library reads once per process).  Each arm is
    a fresh process timing whole moe_forward calls (L2 flushed between calls)."""
    out = {}
    for arm, extra in (("sorted_rows", {}), ("gather4", {"MOE_GATEUP_A": "gather4"})):
        env = dict(os.environ, **extra)
        env.pop("RANK", None)
        env.pop("WORLD_SIZE", None)
        try:
            r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--case", "prefill", "--steps",
                                str(steps), "--warmup", "3"], env=env, capture_output=True, text=True, timeout=600)
            line = json.loads(r.stdout.strip().splitlines()[-1])
            out[arm] = {"us_per_call": line["us_median_eager"], "tokens_per_s": round(16384 / (line["us_median_eager"] * 1e-6), 1)}
        except (subprocess.TimeoutExpired, ValueError, IndexError, OSError, KeyError) as exc:
            out[arm] = {"error": str(exc)}
    out["note"] = ("whole forward per call, median of the eager calls with L2 flushed before each; "
                   "gather4 fuses the row gather into the GEMM's TMA loads")
    return out


def measure_fp8_peak(torch, dev, n: int = 8192):
    """Dense e4m3 GEMM throughput of the vendor library (torch._scaled_mm, bf16
    out), best of 10 x 5 back-to-back n^3 products: the FP8 roofline peak."""
    try:
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        bt = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        one = torch.ones((), device=dev)
        torch._scaled_mm(a, bt.t(), one, one, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(5):
                torch._scaled_mm(a, bt.t(), one, one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) / 5.0)
        del a, bt
        return round(2.0 * n ** 3 / (best * 1e-3) / 1e12, 1)
    except (RuntimeError, AttributeError) as exc:  # no FP8 GEMM in this torch build
        print(f"fp8 peak not measured: {exc}", file=sys.stderr)
        return None


def run_fp8_prefill(m, torch, dev, fp8_peak, bf16_sustained: float, steps: int = 50):
    """The grouped path with e4m3 operands at the prefill shape (per-tensor,
    128x128 blockwise and MXFP8 scales): per-stage device times and GEMM
    throughput."""
    import dataclasses

    import workloads as W

    out = {"fp8_peak_tflops": fp8_peak,
           "fp8_peak_source": "measured live: torch._scaled_mm e4m3 8192^3, best of 10 (burst)",
           "fp8_nominal_tflops": round(2.0 * bf16_sustained, 1),
           "fp8_nominal_source": "2 x the measured sustained bf16 peak (the dense e4m3 : bf16 rate ratio)"}
    for quant in (W.QUANT_FP8_TENSOR, W.QUANT_FP8_BLOCK, W.QUANT_MXFP8):
        wl = dataclasses.replace(W.workload(PREFILL), quant=quant, name=f"{PREFILL}_{quant}")
        w1, w2, s1, s2 = W.make_weights(wl, device=dev)  # drawn on the device (fast); seeded
        d = {"x": W.make_x(wl).to(dev), "scores": W.make_scores(wl).to(dev), "w1": w1, "w2": w2,
             "w1_scale": s1, "w2_scale": s2}
        del w1, w2, s1, s2
        p = m.problem(wl.T, wl.E, wl.k, wl.H, wl.I, wl.quant, m.MOE_PATH_GROUPED)
        opt = None
        s1, s2 = d["w1_scale"], d["w2_scale"]
        if quant == W.QUANT_MXFP8:
            # the weights' MX scales are converted to the blocked layout once, as at load time
            s1 = torch.empty(m.moe_mx_weight_scales_bytes(wl.E, wl.H, wl.I, 1), dtype=torch.uint8, device=dev)
            s2 = torch.empty(m.moe_mx_weight_scales_bytes(wl.E, wl.H, wl.I, 2), dtype=torch.uint8, device=dev)
            m.moe_mx_weight_scales(d["w1_scale"], d["w2_scale"], wl.E, wl.H, wl.I, s1, s2)
            opt = m.forward_options(mx_weight_scales_blocked=True)
        ws = torch.empty(m.moe_workspace_size_ex(p, opt), dtype=torch.uint8, device=dev)
        y = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
        args = (p, opt, d["x"], d["scores"], d["w1"], d["w2"], s1, s2, y, ws)
        for _ in range(5):
            m.moe_forward_ex(*args)
        torch.cuda.synchronize()
        # step time without per-kernel events, then the stages from a profiled pass
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            m.moe_forward_ex(*args)
        e1.record()
        torch.cuda.synchronize()
        step_us = e0.elapsed_time(e1) / steps * 1000.0
        m.moe_profile_start()
        for _ in range(steps):
            m.moe_forward_ex(*args)
        torch.cuda.synchronize()
        stages = m.moe_profile_stop()
        if m.moe_read_device_status(ws) != m.MOE_OK:
            raise RuntimeError("device status not OK after the FP8 prefill steps")
        R = wl.T * wl.k

        def tflops(name, flops):
            t, n = stages.get(name, (float("nan"), 0))
            return round(flops / (t / max(n, 1) / 1000.0) / 1e12, 1) if n else None

        gu = tflops("gateup_gemm", 4.0 * R * wl.H * wl.I)
        dn = tflops("down_gemm", 2.0 * R * wl.H * wl.I)
        nominal = 2.0 * bf16_sustained
        out[quant] = {
            "tokens_per_s": round(wl.T / (step_us * 1e-6), 1), "us_per_step": round(step_us, 1), "steps": steps,
            "gateup_tflops": gu, "down_tflops": dn,
            "gateup_frac_of_fp8_peak": round(gu / fp8_peak, 4) if gu and fp8_peak else None,
            "down_frac_of_fp8_peak": round(dn / fp8_peak, 4) if dn and fp8_peak else None,
            "gateup_frac_of_2x_bf16_sustained": round(gu / nominal, 4) if gu else None,
            "down_frac_of_2x_bf16_sustained": round(dn / nominal, 4) if dn else None,
            "stages_us": {k: round(1000.0 * t / max(n, 1), 1) for k, (t, n) in stages.items()},
        }
        del d, ws, y
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    import __graft_entry__

    __graft_entry__.build()
    import mixture_experts_layer_index_gb300 as m
    import workloads as W

    peaks, peak_src = load_peaks()
    base = W.workload(PREFILL)
    import dataclasses

    wl = dataclasses.replace(base, seed=rank_seed(base.seed, rank))
    if args.tokens:
        wl = dataclasses.replace(wl, T=args.tokens, name=f"{wl.name}_T{args.tokens}")
    inp = W.make_inputs(wl)
    d = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    p = m.problem(wl.T, wl.E, wl.k, wl.H, wl.I, wl.quant)
    ws = torch.empty(m.moe_workspace_size(p), dtype=torch.uint8, device=dev)
    y = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        m.moe_forward(p, d["x"], d["scores"], d["w1"], d["w2"], None, None, y, ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if m.moe_read_device_status(ws) != m.MOE_OK:
        raise RuntimeError("device status not OK after warm-up")

    sampler = ClockSampler(gpu_id_for_smi(torch, local))
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # the timed region: K whole steps and nothing else (no per-kernel events)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall = time.perf_counter()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall_s = time.perf_counter() - t_wall
    ms = ev0.elapsed_time(ev1)
    max_ms = reduce_max(ms, world)
    value = throughput(wl.T, world, args.steps, max_ms)
    # roofline of the dominant kernel: a second pass of the same steps in which only
    # the Gate/Up GEMM is bracketed by an event pair on the launching stream
    m.moe_profile_start_stage("gateup_gemm")
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    timed_stages = m.moe_profile_stop()
    clocks = sampler.stop()

    # per-stage breakdown: a second pass of the same steps with every kernel bracketed
    m.moe_profile_start()
    eb0, eb1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    eb0.record(stream)
    for _ in range(args.steps):
        step()
    eb1.record(stream)
    torch.cuda.synchronize()
    stages = m.moe_profile_stop()
    profiled_step_ms = eb0.elapsed_time(eb1) / args.steps

    # dominant kernel: the Gate/Up grouped GEMM, 2 * R * H * 2I algorithmic FLOPs per launch
    R = wl.T * wl.k
    gu_ms, gu_n = timed_stages.get("gateup_gemm", (float("nan"), 0))
    dn_ms, dn_n = stages.get("down_gemm", (float("nan"), 0))
    gu_flops = 4.0 * R * wl.H * wl.I
    dn_flops = 2.0 * R * wl.H * wl.I
    gu_avg_s = gu_ms / max(gu_n, 1) / 1000.0
    achieved = gu_flops / gu_avg_s / 1e12
    peak = peaks["bf16_tflops_sustained"]
    # our kernel launches in the timed region: the breakdown pass ran the same steps
    launches = sum(n for name, (_, n) in stages.items() if name != "header_reset")

    # e2e: host buffers, every copy inside the timed region, pipelined as a serving
    # loop would run it: step i+1's inputs go up on an upload stream while step i
    # computes, step i's y comes down on a download stream after it; inputs and y
    # are double-buffered on the device.
    xh = inp["x"].pin_memory()
    sh = inp["scores"].pin_memory()
    yh = [torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xd = [d["x"], torch.empty_like(d["x"])]
    sd = [d["scores"], torch.empty_like(d["scores"])]
    yd = [y, torch.empty_like(y)]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n):
        with torch.cuda.stream(up):
            xd[0].copy_(xh, non_blocking=True)
            sd[0].copy_(sh, non_blocking=True)
            ev_in[0].record(up)
        for i in range(n):
            b = i & 1
            if i + 1 < n:  # upload the next step's inputs while this one computes
                with torch.cuda.stream(up):
                    if i >= 1:
                        up.wait_event(ev_comp[1 - b])  # step i-1 has finished reading buffer 1-b
                    xd[1 - b].copy_(xh, non_blocking=True)
                    sd[1 - b].copy_(sh, non_blocking=True)
                    ev_in[1 - b].record(up)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # y[b] of step i-2 is on the host
            m.moe_forward(p, xd[b], sd[b], d["w1"], d["w2"], None, None, yd[b], ws, stream=stream)
            ev_comp[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev_comp[b])
                yh[b].copy_(yd[b], non_blocking=True)
                ev_out[b].record(down)
        stream.wait_stream(down)

    e2e_run(2)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    if m.moe_read_device_status(ws) != m.MOE_OK:
        raise RuntimeError("device status not OK after the e2e steps")
    e2e_ms = reduce_max(e0.elapsed_time(e1), world)
    e2e = {"value": throughput(wl.T, world, args.steps, e2e_ms), "unit": UNIT,
           "h2d_bytes_per_step": xh.numel() * 2 + sh.numel() * 4, "d2h_bytes_per_step": yh[0].numel() * 2,
           "schedule": "copies of step i+1 / i overlapped with step i's compute (separate upload and "
                       "download streams, double-buffered device inputs and outputs); all copies inside "
                       "the timed region"}

    decode = fp8 = w16 = None
    if not args.no_world16 and rank == 0:
        w16 = run_world16(m, torch, dev, peaks, args.decode_reps)
    if not args.no_decode and rank == 0:
        decode = run_decode_sweep(m, torch, dev, peaks, args.decode_reps)
    if not args.no_fp8 and rank == 0:
        fp8 = run_fp8_prefill(m, torch, dev, measure_fp8_peak(torch, dev), peaks["bf16_tflops_sustained"])

    gather_ab = None
    if not args.no_gather_ab and rank == 0 and world == 1:
        gather_ab = gather4_ab()

    cpu = cpu_1t = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp, wl, args.cpu_budget)
        if w16 is not None:
            import workloads as W

            w16wl = W.workload("world16")
            w16["cpu_baseline"] = cpu_baseline(W.make_inputs(w16wl), w16wl, args.cpu_budget / 2)
        cpu_1t = oracle_single_thread()

    if rank != 0:
        return
    per_step_ms = max_ms / args.steps
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(per_step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; random-init weights, N(0,1/fan_in))",
        "config": workload_config(wl, "inputs larger than L2: 1.2 GB of expert weights + 67 MB of x per step"),
        "roofline": {
            "kernel": "gateup_gemm (tcgen05 Gate/Up grouped GEMM, fused TMA gather + SwiGLU)",
            "bound": "tensor",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_source": f"{peak_src} bf16_tflops_sustained (burst {peaks['bf16_tflops']})",
            "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4),
            "traffic": committed_traffic("gateup_gemm"),
            "algorithmic_flops_per_launch": gu_flops,
            "avg_launch_ms": round(gu_avg_s * 1000.0, 5),
        },
        "kernels": {name: {"total_ms": round(t, 3), "launches": n, "avg_us": round(1000.0 * t / max(n, 1), 2),
                           "share": round(t / max(sum(v[0] for v in stages.values()), 1e-9), 4)}
                    for name, (t, n) in stages.items()},
        "kernels_note": ("per-stage CUDA-event times from a third pass of the same steps with every kernel "
                         f"bracketed ({round(profiled_step_ms, 4)} ms/step with those events); the timed region "
                         "has no per-kernel events; roofline.avg_launch_ms comes from a second pass that "
                         "brackets only gateup_gemm"),
        "down_gemm_tflops": round(dn_flops / (dn_ms / max(dn_n, 1) / 1000.0) / 1e12, 1) if dn_n else None,
        "whole_step_tflops": round(6.0 * R * wl.H * wl.I / (per_step_ms / 1000.0) / 1e12, 1),
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_s_timed": round(wall_s, 3),
        "gather_ab": gather_ab,
        "world16": w16,
        "decode": decode,
        "fp8_prefill": fp8,
        "cpu_baseline": cpu,
        "cpu_oracle_single_thread": cpu_1t,
    }
    print(json.dumps(line))


# ----------------------------------------------------------------------------- single case (profiling)
def run_case(args):
    """One workload only, `--warmup` untimed then `--steps` timed calls, for
    profiler captures: prefill | prefill_fp8_tensor | prefill_fp8_block (T from
    --tokens, default 16384) or <decode sweep>:<B> (e.g. hunyuan:8).  Prints one
    short JSON line (not a bench line)."""
    import dataclasses

    import torch

    dev = torch.device("cuda", 0)
    import __graft_entry__

    __graft_entry__.build()
    import mixture_experts_layer_index_gb300 as m
    import workloads as W

    name = args.case
    if ":" in name:
        sweep, B = name.split(":")
        wl = W.workload(sweep, int(B))
        w1, w2, s1, s2 = W.make_weights(W.workload(sweep, 1), device=dev)
    else:
        quant = {"prefill": W.QUANT_BF16, "prefill_fp8_tensor": W.QUANT_FP8_TENSOR,
                 "prefill_fp8_block": W.QUANT_FP8_BLOCK, "prefill_mxfp8": W.QUANT_MXFP8}[name]
        wl = dataclasses.replace(W.workload(PREFILL), quant=quant, T=args.tokens or W.workload(PREFILL).T)
        w1, w2, s1, s2 = W.make_weights(wl, device=dev)
    x, sc = W.make_x(wl).to(dev), W.make_scores(wl).to(dev)
    p = m.problem(wl.T, wl.E, wl.k, wl.H, wl.I, wl.quant)
    ws = torch.empty(m.moe_workspace_size(p), dtype=torch.uint8, device=dev)
    y = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(int(2.5 * 129e6) // 4, dtype=torch.float32, device=dev)
    for i in range(args.warmup):
        m.moe_forward(p, x, sc, w1, w2, s1, s2, y, ws)
    torch.cuda.synchronize()
    times = []
    for i in range(args.steps):
        flush.fill_(float(i))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        m.moe_forward(p, x, sc, w1, w2, s1, s2, y, ws)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1000.0)
    if m.moe_read_device_status(ws) != m.MOE_OK:
        raise RuntimeError("device status not OK")
    path = "route_direct" if m.moe_select_path(p) == m.MOE_PATH_ROUTE_DIRECT else "grouped"
    print(json.dumps({"case": name, "T": wl.T, "quant": wl.quant, "path": path,
                      "us_median_eager": round(statistics.median(times), 2), "steps": args.steps}))


# ----------------------------------------------------------------------------- reference (oracle) arm
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import workloads as W

    wl = W.workload(PREFILL)
    inp = W.make_inputs(wl)
    # calibrate a per-step token sample so that warm-up + steps take about two minutes
    _, t64 = oracle_tokens_per_s(inp, wl, 64, seed=0)
    per_step_s = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(wl.T, 64 * per_step_s / max(t64, 1e-6))))
    for i in range(args.warmup):
        oracle_tokens_per_s(inp, wl, n, seed=100 + i)
    total_s = 0.0
    for i in range(args.steps):
        _, dt = oracle_tokens_per_s(inp, wl, n, seed=1000 + i)
        total_s += dt
    value = n * args.steps / total_s
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1000.0 * total_s / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded; random-init weights, N(0,1/fan_in))",
        "config": workload_config(wl, "CPU run"),
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"{n} sampled tokens of the T={wl.T} batch per step (all routes each, "
                                   "full routing/shuffle), numpy fp64 oracle"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-decode", action="store_true", help="skip the route-direct decode sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8 grouped prefill leg")
    ap.add_argument("--no-world16", action="store_true", help="skip the 16-expert top-8 bf16 layer")
    ap.add_argument("--no-gather-ab", action="store_true", help="skip the gather4 A/B of the Gate/Up operand")
    ap.add_argument("--decode-reps", type=int, default=200)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override T of the prefill workload (smaller cases for profiling; not a bench line)")
    ap.add_argument("--case", default="",
                    help="run one workload only, for profiler captures: prefill, prefill_fp8_tensor, "
                         "prefill_fp8_block, prefill_mxfp8 (T from --tokens) or <decode sweep>:<B>; not a bench line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
