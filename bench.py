#!/usr/bin/env python3
"""Benchmark of the W4A16 decode step on GB300.

One step = the 112 INT4 weight-only projections of a 28-layer Qwen2.5-7B
decode step at M = 1 (per layer: qkv 4608x3584, o 3584x3584, gate_up
37888x3584, down 3584x18944), replayed as one captured CUDA graph through the
C ABI (w4_decode_seq_replay).  Weights (3.36 GB of packed INT4 + FP16 scales,
far larger than the 129 MB L2) and activations are seeded synthetic data.

Prints ONE JSON line (rank 0).  `value` is weight+scale bytes per step over
the step time, in GB/s, summed over ranks (replicas: each rank runs its own
step on its own GPU; there is no exchange).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A16 GEMV achieved HBM GB/s (% of GB300 peak); µs per 28-layer M=1 projection step"
LAYER = [("qkv", 4608, 3584), ("o", 3584, 3584), ("gate_up", 37888, 3584), ("down", 3584, 18944)]
LAYERS = 28
CONFIG_ID = 3  # seed family of the full-decode-step workload
BYTES_PER_STEP = LAYERS * sum((N * K) // 2 + N * (K // 128) * 2 for _, N, K in LAYER)  # 3,364,601,856
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = ("decode step: 28 layers x {qkv 4608x3584, o 3584x3584, gate_up 37888x3584, down 3584x18944} "
            "W4A16 projections, M=1, one CUDA-graph replay per step")


def rank_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(torch, value: float, world: int, device: str = "cuda") -> float:
    """The largest of the ranks' values (each rank passes its own): the
    slowest replica's time is the job's time.  One rank: the value itself."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every replica streams BYTES_PER_STEP per step,
    and the job's step time is the slowest rank's."""
    return world * BYTES_PER_STEP / (ms_per_step * 1e-3) / 1e9


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---- clocks --------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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
        rows = []
        for line in out.splitlines():
            f = [t.strip() for t in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append({"sm": float(f[1]), "max": float(f[2]), "power": float(f[3]),
                             "hw": f[5] == "Active", "hw_th": f[6] == "Active", "sw_th": f[7] == "Active",
                             "pcap": f[8] == "Active"})
            except ValueError:
                continue
        if not rows:
            return None
        load = [r for r in rows if r["power"] > 250] or rows
        reasons = sorted({name for r in load for name, key in
                          (("hw_slowdown", "hw"), ("hw_thermal_slowdown", "hw_th"),
                           ("sw_thermal_slowdown", "sw_th"), ("sw_power_cap", "pcap")) if r[key]})
        return {"sm_mhz": statistics.median(r["sm"] for r in load), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(load),
                "power_w_max": max(r["power"] for r in rows)}


# ---- workload -----------------------------------------------------------------
def build_step(torch, w4, synth, M: int, layers: int = LAYERS):
    """Packed weights of `layers` layers (device-generated, device-packed), x
    and y arenas, and the captured sequence."""
    dev = torch.device("cuda")
    ws, keep, meta = [], [], []
    x_host_parts, xsz, ysz = [], [], []
    for layer in range(layers):
        for pid, (_, N, K) in enumerate(LAYER):
            G = K // 128
            q = torch.empty((N, K), dtype=torch.int8, device=dev)
            s = torch.empty((N, G), dtype=torch.int16, device=dev)
            synth.q_device(synth.seed_of(CONFIG_ID, layer, pid, synth.T_Q), N, K, q)
            synth.scale_device(synth.seed_of(CONFIG_ID, layer, pid, synth.T_SCALE), N, G, s)
            packed = torch.empty(w4.w4_packed_bytes(N, K), dtype=torch.uint8, device=dev)
            ws.append(w4.w4_pack(q, s, N, K, packed))
            keep.append(packed)
            del q, s
            x_host_parts.append(synth.x_full(synth.seed_of(CONFIG_ID, layer, pid, synth.T_X), M, K).ravel())
            xsz.append(M * K)
            ysz.append(M * N)
            meta.append((layer, pid, N, K))
    x_host = np.concatenate(x_host_parts).view(np.int16)
    x_arena = torch.from_numpy(x_host).to(dev)
    y_arena = torch.zeros(sum(ysz), dtype=torch.int16, device=dev)
    xs, ys, xo, yo = [], [], 0, 0
    for nx, ny in zip(xsz, ysz):
        xs.append(x_arena[xo:xo + nx])
        ys.append(y_arena[yo:yo + ny])
        xo += nx
        yo += ny
    return dict(ws=ws, keep=keep, meta=meta, x_host=x_host, x_arena=x_arena, y_arena=y_arena, xs=xs, ys=ys)


def time_replays(torch, fn, reps: int) -> float:
    """Average ms per call of fn() over reps calls, CUDA events on the current stream."""
    s = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(s)
    for _ in range(reps):
        fn()
    b.record(s)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def replay_spread(torch, fn, reps: int = 100) -> dict:
    """Per-call device times of `reps` back-to-back calls of fn(): one CUDA
    event between consecutive calls on the current stream, so each interval
    is one call as the stream saw it (the gap to the next launch included).
    Median and the 10th and 90th percentiles, in microseconds."""
    s = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    torch.cuda.synchronize()
    ev[0].record(s)
    for k in range(reps):
        fn()
        ev[k + 1].record(s)
    torch.cuda.synchronize()
    us = np.array([ev[k].elapsed_time(ev[k + 1]) * 1e3 for k in range(reps)])
    return {"reps": reps, "median_us": float(np.median(us)), "p10_us": float(np.percentile(us, 10)),
            "p90_us": float(np.percentile(us, 90)), "min_us": float(us.min()), "max_us": float(us.max())}


def code_only(src: str) -> str:
    """C/C++ source without its comments, blank space collapsed (string and
    character literals kept as written)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_digest() -> str:
    """The step kernel's sources, comments and blank space removed (so the ncu
    figures taken on the same code stay valid across comment edits)."""
    h = hashlib.sha256()
    for name in ("step.cu", "step_launch.h", "decode_common.cuh", "w4_internal.cuh", "w4_device.cuh", "tc_ptx.cuh"):
        with open(os.path.join(ROOT, "int4_weight_only_pack_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic_per_launch():
    """DRAM bytes per launch of the decode kernel from the committed ncu
    summary, if it was taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "decode_step_M1_traffic.txt")
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m = re.search(r"kernel_source_digest:\s*(\w+)", text)
    t = re.search(r"dram_bytes_per_launch:\s*([0-9.]+)", text)
    if not m or not t or m.group(1) != kernel_source_digest():
        return None
    return float(t.group(1))


# ---- CPU oracle (the reported baseline and the reference arm) --------------------
def oracle_sample(synth, rows_stride: int = 16):
    """A bounded sample of the step: layer 0's four projections at M = 1,
    every `rows_stride`-th output row.  Inputs drawn on the host."""
    probs, nbytes = [], 0
    for pid, (_, N, K) in enumerate(LAYER):
        rows = np.arange(0, N, rows_stride)
        q, s, x = synth.projection_inputs(CONFIG_ID, 0, pid, 1, N, K, rows=rows)
        probs.append((x, q, s))
        nbytes += len(rows) * ((K // 2) + (K // 128) * 2)
    return probs, nbytes


def oracle_step(oracle, probs, threads):
    for x, q, s in probs:
        oracle.linear(x, q, s, threads=threads)


def run_reference(args):
    rank, world, _ = rank_info()
    if rank != 0:
        return 0
    import oracle
    import synth
    cores = host_cores()
    probs, nbytes = oracle_sample(synth)
    for _ in range(args.warmup):
        oracle_step(oracle, probs, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(oracle, probs, cores)
    dt = (time.perf_counter() - t0) / args.steps
    value = nbytes / dt / 1e9
    sample = ("layer 0 of the step, all four projections at M=1, every 16th output row "
              "(%d weight+scale bytes per step)" % nbytes)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": 1, "sample": sample},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "host": {"arch": platform.machine(), "nproc": os.cpu_count()}}
    print(json.dumps(line), flush=True)
    return 0


def cpu_single_gemv_one_thread(oracle, synth, budget_s: float = 4.0):
    """The oracle on one host thread over the single-GEMV workload (qkv
    4608x3584, M = 1), every 16th output row: GB/s of weight bytes."""
    _, N, K = LAYER[0]
    rows = np.arange(0, N, 16)
    q, s, x = synth.projection_inputs(CONFIG_ID, 0, 0, 1, N, K, rows=rows)
    nbytes = len(rows) * ((K // 2) + (K // 128) * 2)
    oracle.linear(x, q, s, threads=1)
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.linear(x, q, s, threads=1)
        n += 1
        if time.perf_counter() - t0 > budget_s or n >= 200:
            break
    dt = (time.perf_counter() - t0) / n
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "qkv 4608x3584 at M=1, every 16th output row (%d weight+scale bytes), %d passes, one thread"
                      % (nbytes, n)}


def cpu_baseline(oracle, synth, budget_s: float = 12.0):
    cores = host_cores()
    probs, nbytes = oracle_sample(synth)
    oracle_step(oracle, probs, cores)  # warm
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_step(oracle, probs, cores)
        n += 1
        if time.perf_counter() - t0 > budget_s or n >= 50:
            break
    dt = (time.perf_counter() - t0) / n
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "layer 0 of the step, four projections at M=1, every 16th output row, %d passes "
                      "(%d weight+scale bytes each), FP64 C oracle over %d threads" % (n, nbytes, cores)}


def run_one_projection(args):
    """One projection of layer 0 at M = --profile-m tokens (1 by default),
    launched --warmup + --steps times back to back: a profiler target.  M <= 16
    runs the decode kernel (weights larger than L2 only for gate_up and down,
    so the printed rate of the others is L2-assisted); larger M runs the
    prefill GEMM with its workspace."""
    import torch
    import int4_weight_only_pack_gb300 as w4
    from int4_weight_only_pack_gb300 import build as w4build
    import synth
    w4build.build()
    synth.build_device()
    pid = [n for n, _, _ in LAYER].index(args.profile_projection)
    _, N, K = LAYER[pid]
    G = K // 128
    q = torch.empty((N, K), dtype=torch.int8, device="cuda")
    s = torch.empty((N, G), dtype=torch.int16, device="cuda")
    synth.q_device(synth.seed_of(CONFIG_ID, 0, pid, synth.T_Q), N, K, q)
    synth.scale_device(synth.seed_of(CONFIG_ID, 0, pid, synth.T_SCALE), N, G, s)
    packed = torch.empty(w4.w4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    w = w4.w4_pack(q, s, N, K, packed)
    del q, s
    M = max(1, args.profile_m)
    x = torch.from_numpy(synth.x_full(synth.seed_of(CONFIG_ID, 0, pid, synth.T_X), M, K).view(np.int16)).cuda()
    y = torch.zeros((M, N), dtype=torch.int16, device="cuda")
    if M <= 16:
        def run():
            w4.w4a16_gemv(x, w, y, M)
    else:
        nbw = w4.w4_workspace_bytes(M, N, K)
        wsb = torch.zeros(max(nbw, 256), dtype=torch.uint8, device="cuda")

        def run():
            w4.w4a16_gemm(x, w, y, M, wsb, nbw)
    for _ in range(args.warmup):
        run()
    ms = time_replays(torch, run, args.steps)
    nb = w4.w4_packed_bytes(N, K)
    line = {"projection": args.profile_projection, "M": M, "N": N, "K": K, "launches": args.steps,
            "us_per_launch": ms * 1e3, "GB/s": nb / (ms * 1e-3) / 1e9}
    if M > 16:
        line["TFLOP/s"] = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        line["status_word"] = int(wsb[:4].view(torch.int32).item())
    print(json.dumps(line), flush=True)
    return 0


def single_gemv_rotated(torch, w4, synth, st, copies=32, reps=20):
    """The single-GEMV workload (qkv 4608x3584, M = 1) through w4a16_gemv over
    `copies` distinct packed weights launched in turn (32 x 8.5 MB = 272 MB,
    over twice the 129 MB L2, so every launch reads its weight from DRAM):
    us per GEMV and weight GB/s, with the spread of the per-launch times."""
    dev = torch.device("cuda")
    pid = 0
    _, N, K = LAYER[pid]
    G = K // 128
    idx = [i for i, m in enumerate(st["meta"]) if m[1] == pid]
    ws = [st["ws"][i] for i in idx]
    keep = []
    layer = LAYERS
    while len(ws) < copies:  # more seeded qkv weights beyond the step's 28 layers
        q = torch.empty((N, K), dtype=torch.int8, device=dev)
        s = torch.empty((N, G), dtype=torch.int16, device=dev)
        synth.q_device(synth.seed_of(CONFIG_ID, layer, pid, synth.T_Q), N, K, q)
        synth.scale_device(synth.seed_of(CONFIG_ID, layer, pid, synth.T_SCALE), N, G, s)
        packed = torch.empty(w4.w4_packed_bytes(N, K), dtype=torch.uint8, device=dev)
        ws.append(w4.w4_pack(q, s, N, K, packed))
        keep.append(packed)
        layer += 1
    x = st["xs"][idx[0]]
    y = torch.zeros((1, N), dtype=torch.int16, device=dev)
    k = [0]

    def one():
        w4.w4a16_gemv(x, ws[k[0] % copies], y, 1)
        k[0] += 1

    for _ in range(2 * copies):
        one()
    spread = replay_spread(torch, one, reps * copies)
    nb = (N * K) // 2 + N * G * 2
    # the same launches captured in one graph (the host's call overhead out of the way): per launch, with
    # and without programmatic dependent launch between consecutive ones
    graph = {}
    for pdl in (False, True):
        g = w4.DecodeSeq(ws[:copies], [x] * copies, [y] * copies, 1, use_pdl=pdl)
        for _ in range(3):
            g.replay()
        us = time_replays(torch, g.replay, reps) * 1e3 / copies
        graph["pdl" if pdl else "no_pdl"] = {"us_per_gemv": us, "GB/s": nb / (us * 1e-6) / 1e9}
        g.close()
    return {"copies": copies, "bytes_per_copy": nb, "rotated_bytes": nb * copies,
            "us_per_gemv": spread["median_us"], "GB/s": nb / (spread["median_us"] * 1e-6) / 1e9,
            "spread": spread, "launch": "w4a16_gemv (decode kernel, library launch shape) called from Python "
                                        "once per launch, one stream, back to back (host call overhead included)",
            "graph_of_rotated_launches": graph}


def small_batch_sweep(torch, w4, synth, st, Ms=(2, 4, 8, 16), reps=50):
    """The full 112-projection step at M tokens (same weights): us/step and
    weight GB/s; weight bytes are read once per step whatever M."""
    out = {}
    for M in Ms:
        xs, ys, keep = [], [], []
        for (layer, pid, N, K) in st["meta"]:
            x = torch.from_numpy(synth.x_full(synth.seed_of(CONFIG_ID, layer, pid, synth.T_X), M, K)
                                 .view(np.int16)).cuda()
            y = torch.zeros((M, N), dtype=torch.int16, device="cuda")
            xs.append(x)
            ys.append(y)
        peak = measured_peaks()[0].get("hbm_gbs", FALLBACK_HBM_GBS)
        entry = {}
        nbw = w4.w4_decode_seq_workspace_bytes(st["ws"], M)
        buf = torch.zeros(nbw + 256, dtype=torch.uint8, device="cuda")
        off = (-buf.data_ptr()) % 256
        for mode, seq in (("persistent", w4.DecodeSeq(st["ws"], xs, ys, M, workspace=buf[off:off + nbw])),
                          ("graph_pdl", w4.DecodeSeq(st["ws"], xs, ys, M, use_pdl=True))):
            for _ in range(3):
                seq.replay()
            ms = time_replays(torch, seq.replay, reps)
            entry[mode] = {"us_per_step": ms * 1e3, "GB/s": BYTES_PER_STEP / (ms * 1e-3) / 1e9,
                           "frac_of_hbm": BYTES_PER_STEP / (ms * 1e-3) / 1e9 / peak,
                           "spread": replay_spread(torch, seq.replay, reps)}
            if mode == "persistent":
                entry[mode]["status_word"] = seq.status()
            seq.close()
        out["M%d" % M] = entry
        del xs, ys, buf
    return out


def prefill_layer(torch, w4, synth, st, M=512, layers=4, reps=5):
    """Prefill-shaped projections (M = 512) of the first layers' weights:
    us per projection and TFLOP/s (2*M*N*K useful flops)."""
    peaks, _ = measured_peaks()
    peak = float(peaks.get("bf16_tflops", 1899.7))
    out = {}
    for pid, (name, N, K) in enumerate(LAYER):
        x = torch.from_numpy(synth.x_full(synth.seed_of(5, 0, pid, synth.T_X), M, K).view(np.int16)).cuda()
        y = torch.zeros((M, N), dtype=torch.int16, device="cuda")
        nb = w4.w4_workspace_bytes(M, N, K)
        wsb = torch.zeros(max(nb, 256), dtype=torch.uint8, device="cuda")
        idx = [i for i, m in enumerate(st["meta"]) if m[1] == pid][:layers]

        def run():
            for i in idx:
                w4.w4a16_gemm(x, st["ws"][i], y, M, wsb, nb)
        run()
        ms = time_replays(torch, run, reps) / len(idx)
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        k = [0]

        def one():
            w4.w4a16_gemm(x, st["ws"][idx[k[0] % len(idx)]], y, M, wsb, nb)
            k[0] += 1
        out[name] = {"us": ms * 1e3, "TFLOP/s": tf, "frac_of_dense_peak": tf / peak,
                     "spread": replay_spread(torch, one, 50),
                     "status_word": int(wsb[:4].view(torch.int32).item())}
    tot_us = sum(v["us"] for v in out.values())
    out["layer"] = {"us": tot_us, "TFLOP/s": 2.0 * M * sum(N * K for _, N, K in LAYER) / (tot_us * 1e-6) / 1e12,
                    "peak_TFLOP/s": peak, "peak_source": "bf16_tflops of MEASURED_PEAKS.json (f16 runs at the "
                                                         "bf16 tensor rate)"}
    return out


def bf16_step(torch, w4, synth, st, reps=100):
    """The same 28-layer step with bfloat16 activations (same weights, x drawn
    from the same seeds and rounded to bfloat16): us/step and weight GB/s."""
    xs, ys = [], []
    for (layer, pid, N, K) in st["meta"]:
        xb = synth.x_full_bf16(synth.seed_of(CONFIG_ID, layer, pid, synth.T_X), 1, K)
        xs.append(torch.from_numpy(xb.view(np.int16)).cuda())
        ys.append(torch.zeros((1, N), dtype=torch.int16, device="cuda"))
    nbw = w4.w4_decode_seq_workspace_bytes(st["ws"], 1)
    buf = torch.zeros(nbw + 256, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 256
    seq = w4.DecodeSeq(st["ws"], xs, ys, 1, workspace=buf[off:off + nbw], act="bf16")
    for _ in range(5):
        seq.replay()
    ms = time_replays(torch, seq.replay, reps)
    peak = measured_peaks()[0].get("hbm_gbs", FALLBACK_HBM_GBS)
    out = {"us_per_step": ms * 1e3, "GB/s": BYTES_PER_STEP / (ms * 1e-3) / 1e9,
           "frac_of_hbm": BYTES_PER_STEP / (ms * 1e-3) / 1e9 / peak, "status_word": seq.status()}
    seq.close()
    return out


def swiglu_step(torch, w4, synth, st, reps=100):
    """The 28-layer step with every gate_up projection fused with its SwiGLU
    (weights packed by w4_pack_glu from the same seeded q and scales, y =
    silu(gate) * up of 18944 columns): us/step and weight GB/s."""
    dev = torch.device("cuda")
    ws, keep, ys, flags = [], [], [], []
    for i, (layer, pid, N, K) in enumerate(st["meta"]):
        if LAYER[pid][0] == "gate_up":
            G = K // 128
            q = torch.empty((N, K), dtype=torch.int8, device=dev)
            s = torch.empty((N, G), dtype=torch.int16, device=dev)
            synth.q_device(synth.seed_of(CONFIG_ID, layer, pid, synth.T_Q), N, K, q)
            synth.scale_device(synth.seed_of(CONFIG_ID, layer, pid, synth.T_SCALE), N, G, s)
            packed = torch.empty(w4.w4_packed_bytes(N, K), dtype=torch.uint8, device=dev)
            ws.append(w4.w4_pack_glu(q, s, N // 2, K, packed))
            keep.append(packed)
            del q, s
            ys.append(torch.zeros((1, N // 2), dtype=torch.int16, device=dev))
            flags.append(w4.W4_OP_SWIGLU)
        else:
            ws.append(st["ws"][i])
            ys.append(torch.zeros((1, N), dtype=torch.int16, device=dev))
            flags.append(0)
    nbw = w4.w4_decode_seq_workspace_bytes(ws, 1)
    buf = torch.zeros(nbw + 256, dtype=torch.uint8, device=dev)
    off = (-buf.data_ptr()) % 256
    seq = w4.DecodeSeq(ws, st["xs"], ys, 1, workspace=buf[off:off + nbw], op_flags=flags)
    for _ in range(5):
        seq.replay()
    ms = time_replays(torch, seq.replay, reps)
    peak = measured_peaks()[0].get("hbm_gbs", FALLBACK_HBM_GBS)
    out = {"us_per_step": ms * 1e3, "GB/s": BYTES_PER_STEP / (ms * 1e-3) / 1e9,
           "frac_of_hbm": BYTES_PER_STEP / (ms * 1e-3) / 1e9 / peak, "status_word": seq.status()}
    seq.close()
    del keep
    return out


def int8_step(torch, w4, st, reps=100):
    """The same 28-layer step on the pages' Path A: x (binary16, as in the
    headline) quantised per token to INT8 inside the kernel and dotted with
    dp4a.  us/step and weight GB/s, to set against the binary16 headline."""
    nbw = w4.w4_decode_seq_workspace_bytes(st["ws"], 1)
    buf = torch.zeros(nbw + 256, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % 256
    ys = [torch.zeros_like(y) for y in st["ys"]]
    seq = w4.DecodeSeq(st["ws"], st["xs"], ys, 1, workspace=buf[off:off + nbw], act="int8")
    for _ in range(5):
        seq.replay()
    ms = time_replays(torch, seq.replay, reps)
    peak = measured_peaks()[0].get("hbm_gbs", FALLBACK_HBM_GBS)
    out = {"us_per_step": ms * 1e3, "GB/s": BYTES_PER_STEP / (ms * 1e-3) / 1e9,
           "frac_of_hbm": BYTES_PER_STEP / (ms * 1e-3) / 1e9 / peak, "status_word": seq.status()}
    seq.close()
    return out


def packed_file_load(torch, w4, st):
    """Layer 0's four packed weights written to packed-weight files and read
    back (header + checksum validation + one host-to-device copy each) into
    device buffers: seconds and GB/s of payload, page-cache warm."""
    import tempfile
    import shutil
    d = tempfile.mkdtemp(prefix="w4pk_")
    try:
        idx = [i for i, m in enumerate(st["meta"]) if m[0] == 0]
        paths, nb = [], 0
        t0 = time.perf_counter()
        for i in idx:
            p = os.path.join(d, "l0_p%d.pk" % i)
            w4.w4_file_write(p, st["ws"][i], src_on_device=True)
            paths.append(p)
            nb += w4.w4_packed_bytes(st["meta"][i][2], st["meta"][i][3])
        t_write = time.perf_counter() - t0
        bufs = [torch.empty(w4.w4_packed_bytes(st["meta"][i][2], st["meta"][i][3]), dtype=torch.uint8,
                            device="cuda") for i in idx]
        for p, b in zip(paths, bufs):  # warm the page cache
            w4.w4_file_read(p, b)
        reps = 3
        t0 = time.perf_counter()
        for _ in range(reps):
            for p, b in zip(paths, bufs):
                w4.w4_file_read(p, b)
        t_read = (time.perf_counter() - t0) / reps
        same = all(torch.equal(b, st["keep"][i][:b.numel()]) for i, b in zip(idx, bufs))
        return {"bytes": nb, "write_s": t_write, "read_s": t_read, "read_GB/s": nb / t_read / 1e9,
                "bit_exact": bool(same)}
    finally:
        shutil.rmtree(d, ignore_errors=True)


# ---- main ------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-extras", action="store_true",
                    help="time the step only (no clock soak, e2e, side measurements or CPU baseline): for profilers")
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="with --no-extras: a step of the first L layers only (a small case for a profiler; "
                         "prints a profiler line, not the benchmark line)")
    ap.add_argument("--profile-projection", choices=[n for n, _, _ in LAYER], default=None,
                    help="launch one projection of layer 0 (library launch shape) --steps times: a small "
                         "case for a profiler")
    ap.add_argument("--act", choices=("fp16", "bf16", "int8"), default="fp16",
                    help="with --no-extras: activation path of the step (bf16 = bfloat16 x and y, x drawn from "
                         "the same seeds; int8 = Path A, x quantised in the kernel)")
    ap.add_argument("--tokens", type=int, default=1,
                    help="with --no-extras: tokens per step (1..16; the benchmark line is always M=1)")
    ap.add_argument("--profile-m", type=int, default=1,
                    help="with --profile-projection: tokens (M > 16 runs the prefill GEMM)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.profile_projection:
        return run_one_projection(args)

    import torch
    rank, world, local = rank_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    import int4_weight_only_pack_gb300 as w4
    from int4_weight_only_pack_gb300 import build as w4build
    import synth
    if rank == 0 or world == 1:
        w4build.build()
        synth.build_device()
    if world > 1:
        dist.barrier()
    torch.cuda.set_device(local)
    M = max(1, min(args.tokens, 16)) if args.no_extras else 1
    layers = max(1, min(args.layers, LAYERS)) if args.no_extras else LAYERS
    st = build_step(torch, w4, synth, M, layers)
    nbw = w4.w4_decode_seq_workspace_bytes(st["ws"], M)
    ws_buf = torch.zeros(nbw + 256, dtype=torch.uint8, device="cuda")
    ws_off = (-ws_buf.data_ptr()) % 256
    act = args.act if args.no_extras else "fp16"
    if act == "bf16":  # bfloat16 x of the same seeds (the binary16 bits would not be valid bfloat16 inputs)
        st["xs"] = [torch.from_numpy(synth.x_full_bf16(synth.seed_of(CONFIG_ID, layer, pid, synth.T_X), M, K)
                                     .view(np.int16).ravel()).cuda() for (layer, pid, N, K) in st["meta"]]
    seq = w4.DecodeSeq(st["ws"], st["xs"], st["ys"], M, workspace=ws_buf[ws_off:ws_off + nbw], act=act)
    for _ in range(args.warmup):
        seq.replay()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # soak ~1.5 s so that the clock record sees the GPU under this load
    sampler = ClockSampler(local) if not args.no_extras else None
    if not args.no_extras:
        soak = max(1, int(1.5 / max(time_replays(torch, seq.replay, 20) * 1e-3, 1e-5)))
        for _ in range(soak):
            seq.replay()
    barrier()
    s = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(s)
    for _ in range(args.steps):
        seq.replay()
    ev1.record(s)
    barrier()
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(torch, ev0.elapsed_time(ev1) / args.steps, world)
    if layers != LAYERS or M != 1:
        nb = BYTES_PER_STEP // LAYERS * layers
        if rank == 0:
            print(json.dumps({"profile_case": "decode step of the first %d layers, M=%d, %s activations" % (layers, M, act),
                              "bytes_per_step": nb, "us_per_step": ms * 1e3, "GB/s": nb / (ms * 1e-3) / 1e9,
                              "status_word": seq.status()}), flush=True)
        seq.close()
        return 0
    value = job_gbs(world, ms)
    per_gpu = job_gbs(1, ms)
    launches = seq.kernels()

    # e2e through the C ABI with host buffers: pinned x in, replay, y out, sync
    xb, yb = st["x_arena"].numel() * 2, st["y_arena"].numel() * 2
    e2e_s = None
    if not args.no_extras:
        x_pin = torch.from_numpy(st["x_host"]).pin_memory()
        y_pin = torch.empty(st["y_arena"].numel(), dtype=torch.int16).pin_memory()
        for _ in range(3):
            seq.run_host(x_pin, st["x_arena"], xb, st["y_arena"], y_pin, yb, s)
        e2e_steps = max(10, min(args.steps, 500))
        barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            seq.run_host(x_pin, st["x_arena"], xb, st["y_arena"], y_pin, yb, s)
        e2e_s = max_over_ranks(torch, (time.perf_counter() - t0) / e2e_steps, world)

    extras = {}
    if not args.no_extras:
        extras["persistent_launch_without_graph_us_per_step"] = time_replays(torch, seq.eager, 50) * 1e3
        extras["persistent_status_word"] = seq.status()
        g = w4.DecodeSeq(st["ws"], st["xs"], st["ys"], M, use_pdl=True)
        extras["graph_of_112_kernels_pdl_us_per_step"] = time_replays(torch, g.replay, 100) * 1e3
        extras["eager_112_kernels_pdl_us_per_step"] = time_replays(torch, g.eager, 20) * 1e3
        g.close()
        nopdl = w4.DecodeSeq(st["ws"], st["xs"], st["ys"], M, use_pdl=False)
        extras["graph_of_112_kernels_no_pdl_us_per_step"] = time_replays(torch, nopdl.replay, 100) * 1e3
        extras["eager_112_kernels_no_pdl_us_per_step"] = time_replays(torch, nopdl.eager, 20) * 1e3
        nopdl.close()
        per = {}
        for pid, (name, N, K) in enumerate(LAYER):
            idx = [i for i, m in enumerate(st["meta"]) if m[1] == pid]
            one = w4.DecodeSeq([st["ws"][i] for i in idx], [st["xs"][i] for i in idx],
                               [st["ys"][i] for i in idx], M, use_pdl=True)
            us = time_replays(torch, one.replay, 100) * 1e3 / len(idx)
            nb = (N * K) // 2 + N * (K // 128) * 2
            cfg = w4.w4a16_gemv_default_config(M, N, K)
            per[name] = {"us": us, "GB/s": nb / (us * 1e-6) / 1e9, "bytes": nb,
                         "launch": {"bands_per_cta": cfg.bands_per_cta, "splits": cfg.splits,
                                    "depth": cfg.depth}}
            one.close()
        extras["per_projection_back_to_back_28_layers"] = per
        # the same 28 projections of one type chained in the persistent step
        # kernel (each still waits for the previous one to finish)
        perp = {}
        for pid, (name, N, K) in enumerate(LAYER):
            idx = [i for i, m in enumerate(st["meta"]) if m[1] == pid]
            wsl = [st["ws"][i] for i in idx]
            nbw1 = w4.w4_decode_seq_workspace_bytes(wsl, M)
            wb1 = torch.zeros(nbw1 + 256, dtype=torch.uint8, device="cuda")
            o1 = (-wb1.data_ptr()) % 256
            one = w4.DecodeSeq(wsl, [st["xs"][i] for i in idx], [st["ys"][i] for i in idx], M,
                               workspace=wb1[o1:o1 + nbw1])
            for _ in range(3):
                one.replay()
            us = time_replays(torch, one.replay, 100) * 1e3 / len(idx)
            nb = (N * K) // 2 + N * (K // 128) * 2
            perp[name] = {"us": us, "GB/s": nb / (us * 1e-6) / 1e9, "bytes": nb,
                          "frac_of_hbm": nb / (us * 1e-6) / 1e9 / measured_peaks()[0].get("hbm_gbs", 6698.2),
                          "status_word": one.status()}
            one.close()
            del wb1
        extras["per_projection_persistent_chain_28_layers"] = perp
        # per projection boundary of the 112-launch graph (all figures CUDA-event timed): its time above
        # the persistent step kernel's (same chain, one launch) and above the HBM-bound floor of the
        # step's bytes at the measured copy bandwidth, each divided by the 112 boundaries
        floor_us = BYTES_PER_STEP / (measured_peaks()[0].get("hbm_gbs", FALLBACK_HBM_GBS) * 1e9) * 1e6
        nproj = LAYERS * len(LAYER)
        extras["graph_of_112_kernels_per_boundary_us"] = {
            "pdl_over_persistent": (extras["graph_of_112_kernels_pdl_us_per_step"] - ms * 1e3) / nproj,
            "no_pdl_over_persistent": (extras["graph_of_112_kernels_no_pdl_us_per_step"] - ms * 1e3) / nproj,
            "pdl_over_hbm_floor": (extras["graph_of_112_kernels_pdl_us_per_step"] - floor_us) / nproj,
            "persistent_over_hbm_floor": (ms * 1e3 - floor_us) / nproj,
            "hbm_floor_us_per_step": floor_us}
        extras["step_replay_spread_M1"] = replay_spread(torch, seq.replay, 100)
        extras["single_gemv_qkv_M1_rotated"] = single_gemv_rotated(torch, w4, synth, st)
        extras["small_batch_step"] = small_batch_sweep(torch, w4, synth, st)
        extras["prefill_M512"] = prefill_layer(torch, w4, synth, st)
        extras["packed_file_layer0"] = packed_file_load(torch, w4, st)
        extras["bf16_activations_step_M1"] = bf16_step(torch, w4, synth, st)
        extras["swiglu_fused_gate_up_step_M1"] = swiglu_step(torch, w4, synth, st)
        extras["path_a_int8_step_M1"] = int8_step(torch, w4, st)

    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    roof = {"bound": "hbm", "achieved": per_gpu, "peak": peak, "unit": "GB/s", "frac": per_gpu / peak,
            "traffic": ncu_traffic_per_launch(),
            "kernel": "persistent decode-step kernel (one launch per step streams all 112 projections); "
                      "achieved = algorithmic bytes per launch (%d) / average launch duration over the timed "
                      "region" % (BYTES_PER_STEP // launches),
            "peak_source": "%s hbm_gbs (MEASURED_PEAKS.json)" % peak_kind if peak_kind == "measured"
            else "fallback 6.8 TB/s"}
    if roof["traffic"] is not None:
        roof["traffic"] = roof["traffic"]

    cpu = None
    if rank == 0 and not args.no_extras:
        import oracle
        cpu = cpu_baseline(oracle, synth)
        extras["cpu_oracle_single_gemv_one_thread"] = cpu_single_gemv_one_thread(oracle, synth)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "us_per_step": ms * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
                "config": {"workload": WORKLOAD, "M": M, "layers": LAYERS, "projections_per_step": len(st["ws"]),
                           "bytes_per_step": BYTES_PER_STEP, "accumulate": "f32",
                           "l2": "inputs larger than L2: 3.36 GB of weights per step vs 129 MB L2",
                           "launch": "one cudaGraphLaunch per step of a one-node graph: the persistent "
                                     "cooperative decode-step kernel (one CTA per SM)",
                           "parallelism": "replicas" if world > 1 else "single GPU"},
                "roofline": roof,
                "cpu_baseline": cpu,
                "e2e": None if e2e_s is None else {
                    "value": job_gbs(world, e2e_s * 1e3), "unit": "GB/s",
                    "us_per_step": e2e_s * 1e6, "h2d_bytes_per_step": xb, "d2h_bytes_per_step": yb,
                    "via": "w4_decode_seq_run_host (pinned host x -> device, replay, device y -> pinned host, sync)"},
                "gpu_launches": launches * args.steps,
                "clocks": clocks,
                "target_us_per_step": 550.0,
                "extras": extras,
                "host": {"arch": platform.machine(), "nproc": os.cpu_count(),
                         "gpu": torch.cuda.get_device_name(local),
                         "sm_count": torch.cuda.get_device_properties(local).multi_processor_count}}
        print(json.dumps(line), flush=True)
    seq.close()
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
