#!/usr/bin/env python
"""Benchmark of the streaming encoder step's paged-KV chunk attention on GB300.

A step is one streaming encoder step of a lockstep cohort through `layers` attention
layers: per layer, the new chunk's K/V are appended into that layer's block-paged pool
and the chunk attends over cache + chunk with the shared Transformer-XL rel-pos term
(one fused launch per layer, oasr_chunk_step_paged).  Each layer has its own pools and
inputs, so the step's working set is several times the 129 MB L2 and no layer is
served from the previous one's cache.

Prints one JSON line (rank 0).  `value` is encoder frames per second per attention layer
(B*T*layers*steps / time) over all ranks, timed on the device with CUDA events around
CUDA-graph replays of the step, inputs resident in HBM.  `e2e` is the same metric with the
step's inputs copied from pinned host memory and its outputs copied back inside the
timed region.  `roofline` relates the fused kernel's algorithmic bytes to its average
launch time and the measured HBM peak.  `cpu_baseline` times the fp64 CPU oracle on a
bounded sample of the same workload.

--impl reference times the oracle itself on the host cores as the reference arm.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_chunk_gb300 import dist as pdist  # noqa: E402
from paged_kv_chunk_gb300 import synthetic as syn  # noqa: E402

METRIC = "encoder frames/s per attention layer and achieved HBM GB/s vs GB300 peak"
UNIT = "frames/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0   # the ~8 TB/s the streaming step's HBM target is stated against
KERNEL_SOURCES = ["chunk_attn.cu", "attn_core.cuh", "ptx.cuh"]
# chunks of 33..64 frames with an even head count run the append, then the tensor-core kernel
TC_STREAM_SOURCES = ["chunk_tc.cu", "append.cu", "tcgen05.cuh", "attn_core.cuh", "ptx.cuh"]


def uses_tc_stream(T, H):
    """Whether the library runs a streaming step of chunk length T over H heads as the paged
    append followed by the tcgen05 kernel (the dispatch rule of chunk_attn.cu)."""
    return 33 <= T <= 64 and H % 2 == 0
PACKED_SOURCES = ["packed_tc.cu", "tcgen05.cuh", "attn_core.cuh", "ptx.cuh"]
# the chunked-limited packed call (even H) runs the packed mode of the streaming tensor-core kernel
CHUNKED_SOURCES = ["chunk_tc.cu", "tcgen05.cuh", "attn_core.cuh", "ptx.cuh"]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="conformer_large",
                    choices=sorted(syn.STREAMING_CONFIGS) + [syn.PACKED.name, NEMOTRON]
                    + sorted(PROJECTIONS))
    ap.add_argument("--two-call", action="store_true",
                    help="time oasr_paged_append + oasr_chunk_relattn_paged instead of the fused step")
    ap.add_argument("--layers", type=int, default=0,
                    help="distinct layer pools per step (0: enough for 4x L2)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work of the cpu_baseline sample (0 disables it)")
    ap.add_argument("--soak-seconds", type=float, default=1.5,
                    help="untimed replays before the timed region, for the clock record")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--mbps", type=int, default=0,
                    help="block-table width (max_blocks_per_seq) of a streaming cohort; entries past "
                         "its pages are -1, as in an engine table sized for unlimited history "
                         "(0: the pages the history needs)")
    return ap.parse_args()


# --------------------------------------------------------------------------- helpers


def workload_bytes(cfg, fused=True):
    """Algorithmic HBM bytes of one layer step (one launch of the fused kernel); a
    heterogeneous cohort reads each stream's own cache length."""
    es = 2 if cfg.dtype == "bf16" else 4
    row = cfg.H * cfg.D * es
    chunk = cfg.B * cfg.T * row
    b = 2 * chunk                       # read k_new, v_new
    b += 2 * chunk                      # write them into the pools
    b += 2 * int(syn.cache_lengths(cfg).sum()) * row   # read the cached K/V
    if not fused:
        b += 2 * chunk                  # re-read the appended chunk
    b += chunk                          # read q
    b += cfg.R * row                    # read the shared rel table once
    b += chunk                          # write out
    return b


def packed_flops(lengths, H, D):
    """Algorithmic flops of one packed call: per (query, key) pair of a segment and head,
    the content dot, the position dot and the P.V row each take 2*D flops."""
    L = np.asarray(lengths, dtype=np.float64)
    return float((L * L).sum()) * H * 6 * D


# The packed row under the Nemotron offline window (chunked_limited: own chunk of 8 frames
# plus 7 earlier chunks, so a 64-frame query block sees 120 keys).
NEMOTRON = "nemotron_offline"
NEMOTRON_CHUNK, NEMOTRON_LEFT = 8, 7


def chunked_pairs(lengths, cs, left):
    """Visible (query, key) pairs of one call under the chunked-limited window."""
    n = 0
    for L in np.asarray(lengths, dtype=np.int64):
        i = np.arange(L)
        lo = np.maximum(0, (i // cs - left) * cs)
        hi = np.minimum(L, (i // cs + 1) * cs)
        n += int((hi - lo).sum())
    return n


def packed_bytes(total, R, H, D, es=2):
    return (4 * total + R) * H * D * es


def measured_tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digest(sources=None):
    """Digest of the kernel sources' code: comments and blank space are dropped first, so a
    comment edit does not void a profile taken on the same code."""
    h = hashlib.sha256()
    for name in (sources or KERNEL_SOURCES):
        with open(os.path.join(ROOT, "paged_kv_chunk_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


TRAFFIC_FILE = os.path.join("profiles", "traffic.json")


def profiled_traffic(profile_name, sources=None):
    """(DRAM bytes per launch, where from) of the ncu capture recorded under `profile_name` in
    profiles/traffic.json, when that capture was taken on the current kernel source; else
    (None, why not).  The bytes are dram__bytes_read.sum + dram__bytes_write.sum of one launch
    of an earlier capture, not of this run."""
    path = os.path.join(ROOT, TRAFFIC_FILE)
    try:
        with open(path) as f:
            rec = json.load(f).get(profile_name)
    except (OSError, ValueError):
        rec = None
    if not rec:
        return None, "no ncu capture recorded for this workload"
    digest = source_digest(sources)
    if rec.get("kernel_source_sha") != digest:
        return None, (f"the recorded capture is of kernel source {rec.get('kernel_source_sha')}, "
                      f"not the current {digest}")
    return float(rec["dram_bytes_per_launch"]), (
        f"ncu capture of kernel source {digest} recorded in {TRAFFIC_FILE} (not this run): "
        f"{rec.get('capture')}")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = list(csv.reader(io.StringIO(self.tmp.read())))
        self.tmp.close()
        os.unlink(self.tmp.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    return pdist.setup()


def barrier(world):
    pdist.barrier()


def max_over_ranks(x, world):
    return pdist.max_over_ranks(x)


# ------------------------------------------------------------------ CPU oracle legs


def oracle_layer_inputs(cfg, seed):
    x = syn.streaming_inputs(cfg, seed)
    x["cache_seqlens"] = syn.cache_lengths(cfg)   # a heterogeneous cohort's own lengths
    kp = syn.canary_pool(x["num_blocks"], cfg.block_size, cfg.H, cfg.D, cfg.dtype)
    vp = kp.copy()
    return x, kp, vp


def oracle_layer_step(oracle, cfg, x, kp, vp):
    """One layer step on the CPU oracle: append the chunk, then chunk attention (stream by
    stream over its own cache length in a heterogeneous cohort)."""
    oracle.paged_append(syn.to_bits(x["k_new"], cfg.dtype), syn.to_bits(x["v_new"], cfg.dtype),
                        kp, vp, x["block_table"], x["cache_seqlens"])
    if not cfg.hetero:
        oracle.chunk_relattn(x["q"], x["cache_k"], x["cache_v"], x["k_new"], x["v_new"],
                             x["pos_bias_u"], x["pos_bias_v"], x["rel"])
        return
    for b, c in enumerate(x["cache_seqlens"]):
        s = slice(b, b + 1)
        oracle.chunk_relattn(x["q"][s], x["cache_k"][s, :c], x["cache_v"][s, :c], x["k_new"][s],
                             x["v_new"][s], x["pos_bias_u"], x["pos_bias_v"], x["rel"])


def cpu_baseline(cfg, seconds):
    import oracle
    oracle.build()
    x, kp, vp = oracle_layer_inputs(cfg, cfg.seed)
    oracle_layer_step(oracle, cfg, x, kp, vp)   # untimed first call
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_layer_step(oracle, cfg, x, kp, vp)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    cores = oracle.num_threads()
    # the same on one thread, on a shorter sample
    oracle.set_num_threads(1)
    n1, t1 = 0, time.perf_counter()
    try:
        while True:
            oracle_layer_step(oracle, cfg, x, kp, vp)
            n1 += 1
            el1 = time.perf_counter() - t1
            if el1 >= seconds / 2:
                break
    finally:
        oracle.set_num_threads(cores)
    return {"value": cfg.B * cfg.T * n / el, "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"{n} layer steps (append + chunk attention of all {cfg.B} streams x "
                      f"{cfg.H} heads, one layer) of the {cfg.name} cohort, {el:.1f} s, "
                      "fp64 C oracle with OpenMP",
            "single_thread": {"value": cfg.B * cfg.T * n1 / el1, "unit": UNIT, "cores": 1,
                              "sample": f"{n1} layer steps, {el1:.1f} s"}}


def run_reference(args, cfg, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    x, kp, vp = oracle_layer_inputs(cfg, cfg.seed)
    for _ in range(args.warmup):
        oracle_layer_step(oracle, cfg, x, kp, vp)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_layer_step(oracle, cfg, x, kp, vp)
    el = time.perf_counter() - t0
    value = cfg.B * cfg.T * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{cfg.name}_streaming", "B": cfg.B, "H": cfg.H, "D": cfg.D,
                   "T": cfg.T, "cache": (f"U{{0..{cfg.C}}} per stream" if cfg.hetero else cfg.C),
                   "block_size": cfg.block_size, "layers": 1},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"each step: one layer (append + chunk attention) of the "
                                   f"{cfg.name} cohort on the fp64 C oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def sequential_e2e(stream, h2d_pairs, run, d2h_pairs, steps, warmup, world):
    """End to end through the public API: every step copies its inputs from pinned host memory
    (h2d_pairs: (device tensor, pinned host tensor)), runs, and copies its outputs back
    (d2h_pairs: (pinned host tensor, device tensor)), all on `stream`, inside the timed
    region.  Returns (ms for all steps, max over ranks; H2D bytes per step; D2H bytes)."""
    def one():
        for dst, src in h2d_pairs:
            dst.copy_(src, non_blocking=True)
        run()
        for dst, src in d2h_pairs:
            dst.copy_(src, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0 = time.perf_counter()
        e0.record(stream)
        for _ in range(steps):
            one()
        e1.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - w0
    barrier(world)
    ms = max_over_ranks(max(e0.elapsed_time(e1), 1e3 * wall), world)
    h2d = sum(t.numel() * t.element_size() for _, t in h2d_pairs)
    d2h = sum(t.numel() * t.element_size() for t, _ in d2h_pairs)
    return ms, int(h2d), int(d2h)


def offline_oracle_sample(name):
    """(step, frames, workload, sample): one call of the oracle on a bounded sample of the
    packed row, the Nemotron window or a projection workload, and what it covers."""
    import oracle
    oracle.build()
    if name in PROJECTIONS:
        p = PROJECTIONS[name]
        H, R = p["H"], p["R"]
        M, d = p["B"] * p["T"], 64 * H
        rng = np.random.default_rng(p["seed"])
        x, pe = rng.standard_normal((M, d)) * syn.SIGMA, rng.standard_normal((R, d)) * syn.SIGMA
        wq, wp = rng.standard_normal((3 * d, d)) * d ** -0.5, rng.standard_normal((d, d)) * d ** -0.5
        bq = rng.standard_normal(3 * d) * syn.SIGMA

        def step():
            oracle.project_qkv_pos(x, wq, bq, pe, wp, H)
        frames, workload = M, f"{name}_qkv_pos"
        sample = f"each step: one layer's projections ({M} frames, d {d}, {R} rel rows), float64"
    else:
        window = (NEMOTRON_CHUNK, NEMOTRON_LEFT) if name == NEMOTRON else None
        cfg = syn.PACKED
        x = syn.packed_inputs(cfg, cfg.seed)
        cu = x["cu_seqlens"]
        sq = np.cumsum(np.asarray(x["lengths"], np.float64) ** 2)
        n = int(min(len(sq), np.searchsorted(sq, 1.5e6) + 1))   # first segments, ~1.5e6 pairs
        e = int(cu[n])
        sub = {k: x[k][:e] for k in ("q", "k", "v")}

        def step():
            if window:
                oracle.packed_relattn_chunked(sub["q"], sub["k"], sub["v"], cu[:n + 1],
                                              x["pos_bias_u"], x["pos_bias_v"], x["rel"], *window)
            else:
                oracle.packed_relattn(sub["q"], sub["k"], sub["v"], cu[:n + 1], x["pos_bias_u"],
                                      x["pos_bias_v"], x["rel"])
        frames = e
        workload = "nemotron_chunked_offline" if window else "packed_varlen_offline"
        sample = f"each step: the first {n} of the {cfg.num_seqs} utterances ({e} frames) on the fp64 C oracle"
    return step, frames, workload, sample


def offline_cpu_baseline(name, seconds):
    """cpu_baseline of an offline workload: the oracle on its bounded sample for ~seconds."""
    import oracle
    step, frames, _, sample = offline_oracle_sample(name)
    step()
    n, t0 = 0, time.perf_counter()
    while True:
        step()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": frames * n / el, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{sample}; {n} steps in {el:.1f} s"}


def run_reference_offline(args, name, rank):
    """Reference arm of the packed row, the Nemotron window and the projections: the oracle
    on the host cores, each step a bounded sample of the same workload."""
    if rank != 0:
        return
    import oracle
    step, frames, workload, sample = offline_oracle_sample(name)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = frames * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm


def run_ours(args, cfg, rank, world, local):
    from paged_kv_chunk_gb300 import build as pkg_build
    from paged_kv_chunk_gb300 import capi
    pkg_build.build()
    capi.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    tdtype = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    es = 2 if cfg.dtype == "bf16" else 4
    touched = workload_bytes(cfg, fused=not args.two_call)
    layers = args.layers or max(1, math.ceil(4 * L2_BYTES / touched))
    rng = np.random.default_rng(cfg.seed + 1000 * rank)
    gen = torch.Generator(device=dev)
    gen.manual_seed(cfg.seed + 7919 * rank)
    B, T, H, D = cfg.B, cfg.T, cfg.H, cfg.D
    nb, bs = cfg.pool_blocks, cfg.block_size

    def dev_normal(shape):
        return (torch.randn(shape, generator=gen, device=dev) * syn.SIGMA).to(tdtype)

    pools = [(dev_normal((nb, bs, H, D)), dev_normal((nb, bs, H, D))) for _ in range(layers)]
    params = [(dev_normal((H, D)), dev_normal((H, D)), dev_normal((cfg.R, H, D)))
              for _ in range(layers)]
    mbps = max(args.mbps, cfg.mbps)
    bt_h = np.full((B, mbps), -1, np.int32)
    bt_h[:, :cfg.mbps] = syn.block_table(rng, B, cfg.mbps, nb)
    cs_h = syn.cache_lengths(cfg)
    bt = torch.from_numpy(bt_h).to(dev)
    cs = torch.from_numpy(cs_h).to(dev)
    # per-step inputs of every layer (q, k_new, v_new) and outputs, device-resident
    x_h = torch.from_numpy(syn.normal(rng, (layers, 3, B, T, H, D), cfg.dtype)).to(tdtype)
    x_d = x_h.to(dev)
    out_d = torch.empty((layers, B, T, H, D), dtype=tdtype, device=dev)

    def step_calls(x, out):
        for l in range(layers):
            kp, vp = pools[l]
            u, vb, rel = params[l]
            if args.two_call:
                capi.oasr_paged_append(x[l, 1], x[l, 2], kp, vp, bt, cs)
                capi.oasr_chunk_relattn_paged(x[l, 0], kp, vp, bt, cs, u, vb, rel, out=out[l])
            else:
                capi.oasr_chunk_step_paged(x[l, 0], x[l, 1], x[l, 2], kp, vp, bt, cs, u, vb, rel,
                                           out=out[l])
        if cfg.window:
            # the step's commit: the block table is shared by the layers, so once per step
            capi.oasr_window_commit(bt, cs, T, bs, cfg.window)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        step_calls(x_d, out_d)              # eager once: kernel attributes, lazy loading
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step_calls(x_d, out_d)
    torch.cuda.synchronize()

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        t_end = time.perf_counter() + args.soak_seconds
        while time.perf_counter() < t_end:
            for _ in range(20):
                graph.replay()
            stream.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    clocks = sampler.stop() if sampler else None
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, world)
    frames = B * T * layers * args.steps * world
    value = frames / (ms_max / 1e3)
    launch_us = 1e3 * ms / (args.steps * layers)

    # ---- one cold-L2 launch: layer 0's step alone, L2 overwritten (2x its size) before each
    cold = None
    if rank == 0:
        flush = torch.empty(int(2 * L2_BYTES), dtype=torch.uint8, device=dev)
        n_cold = 20
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_cold)]
        kp, vp = pools[0]
        u, vb, rel = params[0]
        with torch.cuda.stream(stream):
            for i in range(n_cold):
                flush.fill_(i & 0xFF)
                evs[i][0].record(stream)
                if args.two_call:
                    capi.oasr_paged_append(x_d[0, 1], x_d[0, 2], kp, vp, bt, cs)
                    capi.oasr_chunk_relattn_paged(x_d[0, 0], kp, vp, bt, cs, u, vb, rel,
                                                  out=out_d[0])
                else:
                    capi.oasr_chunk_step_paged(x_d[0, 0], x_d[0, 1], x_d[0, 2], kp, vp, bt, cs, u,
                                               vb, rel, out=out_d[0])
                evs[i][1].record(stream)
        torch.cuda.synchronize()
        del flush
        cold_us = float(np.median([1e3 * a.elapsed_time(b) for a, b in evs[3:]]))
        cold = {"launch_us": cold_us, "achieved_gbs": touched / (cold_us * 1e-6) / 1e9,
                "launches": n_cold - 3,
                "how": "median of single eager launches of one layer's step, each after a "
                       "write of 2x L2 on the same stream, CUDA events around the launch"}

    # ---- end to end: pinned host inputs -> device, the step, outputs -> pinned host.  Every
    # step's inputs are copied in and its outputs copied out inside the timed region; the
    # copies of step i+1 overlap the compute of step i (two device input/output sets, one
    # graph per set, H2D and D2H on streams of their own).
    e2e = None
    if not args.no_e2e:
        x_pin = x_h.pin_memory()
        out_pin = torch.empty(out_d.shape, dtype=tdtype).pin_memory()
        bt_pin = torch.from_numpy(bt_h).pin_memory()
        cs_pin = torch.from_numpy(cs_h).pin_memory()
        x2, out2 = [x_d, torch.empty_like(x_d)], [out_d, torch.empty_like(out_d)]
        bt2, cs2 = [bt.clone(), bt.clone()], [cs.clone(), cs.clone()]
        graphs = []
        for p_ in range(2):
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_, stream=stream):
                for l in range(layers):
                    kp, vp = pools[l]
                    u, vb, rel = params[l]
                    if args.two_call:
                        capi.oasr_paged_append(x2[p_][l, 1], x2[p_][l, 2], kp, vp, bt2[p_], cs2[p_])
                        capi.oasr_chunk_relattn_paged(x2[p_][l, 0], kp, vp, bt2[p_], cs2[p_], u, vb,
                                                      rel, out=out2[p_][l])
                    else:
                        capi.oasr_chunk_step_paged(x2[p_][l, 0], x2[p_][l, 1], x2[p_][l, 2], kp, vp,
                                                   bt2[p_], cs2[p_], u, vb, rel, out=out2[p_][l])
                if cfg.window:
                    capi.oasr_window_commit(bt2[p_], cs2[p_], T, bs, cfg.window)
            graphs.append(g_)
        torch.cuda.synchronize()
        h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def ev():
            return torch.cuda.Event()

        def run_steps(n):
            """n pipelined steps; returns after enqueueing (the caller synchronises)."""
            h2d_done, comp_done, d2h_done = {}, {}, {}

            def h2d(i):
                p_ = i & 1
                with torch.cuda.stream(h2d_s):
                    if i >= 2:
                        h2d_s.wait_event(comp_done[i - 2])   # the set's last reader is done
                    x2[p_].copy_(x_pin, non_blocking=True)
                    if not cfg.window:   # a windowed cohort's tables live on the device
                        bt2[p_].copy_(bt_pin, non_blocking=True)
                        cs2[p_].copy_(cs_pin, non_blocking=True)
                    h2d_done[i] = ev()
                    h2d_done[i].record(h2d_s)

            h2d(0)
            for i in range(n):
                p_ = i & 1
                stream.wait_event(h2d_done[i])
                if i >= 2:
                    stream.wait_event(d2h_done[i - 2])       # its outputs have been read back
                graphs[p_].replay()
                comp_done[i] = ev()
                comp_done[i].record(stream)
                if i + 1 < n:
                    h2d(i + 1)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(comp_done[i])
                    out_pin.copy_(out2[p_], non_blocking=True)
                    d2h_done[i] = ev()
                    d2h_done[i].record(d2h_s)

        run_steps(max(3, args.warmup))
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0 = time.perf_counter()
        e0.record(stream)
        h2d_s.wait_event(e0)
        run_steps(args.steps)
        stream.wait_stream(d2h_s)
        stream.wait_stream(h2d_s)
        e1.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - w0
        barrier(world)
        e_ms = max(e0.elapsed_time(e1), 1e3 * wall)
        e_ms = max_over_ranks(e_ms, world)
        h2d = x_pin.numel() * es + (0 if cfg.window else bt_pin.numel() * 4 + cs_pin.numel() * 4)
        e2e = {"value": frames / (e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(out_pin.numel() * es),
               "path": "per step: pinned host q/k_new/v_new (and tables) -> H2D copy -> CUDA-graph "
                       "replay of the per-layer oasr_chunk_step_paged calls -> D2H copy of the "
                       "outputs; step i+1's H2D overlaps step i's compute (two device buffer sets, "
                       "H2D and D2H on streams of their own)"}

    if rank != 0:
        return
    peak, peak_kind = measured_hbm_peak()
    achieved = touched / (launch_us * 1e-6) / 1e9
    tc = uses_tc_stream(T, H)
    traffic, traffic_src = ((None, "not captured for the two-call step") if args.two_call
                            else profiled_traffic(f"chunk_step_{cfg.name}",
                                                  TC_STREAM_SOURCES if tc else None))
    if tc:
        kernel = "paged_append_kernel + chunk_attn_tc_kernel"
    elif args.two_call:
        kernel = "paged_append_kernel + chunk_attn_bf16_kernel"
    else:
        kernel = "chunk_attn_bf16_kernel (fused append + attention)"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
        "config": {"workload": f"{cfg.name}_streaming", "B": B, "H": H, "D": D, "T": T,
                   **({"window_frames": cfg.window, "commit": "oasr_window_commit once per step"}
                      if cfg.window else {}),
                   "cache": (f"U{{0..{cfg.C}}} per stream (mean {cs_h.mean():.1f})" if cfg.hetero
                             else cfg.C),
                   "block_size": bs, "pool_blocks": nb, "rel_rows": cfg.R,
                   "max_blocks_per_seq": mbps,
                   "layers": layers, "global_batch": B * world, "seq_len": cfg.K,
                   "parallelism": f"dp{world}",
                   "l2": f"inputs larger than L2: {layers} distinct layer pools, "
                         f"{layers * touched / 1e6:.0f} MB touched per step",
                   "timing": "CUDA events around graph replays of the step on the launching stream",
                   "soak_s": args.soak_seconds},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "traffic_source": traffic_src,
                     "frac_of_8tbs": achieved / NOMINAL_HBM_GBS,
                     "kernel": kernel,
                     "algorithmic_bytes_per_launch": touched,
                     "avg_launch_us": launch_us, "peak_kind": peak_kind,
                     **({"cold_l2": {**cold, "frac": cold["achieved_gbs"] / peak}} if cold else {})},
        "gpu_launches": args.steps * (layers * (2 if args.two_call or tc else 1) + (1 if cfg.window else 0)),
        "clocks": clocks,
    }
    if e2e:
        line["e2e"] = e2e
    if world == 1 and args.cpu_seconds > 0:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_seconds)
    print(json.dumps(line), flush=True)


# The projections that feed the path, at the Conformer cohorts' shapes: q/k/v with bias for
# the B*T frames of a step and the positional projection of the R-row table.
PROJECTIONS = {"projection_small": dict(B=64, T=16, H=4, R=287, seed=1020),
               "projection_large": dict(B=256, T=16, H=8, R=543, seed=1021)}


def run_projection(args, rank, world, local, name):
    """One step = the projections of `layers` distinct layers (inputs and weights larger than
    L2 between steps), one oasr_project_qkv_pos launch per layer, replayed as a CUDA graph."""
    from paged_kv_chunk_gb300 import build as pkg_build
    from paged_kv_chunk_gb300 import capi
    pkg_build.build()
    capi.load()
    p = PROJECTIONS[name]
    B, T, H, R = p["B"], p["T"], p["H"], p["R"]
    M, d = B * T, 64 * H
    dev = torch.device("cuda", torch.cuda.current_device())
    gen = torch.Generator(device=dev)
    gen.manual_seed(p["seed"] + 7919 * rank)
    per_layer = 2 * (M * d + 3 * d * d + 3 * d + R * d + d * d + 3 * M * d + R * d)
    layers = args.layers or max(1, math.ceil(4 * L2_BYTES / per_layer))

    def rnd(shape, sigma):
        return (torch.randn(shape, generator=gen, device=dev) * sigma).to(torch.bfloat16)

    ins = [(rnd((M, d), syn.SIGMA), rnd((3 * d, d), d ** -0.5), rnd((3 * d,), syn.SIGMA),
            rnd((R, d), syn.SIGMA), rnd((d, d), d ** -0.5)) for _ in range(layers)]
    outs = [(torch.empty((M, H, 64), dtype=torch.bfloat16, device=dev),
             torch.empty((M, H, 64), dtype=torch.bfloat16, device=dev),
             torch.empty((M, H, 64), dtype=torch.bfloat16, device=dev),
             torch.empty((R, H, 64), dtype=torch.bfloat16, device=dev)) for _ in range(layers)]

    def step():
        for l in range(layers):
            x, wq, bq, pe, wp = ins[l]
            q, k, v, rel = outs[l]
            capi.oasr_project_qkv_pos(x, wq, bq, pe, wp, H, q=q, k=k, v=v, rel=rel)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        t_end = time.perf_counter() + args.soak_seconds
        while time.perf_counter() < t_end:
            graph.replay()
        barrier(world)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    e2e = None
    if not args.no_e2e:
        x_pin = [ins[l][0].cpu().pin_memory() for l in range(layers)]
        o_pin = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs[l]]
                 for l in range(layers)]
        e_ms, hb, db = sequential_e2e(
            stream, [(ins[l][0], x_pin[l]) for l in range(layers)], graph.replay,
            [(o_pin[l][i], outs[l][i]) for l in range(layers) for i in range(4)],
            args.steps, max(3, args.warmup), world)
        e2e = {"value": M * layers * args.steps * world / (e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": hb, "d2h_bytes_per_step": db,
               "path": "per step: pinned host x of every layer -> H2D -> graph replay of the "
                       "oasr_project_qkv_pos calls -> D2H of q, k, v and rel (weights resident)"}
    if rank != 0:
        return
    per_launch_s = ms / 1e3 / (args.steps * layers)
    flops = 2.0 * M * 3 * d * d + 2.0 * R * d * d
    peak, kind = measured_tensor_peak()
    achieved = flops / per_launch_s / 1e12
    line = {
        "metric": METRIC, "value": M * layers * args.steps * world / (ms / 1e3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{name}_qkv_pos", "frames": M, "d_model": d, "H": H, "rel_rows": R,
                   "layers": layers,
                   "l2": f"inputs larger than L2: {layers} distinct layers, {layers * per_layer / 1e6:.0f} MB per step",
                   "timing": "CUDA events around graph replays on the launching stream"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None, "kernel": "project_tc_kernel",
                     "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": per_layer,
                     "achieved_gbs": per_layer / per_launch_s / 1e9,
                     "avg_launch_us": per_launch_s * 1e6, "peak_kind": kind},
        "gpu_launches": args.steps * layers, "clocks": clocks,
    }
    if e2e:
        line["e2e"] = e2e
    if world == 1 and args.cpu_seconds > 0:
        line["cpu_baseline"] = offline_cpu_baseline(name, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def run_packed(args, rank, world, local, window=None):
    """The offline packed row: one call = one attention layer over all utterances
    (window = (chunk, left) for the chunked-limited Nemotron mask)."""
    from paged_kv_chunk_gb300 import build as pkg_build
    from paged_kv_chunk_gb300 import capi
    pkg_build.build()
    capi.load()
    cfg = syn.PACKED
    x = syn.packed_inputs(cfg, cfg.seed + 1000 * rank)
    dev = torch.device("cuda", torch.cuda.current_device())
    d = {k: torch.from_numpy(x[k]).to(torch.bfloat16).to(dev)
         for k in ("q", "k", "v", "pos_bias_u", "pos_bias_v", "rel")}
    cu = torch.from_numpy(x["cu_seqlens"]).to(dev)
    out = torch.empty_like(d["q"])
    total = int(x["cu_seqlens"][-1])

    def call():
        if window:
            capi.oasr_packed_relattn_chunked(d["q"], d["k"], d["v"], cu, x["max_seqlen"],
                                             d["pos_bias_u"], d["pos_bias_v"], d["rel"], window[0],
                                             window[1], out=out)
        else:
            capi.oasr_packed_relattn_varlen(d["q"], d["k"], d["v"], cu, x["max_seqlen"],
                                            d["pos_bias_u"], d["pos_bias_v"], d["rel"], out=out)

    stream = torch.cuda.Stream(device=dev)
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize()
        t_end = time.perf_counter() + args.soak_seconds
        while time.perf_counter() < t_end:
            call()
            stream.synchronize()
        barrier(world)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            call()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    e2e = None
    if not args.no_e2e:
        pins = {k: d[k].cpu().pin_memory() for k in ("q", "k", "v")}
        cu_pin = cu.cpu().pin_memory()
        out_pin = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        e_ms, hb, db = sequential_e2e(
            stream, [(d[k], pins[k]) for k in ("q", "k", "v")] + [(cu, cu_pin)], call,
            [(out_pin, out)], args.steps, max(3, args.warmup), world)
        e2e = {"value": total * args.steps * world / (e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": hb, "d2h_bytes_per_step": db,
               "path": "per call: pinned host q, k, v and cu_seqlens -> H2D -> the packed call -> "
                       "D2H of out (u, v and rel resident)"}
    if rank != 0:
        return
    per_call_s = ms / 1e3 / args.steps
    if window:
        flops = float(chunked_pairs(x["lengths"], *window)) * cfg.H * 6 * cfg.D
    else:
        flops = packed_flops(x["lengths"], cfg.H, cfg.D)
    peak, kind = measured_tensor_peak()
    achieved = flops / per_call_s / 1e12
    if window:
        # a query sees at most (left + 1) chunks of keys: the call is bound by reading q, k, v
        # and the rel table once and writing out, not by its few products
        nbytes = packed_bytes(total, x["rel"].shape[0], cfg.H, cfg.D)
        hpeak, hkind = measured_hbm_peak()
        hach = nbytes / per_call_s / 1e9
        traffic, traffic_src = profiled_traffic("packed_chunked_nemotron_offline", CHUNKED_SOURCES)
        roofline = {"bound": "hbm", "achieved": hach, "peak": hpeak, "unit": "GB/s",
                    "frac": hach / hpeak, "traffic": traffic, "traffic_source": traffic_src,
                    "kernel": "chunk_attn_tc_kernel (packed mode)",
                    "algorithmic_bytes_per_launch": nbytes, "avg_launch_us": per_call_s * 1e6,
                    "peak_kind": hkind,
                    "tensor": {"achieved_tflops": achieved, "peak_tflops": peak,
                               "frac": achieved / peak, "algorithmic_flops_per_launch": flops}}
    else:
        traffic, traffic_src = profiled_traffic("packed_varlen", PACKED_SOURCES)
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak,
                    "traffic": traffic, "traffic_source": traffic_src,
                    "kernel": "packed_attn_tc_kernel", "algorithmic_flops_per_launch": flops,
                    "avg_launch_us": per_call_s * 1e6, "peak_kind": kind}
    line = {
        "metric": METRIC, "value": total * args.steps * world / (ms / 1e3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "nemotron_chunked_offline" if window else "packed_varlen_offline",
                   "num_seqs": cfg.num_seqs,
                   "lengths": f"U{{{cfg.min_len}..{cfg.max_len}}}", "total_frames": total,
                   "H": cfg.H, "D": cfg.D, "rel_rows": int(x["rel"].shape[0]),
                   **({"chunk_frames": window[0], "left_chunks": window[1]} if window else {}),
                   "l2": f"inputs larger than L2: {packed_bytes(total, x['rel'].shape[0], cfg.H, cfg.D) / 1e6:.0f} MB per call"},
        "roofline": roofline,
        "gpu_launches": args.steps, "clocks": clocks,
    }
    if e2e:
        line["e2e"] = e2e
    if world == 1 and args.cpu_seconds > 0:
        line["cpu_baseline"] = offline_cpu_baseline(NEMOTRON if window else syn.PACKED.name,
                                                    args.cpu_seconds)
    print(json.dumps(line), flush=True)


def torchrun_argv(nproc, argv, port):
    """The command that runs this benchmark as `nproc` ranks of one node (one per GPU), with
    the same arguments."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            f"--nproc-per-node={nproc}", "--master-addr", "127.0.0.1", "--master-port", str(port),
            os.path.join(ROOT, "bench.py")] + list(argv)


def free_port():
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def relaunch_ranks(args):
    """`--gpus N` outside a launcher: run N ranks under torch.distributed.run and return its
    exit code (None when this process is already a rank, or N is 1)."""
    if args.gpus <= 1 or "WORLD_SIZE" in os.environ:
        return None
    if torch.cuda.is_available() and torch.cuda.device_count() < args.gpus:
        sys.stderr.write(f"--gpus {args.gpus}: only {torch.cuda.device_count()} GPUs visible\n")
        return 2
    return subprocess.run(torchrun_argv(args.gpus, sys.argv[1:], free_port())).returncode


def main():
    args = parse_args()
    rc = relaunch_ranks(args)
    if rc is not None:
        sys.exit(rc)
    if args.impl == "reference" and (args.config in PROJECTIONS
                                     or args.config in (syn.PACKED.name, NEMOTRON)):
        run_reference_offline(args, args.config, int(os.environ.get("RANK", "0")))
        return
    if args.config in PROJECTIONS:
        rank, world, local = dist_setup()
        run_projection(args, rank, world, local, args.config)
        return
    if args.config in (syn.PACKED.name, NEMOTRON):
        rank, world, local = dist_setup()
        run_packed(args, rank, world, local,
                   window=(NEMOTRON_CHUNK, NEMOTRON_LEFT) if args.config == NEMOTRON else None)
        return
    cfg = syn.STREAMING_CONFIGS[args.config]
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, cfg, rank, int(os.environ.get("WORLD_SIZE", "1")))
        return
    rank, world, local = dist_setup()
    run_ours(args, cfg, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
