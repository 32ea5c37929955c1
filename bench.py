#!/usr/bin/env python3
"""Benchmark of the absorbed MLA decode hot path on GB300.

One step = one pass of the whole path (absorb -> paged decode with split
combine -> decompress) over one batch of the workload, as one decoding layer
would run it. Default workload: GLM-5.2 dims decode (H=64, d_nope 192, d_rope
64, d_v 256, kv_rank 512, bf16, batch 8, seq_lens U[1,4096] with one empty
request, 16-row blocks). The KV cache stays resident in HBM (it is the
server's state); each layer of a model has its own cache, so the benchmark
cycles through NL distinct layers (own cache and weights, shared block table)
whose total exceeds 4x the L2 size: every step reads its operands from HBM.

Prints ONE JSON line (rank 0). --impl reference runs the CPU oracle instead,
on a bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode tokens/s/GPU & µs/layer; % of max(HBM, bf16-tensor) roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_fingerprint():
    """sha1 of the pair decode kernel's code: tc_decode.cu and the headers it
    includes, with comments, blank lines and indentation dropped (a comment
    edit does not change the kernel)."""
    import hashlib
    h = hashlib.sha1()
    for name in ("tc_decode.cu", "tc_split.cuh", "sm100.cuh"):
        path = os.path.join(ROOT, "mla_latent_cache_absorbed_gb300", "csrc", name)
        if not os.path.exists(path):
            return None
        for line in open(path):
            code = line.split("//", 1)[0].strip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()


def profiled_traffic(config_name):
    """DRAM bytes (read + write) per launch of the pair decode kernel from the
    committed ncu summary of this workload, or None when there is none or the
    kernel has changed since it was captured (the summary records the
    kernel_fingerprint() it was taken on)."""
    prof = os.path.join(ROOT, "profiles", f"decode_pair_{config_name}.md")
    if not os.path.exists(prof):
        return None
    text = open(prof).read()
    m_t = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    m_h = re.search(r"kernel_fingerprint:\s*([0-9a-f]+)", text)
    fp = kernel_fingerprint()
    if not (m_t and m_h and fp) or not fp.startswith(m_h.group(1)):
        return None
    return int(m_t.group(1))


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(rank):
    """Workload seed of a rank: rank 0 runs the named workload itself, every
    other rank an independent batch of the same shape (weak scaling: requests
    shard across GPUs, nothing is exchanged)."""
    return None if rank == 0 else 1000 + rank


def max_over_ranks(ms, device):
    """The slowest rank's time (the job ends when the last rank ends)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(rows_per_rank, world, steps, ms_total):
    """Decode tokens per second of the whole job: every rank decodes its own
    rows_per_rank query rows per step."""
    return rows_per_rank * world * steps / (ms_total / 1e3)


# ---------------------------------------------------------------- workload facts
def algorithmic(wl):
    """Algorithmic bytes and flops of one step (per unit definitions).

    decode bytes = cache rows read once per request (sum S_b * W * e)
                 + q_abs (B*T*H*W*e) + o_lat (B*T*H*R*e) + lse (B*T*H*4)
    decode flops = 2 * H * sum over query rows of visible keys * (W + R)
    absorb bytes = w_uk + q_nope + q_pe + q_abs;  flops 2*B*T*H*Dn*R
    decompress   = w_uv + o_lat + out;             flops 2*B*T*H*R*Dv
    """
    g = wl.geom
    e = 2 if g.dtype == "bf16" else 4
    H, R, W, T, Dn, Dv, P = g.n_head, g.kv_rank, g.width, g.t_q, g.d_nope, g.d_v, g.d_rope
    S = wl.seq_lens.astype(np.int64)
    rows = wl.rows
    cache = int(S.sum()) * W * e
    dec_bytes = cache + rows * H * W * e + rows * H * R * e + rows * H * 4
    vis = 0
    for s in S:
        if s > 0:
            vis += sum(int(s) - T + t + 1 for t in range(T))
    dec_flops = 2 * H * vis * (W + R)
    abs_bytes = H * Dn * R * e + rows * H * (Dn + P) * e + rows * H * W * e
    abs_flops = 2 * rows * H * Dn * R
    dcp_bytes = H * Dv * R * e + rows * H * R * e + rows * H * Dv * e
    dcp_flops = 2 * rows * H * R * Dv
    return {"decode": (dec_bytes, dec_flops), "absorb": (abs_bytes, abs_flops),
            "decompress": (dcp_bytes, dcp_flops), "cache_bytes": cache}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
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
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.25)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        self.proc.wait(timeout=5)
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------- oracle (CPU) leg
def oracle_sample(wl, budget_s: float, threads: int):
    """Time the CPU oracle's full path on a bounded sample of query rows.

    The absorb and decompress run on every row; the decode on a growing set
    of query rows (spread over all requests and heads) until the budget is
    used. Returns (tokens/s estimate for the whole step, description, threads).
    """
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    from mla_latent_cache_absorbed_gb300 import workloads as W
    g = wl.geom
    H, R, T = g.n_head, g.kv_rank, g.t_q
    lib = oracle.load()
    t0 = time.perf_counter()
    q_abs = oracle.absorb_q(wl.q_nope, wl.q_pe, wl.w_uk, lib=lib)
    t_abs = time.perf_counter() - t0
    q_abs = W.round_bf16(q_abs) if g.dtype == "bf16" else q_abs
    q4 = q_abs.reshape(wl.batch, T, H, -1)
    total_rows = wl.rows * H
    rng = np.random.default_rng(0)
    order = rng.permutation(total_rows)
    chunk = max(1, min(64, total_rows // max(1, threads)))
    done = 0
    t0 = time.perf_counter()

    def work(ids):
        oracle.decode_rows(q4, wl.kv_cache, wl.block_table, wl.seq_lens, T, R, wl.scale,
                           ids, lib=lib, allow_errors=True)

    with ThreadPoolExecutor(threads) as ex:
        while done < total_rows and time.perf_counter() - t0 < budget_s:
            batch = [order[done + i * chunk: done + (i + 1) * chunk] for i in range(threads)]
            batch = [b for b in batch if b.size]
            list(ex.map(work, batch))
            done += sum(b.size for b in batch)
    t_dec = time.perf_counter() - t0
    frac = done / total_rows
    o_in = np.zeros((wl.rows, H, R), np.float32)
    t0 = time.perf_counter()
    oracle.decompress(o_in, wl.w_uv, lib=lib)
    t_dcp = time.perf_counter() - t0
    t_step = t_abs + t_dec / frac + t_dcp
    desc = (f"absorb and decompress on all {wl.rows} query rows x {H} heads; decode on "
            f"{done} of {total_rows} (query row, head) pairs ({100 * frac:.2f}%), "
            f"extrapolated to the whole step")
    return wl.rows / t_step, desc, threads, t_step


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    vals = []
    desc = ""
    budget = max(2.0, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup + args.steps):
        v, desc, threads, t_step = oracle_sample(wl, budget, threads)
        if i >= args.warmup:
            vals.append(t_step)
    t = statistics.mean(vals)
    value = wl.rows / t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_dict(wl, world=1),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def config_dict(wl, world):
    g = wl.geom
    return {"workload": f"{wl.name}: H={g.n_head} d_nope={g.d_nope} d_rope={g.d_rope} "
                        f"d_v={g.d_v} kv_rank={g.kv_rank} t_q={g.t_q} {g.dtype} "
                        f"batch={wl.batch} block=16",
            "batch": wl.batch, "t_q": g.t_q,
            "seq_lens_sum": int(wl.seq_lens.sum()), "seq_lens_max": int(wl.seq_lens.max()),
            "l2": "inputs larger than L2: steps cycle through distinct per-layer caches and "
                  "weights totalling > 4x L2",
            "parallelism": f"replicas x{world} (requests shard, no collective)"}


# ---------------------------------------------------------------- GPU leg
def run_ours(args, wl):
    import torch
    import torch.distributed as dist
    from mla_latent_cache_absorbed_gb300 import _native as N
    from mla_latent_cache_absorbed_gb300 import device as D
    from mla_latent_cache_absorbed_gb300 import workloads as W

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    N.load()
    g = wl.geom
    peaks, peaks_src = load_peaks()

    # layers: distinct caches / weights / queries, shared block table
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_layer = (wl.kv_cache.nbytes + wl.w_uk.nbytes // 2 + wl.w_uv.nbytes // 2)
    nl = max(2, min(64, math.ceil(4 * l2 / max(1, per_layer))))
    base = D.upload(wl, device=dev)
    layers = [base]
    for i in range(1, nl):
        c = D.upload(wl, device=dev)  # same values, distinct memory
        layers.append(c)
    for c in layers:
        D.attend_workspace(c)  # allocated before any graph capture
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)

    def step(k, which="all"):
        # the step is the fused call a decode step makes; the stage timings
        # below run each stage as its own call
        c = layers[k % nl]
        if which == "all":
            D.attend(c, stream)
        elif which == "absorb":
            D.absorb(c, stream)
        elif which == "decode":
            D.decode(c, stream)
        elif which == "decompress":
            D.decompress(c, stream)

    # eager warm-up (one-time setup of the library happens outside capture)
    for k in range(max(3, args.warmup)):
        step(k)
    torch.cuda.synchronize()

    def capture(n, which="all"):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for k in range(n):
                step(k, which)
        return gr

    g_full = capture(nl)

    def replay(graph_full, n_steps, graph_rem_cache):
        full, rem = divmod(n_steps, nl)
        for _ in range(full):
            graph_full.replay()
        if rem:
            if rem not in graph_rem_cache:
                graph_rem_cache[rem] = capture(rem, graph_rem_cache["which"])
            graph_rem_cache[rem].replay()

    rem_all = {"which": "all"}
    # timing probe to choose K when not given
    replay(g_full, nl, rem_all)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    replay(g_full, 4 * nl, rem_all)
    torch.cuda.synchronize()
    est = (time.perf_counter() - t0) / (4 * nl)
    steps = args.steps if args.steps else int(min(200000, max(100, 2.0 / max(est, 1e-7))))
    warmup = max(3, args.warmup)

    replay(g_full, warmup, rem_all)
    if steps % nl and (steps % nl) not in rem_all:
        rem_all[steps % nl] = capture(steps % nl)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(local)
    sampler.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    replay(g_full, steps, rem_all)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms_total = ev0.elapsed_time(ev1)
    clocks = sampler.stop()
    if world > 1:
        ms_total = max_over_ranks(ms_total, dev)
        dist.barrier()
    ms_per_step = ms_total / steps
    value = whole_job_rate(wl.rows, world, steps, ms_total)

    # per-stage kernel times (same layers, same launch configuration)
    stage_ms = {}
    for which in ("absorb", "decode", "decompress"):
        gs = capture(nl, which)
        rem = {"which": which}
        n = max(nl, min(steps, 20 * nl))
        replay(gs, nl, rem)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        replay(gs, n, rem)
        e1.record(stream)
        torch.cuda.synchronize()
        stage_ms[which] = e0.elapsed_time(e1) / n
    alg = algorithmic(wl)
    dominant = max(stage_ms, key=stage_ms.get)
    dom_bytes, dom_flops = alg[dominant]
    dom_s = stage_ms[dominant] / 1e3
    hbm_peak = peaks["hbm_gbs"]
    tc_peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    t_hbm = dom_bytes / (hbm_peak * 1e9)
    t_tc = dom_flops / (tc_peak * 1e12)
    if t_tc > t_hbm:
        roof = {"bound": "tensor", "achieved": dom_flops / dom_s / 1e12, "peak": tc_peak,
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": dom_bytes / dom_s / 1e9, "peak": hbm_peak,
                "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = profiled_traffic(wl.name) if dominant == "decode" else None
    roof["kernel"] = dominant
    if dominant == "decode":
        # the decode stage is the pair kernel plus the split combine; the
        # committed ncu traffic is the pair kernel's (the combine re-reads the
        # partials the pair kernel wrote, from L2)
        roof["traffic_kernel"] = "decode_pair_kernel"
    roof["peak_source"] = f"{peaks_src} (MEASURED_PEAKS.json)" if peaks_src == "measured" \
        else "fallback (profiling recipe)"
    dec_bytes, dec_flops = alg["decode"]
    dec_s = stage_ms["decode"] / 1e3
    t_roof = max(dec_bytes / (hbm_peak * 1e9), dec_flops / (tc_peak * 1e12))
    decode_roofline = {"us_per_layer": stage_ms["decode"] * 1e3,
                       "roofline_us": t_roof * 1e6, "frac": t_roof / dec_s,
                       "bytes": dec_bytes, "flops": dec_flops}

    # the next row of the path: appending new tokens' latent rows to the cache
    cache_append = measure_cache_append(wl, base, stream, hbm_peak)

    # end to end through the C ABI with host buffers
    e2e = run_e2e(args, wl, layers, stream, nl, steps)

    # CPU baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc, threads, _ = oracle_sample(wl, args.cpu_budget, os.cpu_count() or 1)
        cpu = {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": desc}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": steps, "warmup": warmup, "ms_per_step": ms_per_step,
            "us_per_layer": ms_per_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if g.dtype == "bf16" else "f32", "data": "synthetic",
            "config": config_dict(wl, world),
            "roofline": roof, "decode_roofline": decode_roofline,
            "stages_ms": stage_ms, "e2e": e2e, "cpu_baseline": cpu,
            "gpu_launches": steps * LAUNCHES_PER_STEP(wl),
            "clocks": clocks, "layers": nl, "cache_append": cache_append,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def measure_cache_append(wl, dc, stream, hbm_peak):
    """mla_cache_append (the page's do_kv_cache_update) on this workload's
    cache: one new token per query row (the decode step's append) and a
    32768-token chunk (a prefill chunk), bf16 rows into the bf16 cache, unique
    random slots. CUDA-graph replays timed with events; algorithmic bytes =
    tokens x (W x 2 read + W x 2 written + 8 slot bytes). The same two
    launches of mla_cache_append_rmsnorm_rope (RmsNorm of the latent and rope
    of k_pe fused in, "aclnnMlaProlog" key formulas) add 8 position bytes a
    token and the R x 2 bytes of gamma once; their positions are the decode
    rows' own (seq_len - t_q + t) and 0 .. n-1 for the chunk."""
    import torch
    from mla_latent_cache_absorbed_gb300 import _native as N
    g = wl.geom
    if g.dtype != "bf16":
        return None
    W, R, P = g.width, g.kv_rank, g.d_rope
    dev = dc.kv_cache.device
    num_slots = dc.num_blocks * 16
    res = {}
    rng = np.random.default_rng(99)
    # a scratch cache of the same geometry: the measured caches stay intact
    cache = torch.empty((dc.num_blocks, 16, W), dtype=torch.bfloat16, device=dev)
    gamma = (torch.rand(R, device=dev) + 0.5).to(torch.bfloat16)
    cases = [(lab + sfx, n, fused) for fused, sfx in ((False, ""), (True, "_rmsnorm_rope"))
             for lab, n in (("decode_step", wl.rows), ("chunk_32k", 32768))]
    for label, n, fused in cases:
        n = min(n, num_slots)
        kv_c = torch.randn(n, R, device=dev).to(torch.bfloat16)
        k_pe = torch.randn(n, max(P, 1), device=dev).to(torch.bfloat16)
        slots = torch.from_numpy(rng.choice(num_slots, size=n, replace=False).astype(np.int64)).to(dev)
        if n == wl.rows:   # the decode step: each query row's own position in its request
            T = g.t_q
            pos = np.repeat(np.asarray(wl.seq_lens, np.int64), T) - T + np.tile(np.arange(T), wl.batch)
        else:              # a prefill chunk: consecutive positions
            pos = np.arange(n)
        positions = torch.from_numpy(np.maximum(pos, 0).astype(np.int64)).to(dev)
        reps = 200 if n < 4096 else 20

        def call():
            if fused:
                N.mla_cache_append_rmsnorm_rope(cache, kv_c, k_pe if P else None, gamma,
                                                positions if P else None, slots, n,
                                                dc.num_blocks, 1, 1e-6, 10000.0, dc.dims, None,
                                                stream)
            else:
                N.mla_cache_append(cache, kv_c, k_pe if P else None, slots, n, dc.num_blocks, 1,
                                   dc.dims, None, stream)

        call()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for _ in range(reps):
                call()
        gr.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gr.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        nbytes = n * (W * 2 * 2 + 8) + ((n * 8 if P else 0) + R * 2 if fused else 0)
        res[label] = {"tokens": n, "us": us, "bytes": nbytes,
                      "achieved_GBps": nbytes / (us * 1e-6) / 1e9,
                      "frac_of_hbm": nbytes / (us * 1e-6) / 1e9 / hbm_peak}
    return res


def LAUNCHES_PER_STEP(wl):
    """Kernels of this library launched per fused step: absorb, decode and the
    decompress that merges the split rows (bf16, up to 256 query rows per
    request); the f32 path and larger query blocks (prefill chunks) run the
    decode's combine as a fourth kernel."""
    g = wl.geom
    return 3 if g.dtype == "bf16" and g.t_q * g.n_head <= 256 else 4


def run_e2e(args, wl, layers, stream, nl, steps):
    """Same metric through the C ABI with the step's inputs in pinned host
    memory. Per step: one copy in of the step's q_nope, q_pe, block_table and
    seq_lens (packed in one pinned buffer, 256-byte aligned sections), the
    fused call, and one copy out of the output rows; the cache is resident
    server state. Copies run on their own stream, so step k's copies overlap
    the neighbouring steps' kernels (each layer's buffers are reused only
    after the step that last read them has finished). As a serving loop
    would, at least 16 steps (whole passes over the layers) are captured once
    in a CUDA graph (copies included) and replayed."""
    import torch
    from mla_latent_cache_absorbed_gb300 import device as D
    g = wl.geom
    tdt = torch.bfloat16 if g.dtype == "bf16" else torch.float32
    parts = [torch.from_numpy(wl.q_nope).to(tdt), torch.from_numpy(wl.q_pe).to(tdt),
             torch.from_numpy(wl.block_table), torch.from_numpy(wl.seq_lens)]
    offs, size = [], 0
    for t in parts:
        offs.append(size)
        size += (t.numel() * t.element_size() + 255) // 256 * 256
    hbuf = torch.empty(size, dtype=torch.uint8).pin_memory()
    for t, o in zip(parts, offs):
        hbuf[o:o + t.numel() * t.element_size()].copy_(t.contiguous().view(-1).view(torch.uint8))
    # each layer's inputs become views into one device buffer of that layout
    dbufs = []
    for c in layers:
        db = torch.empty(size, dtype=torch.uint8, device=c.out.device)
        views = []
        for t, o in zip(parts, offs):
            nb = t.numel() * t.element_size()
            views.append(db[o:o + nb].view(t.dtype).view(t.shape))
        c.q_nope, c.q_pe, c.block_table, c.seq_lens = views
        dbufs.append(db)
    hout = torch.empty(tuple(layers[0].out.shape), dtype=tdt).pin_memory()
    cs = torch.cuda.Stream(device=layers[0].out.device)
    n = max(10, min(steps, 2000))

    def run(count):
        last = [None] * nl      # the event after each layer's latest call
        prev = None             # (layer, its call's event): output not yet copied out
        fork = torch.cuda.Event()
        fork.record(stream)
        cs.wait_event(fork)     # the copy stream joins the calling stream's work
        for k in range(count):
            i = k % nl
            c = layers[i]
            with torch.cuda.stream(cs):
                if last[i] is not None:
                    cs.wait_event(last[i])
                dbufs[i].copy_(hbuf, non_blocking=True)
                h2d = torch.cuda.Event()
                h2d.record(cs)
            stream.wait_event(h2d)
            D.attend(c, stream)
            ev = torch.cuda.Event()
            ev.record(stream)
            last[i] = ev
            if prev is not None:
                with torch.cuda.stream(cs):
                    cs.wait_event(prev[1])
                    hout.copy_(prev[0].out, non_blocking=True)
            prev = (c, ev)
        with torch.cuda.stream(cs):
            cs.wait_event(prev[1])
            hout.copy_(prev[0].out, non_blocking=True)
            join = torch.cuda.Event()
            join.record(cs)
        stream.wait_event(join)  # and finishes before the calling stream goes on

    run(3)
    torch.cuda.synchronize()
    per_graph = nl * -(-16 // nl)  # whole passes over the layers, >= 16 steps
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        run(per_graph)
    reps = max(2, -(-n // per_graph))
    n = reps * per_graph
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    h2d_bytes = sum(t.numel() * t.element_size() for t in parts)
    d2h = hout.numel() * hout.element_size()
    return {"value": wl.rows * n / (ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d_bytes), "d2h_bytes_per_step": int(d2h),
            "steps": n, "ms_per_step": ms / n,
            "copies": "one packed copy in and one copy out per step, on their own "
                      "stream, overlapping the neighbouring steps' kernels; >= 16 steps "
                      "form one captured CUDA graph"}


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (default: ~2 s worth)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="glm52_decode")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle decode work in the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    from mla_latent_cache_absorbed_gb300 import workloads as W
    rank, world, _ = dist_env()
    wl = W.make_workload(args.config, seed=rank_seed(rank))
    if args.impl == "reference":
        if args.steps == 0:
            args.steps = 3
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
