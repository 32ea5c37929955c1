#!/usr/bin/env python3
"""Benchmark of the absorbed MLA decode hot path on GB300.

One step = one pass of the whole path (absorb -> paged decode with split
combine -> decompress) over one batch of the workload, as one decoding layer
would run it. The headline workload is the largest of the five: GLM-5.2 dims
causal multi-token decode (H=64, d_nope 192, d_rope 64, d_v 256, kv_rank 512,
bf16, t_q=4, batch 32, seq_lens U[8192, 65536], 16-row blocks, interleaved
rope permuted to NEOX at load). The default run also measures the other four
workloads (tiny f32, GLM-5.2 decode, DeepSeek-V3 geometry, GLM-5.3-Flash
NoPE) the same way and reports them under "per_config".

The KV cache stays resident in HBM (it is the server's state); each layer of
a model has its own cache, so the benchmark cycles through NL distinct layers
(own cache and weights, shared block table) whose total exceeds 4x the L2
size, or one layer when one layer's cache alone does: every step reads its
operands from HBM.

Prints ONE JSON line (rank 0). --impl reference runs the CPU oracle instead,
on a bounded sample of the headline workload, on the host cores.
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
HEADLINE = "glm52_causal_t4"
ALL_CONFIGS = ("tiny_f32", "glm52_decode", "deepseek_decode", "glm53_flash_nope",
               "glm52_causal_t4")
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
def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def oracle_sample(wl, budget_s: float, threads: int):
    """Time the CPU oracle's full path on a bounded sample of the step.

    The absorb and the decompress run on a sample of query rows (all rows
    when few), the decode on a growing random set of (query row, head) pairs
    spread over all requests, until the budget is used; each part's time is
    scaled to the whole step. The oracle runs as it stands: its decode is
    called from `threads` host threads on disjoint pairs (the C code releases
    the GIL), the absorb and the decompress are single calls. Returns
    (tokens/s estimate for the whole step, description, threads, step seconds).
    """
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    from mla_latent_cache_absorbed_gb300 import workloads as W
    g = wl.geom
    H, R, T = g.n_head, g.kv_rank, g.t_q
    lib = oracle.load()
    nr = min(wl.rows, 16)
    t0 = time.perf_counter()
    oracle.absorb_q(wl.q_nope[:nr], wl.q_pe[:nr], wl.w_uk, lib=lib)
    t_abs = (time.perf_counter() - t0) * wl.rows / nr
    # the decode's queries for every row (the sampled decode reads any row):
    # the same absorb, untimed, worked out once per workload
    q4 = getattr(wl, "_oracle_q_abs", None)
    if q4 is None:
        q_abs = oracle.absorb_q(wl.q_nope, wl.q_pe, wl.w_uk, lib=lib)
        q_abs = W.round_to(q_abs, g.dtype) if g.dtype != "f32" else q_abs
        q4 = q_abs.reshape(wl.batch, T, H, -1)
        wl._oracle_q_abs = q4
    total_rows = wl.rows * H
    rng = np.random.default_rng(0)
    order = rng.permutation(total_rows)
    chunk = max(1, min(64, total_rows // max(1, threads)))
    done = 0

    def work(ids):
        oracle.decode_rows(q4, wl.kv_cache, wl.block_table, wl.seq_lens, T, R, wl.scale,
                           ids, lib=lib, allow_errors=True)

    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        while done < total_rows and time.perf_counter() - t0 < budget_s:
            batch = [order[done + i * chunk: done + (i + 1) * chunk] for i in range(threads)]
            batch = [b for b in batch if b.size]
            list(ex.map(work, batch))
            done += sum(b.size for b in batch)
    t_dec = time.perf_counter() - t0
    frac = done / total_rows
    o_in = np.zeros((nr, H, R), np.float32)
    t0 = time.perf_counter()
    oracle.decompress(o_in, wl.w_uv, lib=lib)
    t_dcp = (time.perf_counter() - t0) * wl.rows / nr
    t_step = t_abs + t_dec / frac + t_dcp
    desc = (f"absorb and decompress timed on {nr} of {wl.rows} query rows x {H} heads; "
            f"decode on {done} of {total_rows} (query row, head) pairs ({100 * frac:.2f}%) "
            f"from {threads} host thread(s); each part scaled to the whole step")
    return wl.rows / t_step, desc, threads, t_step


def cpu_baseline(wl, budget_s: float):
    """The oracle on all host cores and on one, each on a bounded sample."""
    threads = os.cpu_count() or 1
    v, desc, threads, _ = oracle_sample(wl, budget_s, threads)
    v1, desc1, _, _ = oracle_sample(wl, max(1.0, budget_s / 3), 1)
    return {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": desc, "cpu_model": cpu_model(),
            "single_thread": {"value": v1, "unit": "tokens/s", "cores": 1, "sample": desc1}}


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    vals = []
    desc = ""
    budget = max(1.0, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
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
        "config": config_dict(wl, world=1, nl=None),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                         "kind": "oracle", "sample": desc, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def layer_count(per_layer_bytes, l2_bytes):
    """Distinct layers the timed loop cycles through: one when a layer's
    operands alone exceed 4x L2, else enough to exceed it together (2..64)."""
    if per_layer_bytes >= 4 * l2_bytes:
        return 1
    return max(2, min(64, math.ceil(4 * l2_bytes / max(1, per_layer_bytes))))


def stage_steps(nl, steps):
    """Steps the per-stage timing replays: whole passes over the nl layers
    (so only the pre-captured full graph runs between the events), at least
    one pass and about as many steps as the timed loop, at most 20 passes."""
    return nl * max(1, min(steps, 20 * nl) // nl)


def config_dict(wl, world, nl):
    g = wl.geom
    if nl is None:
        l2 = "CPU run"
    elif nl * (wl.kv_cache.nbytes + wl.w_uk.nbytes // 2 + wl.w_uv.nbytes // 2) > (1 << 29):
        l2 = ("inputs larger than L2: steps cycle through distinct per-layer caches and "
              "weights totalling > 4x L2")
        if nl == 1:
            l2 = "inputs larger than L2: one layer's cache alone exceeds 4x L2"
    else:
        l2 = "parity-size workload: its working set fits in L2"
    return {"workload": f"{wl.name}: H={g.n_head} d_nope={g.d_nope} d_rope={g.d_rope} "
                        f"d_v={g.d_v} kv_rank={g.kv_rank} t_q={g.t_q} {g.dtype} "
                        f"batch={wl.batch} block=16",
            "batch": wl.batch, "t_q": g.t_q,
            "seq_lens_sum": int(wl.seq_lens.sum()), "seq_lens_max": int(wl.seq_lens.max()),
            "l2": l2,
            "parallelism": f"replicas x{world} (requests shard, no collective)"}


# ---------------------------------------------------------------- GPU leg
def measure_config(args, wl, dev, stream, peaks, peaks_src, world, sample_clocks):
    """Time one workload: the fused step (the headline value), each stage as
    its own call, the decode's roofline fraction and the e2e rate."""
    import torch
    import torch.distributed as dist
    from mla_latent_cache_absorbed_gb300 import device as D

    g = wl.geom
    local = dev.index
    # layers: distinct caches / weights / queries, shared block table
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_layer = (wl.kv_cache.nbytes + wl.w_uk.nbytes // 2 + wl.w_uv.nbytes // 2)
    nl = layer_count(per_layer, l2)
    layers = [D.upload(wl, device=dev) for _ in range(nl)]  # same values, distinct memory
    for c in layers:
        D.attend_workspace(c)  # allocated before any graph capture
    torch.cuda.synchronize()

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

    # every graph a timed region replays is captured before it starts
    g_full = capture(nl)
    graphs = {}

    def prepare(n_steps, which="all"):
        rem = n_steps % nl
        if rem and (which, rem) not in graphs:
            graphs[(which, rem)] = capture(rem, which)

    def replay(graph_full, n_steps, which="all"):
        for _ in range(n_steps // nl):
            graph_full.replay()
        if n_steps % nl:
            graphs[(which, n_steps % nl)].replay()

    # timing probe to choose K when not given
    replay(g_full, nl)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    replay(g_full, 4 * nl)
    torch.cuda.synchronize()
    est = (time.perf_counter() - t0) / (4 * nl)
    steps = args.steps if args.steps else int(min(200000, max(100, 2.0 / max(est, 1e-7))))
    warmup = max(3, args.warmup)

    prepare(warmup)
    prepare(steps)
    replay(g_full, warmup)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(local) if sample_clocks else None
    if sampler:
        sampler.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    replay(g_full, steps)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms_total = ev0.elapsed_time(ev1)
    clocks = sampler.stop() if sampler else None
    if world > 1:
        ms_total = max_over_ranks(ms_total, dev)
        dist.barrier()
    ms_per_step = ms_total / steps
    value = whole_job_rate(wl.rows, world, steps, ms_total)

    # per-stage kernel times (same layers, same launch configuration): whole
    # passes over the layers, all graphs captured before the events
    stage_ms = {}
    n_stage = stage_steps(nl, steps)
    for which in ("absorb", "decode", "decompress"):
        gs = capture(nl, which)
        replay(gs, nl, which)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        replay(gs, n_stage, which)
        e1.record(stream)
        torch.cuda.synchronize()
        stage_ms[which] = e0.elapsed_time(e1) / n_stage
        del gs
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
                       "bound": "tensor" if dec_flops / (tc_peak * 1e12) > dec_bytes / (hbm_peak * 1e9)
                       else "hbm",
                       "bytes": dec_bytes, "flops": dec_flops}
    del g_full
    graphs.clear()

    # end to end through the C ABI with host buffers
    e2e = run_e2e(args, wl, layers, stream, nl, steps)
    res = {"value": value, "unit": "tokens/s", "steps": steps, "warmup": warmup,
           "ms_per_step": ms_per_step, "us_per_layer": ms_per_step * 1e3,
           "dtype": g.dtype, "config": config_dict(wl, world, nl),
           "roofline": roof, "decode_roofline": decode_roofline, "stages_ms": stage_ms,
           "e2e": e2e, "gpu_launches": steps * LAUNCHES_PER_STEP(wl), "layers": nl,
           "clocks": clocks}
    return res, layers


def run_ours(args):
    import torch
    import torch.distributed as dist
    from mla_latent_cache_absorbed_gb300 import _native as N

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    N.load()
    peaks, peaks_src = load_peaks()
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)

    headline = args.config or HEADLINE
    names = [headline] if args.config else [c for c in ALL_CONFIGS if c != headline] + [headline]
    per_config = {}
    head = None
    for name in names:
        wl = make_bench_workload(name, args.batch, rank)
        res, layers = measure_config(args, wl, dev, stream, peaks, peaks_src, world,
                                     sample_clocks=(name == headline))
        if name == headline:
            head = (wl, res, layers)
        else:
            del layers
            torch.cuda.empty_cache()
        per_config[name] = {k: res[k] for k in ("value", "unit", "ms_per_step", "us_per_layer",
                                                "dtype", "decode_roofline", "stages_ms", "e2e",
                                                "layers")}
        per_config[name]["workload"] = res["config"]["workload"]
        per_config[name]["l2"] = res["config"]["l2"]
    wl, res, layers = head
    g = wl.geom

    # the next row of the path: appending new tokens' latent rows to the cache
    cache_append = measure_cache_append(wl, layers[0], stream, peaks["hbm_gbs"])
    # the query half of the prolog (RmsNorm, projections, rope, absorb) for the same rows
    prolog_q = measure_prolog_q(wl, stream, peaks["hbm_gbs"],
                                torch.cuda.get_device_properties(dev).L2_cache_size)

    # CPU baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_budget)

    if rank == 0:
        line = {
            "metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": res["steps"], "warmup": res["warmup"], "ms_per_step": res["ms_per_step"],
            "us_per_layer": res["us_per_layer"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if g.dtype == "bf16" else g.dtype, "data": "synthetic",
            "config": res["config"],
            "roofline": res["roofline"], "decode_roofline": res["decode_roofline"],
            "stages_ms": res["stages_ms"], "e2e": res["e2e"], "cpu_baseline": cpu,
            "gpu_launches": res["gpu_launches"],
            "clocks": res["clocks"], "layers": res["layers"], "cache_append": cache_append,
            "prolog_q": prolog_q,
            "per_config": per_config,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def make_bench_workload(name, batch, rank):
    """The named workload (rank > 0: an independent batch of the same shape);
    with `batch`, only its first `batch` requests (profiling captures)."""
    from mla_latent_cache_absorbed_gb300 import workloads as W
    seed = rank_seed(rank)
    if batch:
        s = W._SEEDS[name] if seed is None else seed
        sl = W.default_seq_lens(name, np.random.default_rng(s))[:batch]
        return W.make_workload(name, seed=seed, seq_lens=sl)
    return W.make_workload(name, seed=seed)


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


def measure_prolog_q(wl, stream, hbm_peak, l2_bytes, q_rank=1536):
    """mla_prolog_q (the query half of the "aclnnMlaProlog" formulas: RmsNorm
    of c_q, W^UQ / W^QR, rope, absorb) for this workload's query rows, on the
    tensor-core path. Distinct weight copies are cycled so that their total
    exceeds 4x L2 (every call streams its weights from HBM); CUDA-graph
    replays timed with events. Algorithmic bytes per call = W^UQ and W^QR
    columns (q_rank x H x (d_nope + d_rope) x 2) + W^UK (H x d_nope x kv_rank
    x 2) + c_q and gamma read + q_abs written + 8 position bytes a row."""
    import torch
    from mla_latent_cache_absorbed_gb300 import _native as N
    from mla_latent_cache_absorbed_gb300 import device as D
    from mla_latent_cache_absorbed_gb300 import workloads as W
    g = wl.geom
    if g.dtype != "bf16":
        return None
    x = W.make_prolog_q(g, wl.rows, q_rank=q_rank)
    dev = torch.device("cuda", torch.cuda.current_device())
    H, Dn, P, R = g.n_head, g.d_nope, g.d_rope, g.kv_rank
    wbytes = (q_rank * H * (Dn + P) + H * Dn * R) * 2
    ncopy = max(1, min(16, math.ceil(4 * l2_bytes / wbytes)))
    t = lambda a: D.host_to_device(a, "bf16", dev)
    copies = [(t(x.w_uq), t(x.w_qr) if P else None, t(x.w_uk)) for _ in range(ncopy)]
    cq, gq = t(x.c_q), t(x.gamma_q)
    pos = torch.from_numpy(x.positions).to(dev)
    q_abs = torch.empty((wl.rows, H, R + P), dtype=torch.bfloat16, device=dev)
    dims = N.MlaDims.from_geometry(g)

    def call(k):
        wuq, wqr, wuk = copies[k % ncopy]
        N.mla_prolog_q(q_abs, cq, gq, wuq, wqr, wuk, pos if P else None, wl.rows, q_rank, x.eps,
                       x.rope_base, dims, None, stream)

    for k in range(ncopy):
        call(k)
    torch.cuda.synchronize()
    reps = ncopy * max(1, 48 // ncopy)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        for k in range(reps):
            call(k)
    gr.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    gr.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / reps
    nbytes = wbytes + wl.rows * q_rank * 2 + q_rank * 2 + wl.rows * H * (R + P) * 2 + wl.rows * 8
    return {"rows": wl.rows, "q_rank": q_rank, "us": us, "bytes": nbytes,
            "achieved_GBps": nbytes / (us * 1e-6) / 1e9,
            "frac_of_hbm": nbytes / (us * 1e-6) / 1e9 / hbm_peak, "weight_copies": ncopy}


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


def spawn_ranks(n):
    """`--gpus N` without a launcher: run this command as N ranks (one per
    GPU) under torch.distributed.run on this node and return its exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr=127.0.0.1",
           f"--master-port={29500 + os.getpid() % 1000}", os.path.abspath(__file__),
           *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1,
                    help="ranks (one per GPU); without a launcher, N > 1 starts them itself")
    ap.add_argument("--steps", type=int, default=0, help="timed steps (default: ~2 s worth)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=None,
                    help=f"one workload only (default: the headline {HEADLINE} plus the "
                         f"other four under per_config)")
    ap.add_argument("--batch", type=int, default=0,
                    help="only the workload's first N requests (smaller profiling cases)")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle decode work in the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    rank, world, _ = dist_env()
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(spawn_ranks(args.gpus))
    if "WORLD_SIZE" in os.environ and args.gpus != world:
        sys.exit(f"--gpus {args.gpus} but the launcher started {world} ranks")
    if args.impl == "reference":
        if args.steps == 0:
            args.steps = 3
        if rank == 0:  # the other ranks exit without work
            run_reference(args, make_bench_workload(args.config or HEADLINE, args.batch, rank))
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
