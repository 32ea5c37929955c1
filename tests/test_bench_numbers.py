"""The bench's roofline numerators and launch counts, on CPU.

The roofline fraction divides algorithmic work by a measured time, so the
work must be what the method needs and no more: every cache row once per
request, the queries, the latent output and the LSE; and QK plus PV flops
over the keys each query row can see (the causal horizon seq_len - t_q + t + 1
of query t). These tests count both by brute force on small workloads.
"""
import numpy as np
import pytest

import bench
from mla_latent_cache_absorbed_gb300 import workloads as W


def brute_force(wl):
    g = wl.geom
    e = 2 if g.dtype == "bf16" else 4
    H, R, Wd, T = g.n_head, g.kv_rank, g.width, g.t_q
    cache = sum(int(s) for s in wl.seq_lens) * Wd * e
    visible = 0
    for s in wl.seq_lens:
        for t in range(T):
            if s > 0:
                visible += int(s) - T + t + 1            # keys 0 .. s - T + t
    rows = wl.batch * T
    dec_bytes = cache + rows * H * (Wd * e + R * e + 4)
    dec_flops = 2 * H * visible * (Wd + R)              # QK over Wd, PV over R
    return dec_bytes, dec_flops


@pytest.mark.parametrize("name,t_q,lens", [
    ("tiny_f32", 1, [37, 64]),
    ("glm52_decode", 1, [5, 0, 40]),
    ("glm52_decode", 4, [4, 9, 100]),
    ("glm52_decode", 16, [16, 17, 0]),
    ("glm53_flash_nope", 2, [2, 33]),
])
def test_decode_work_matches_brute_force(name, t_q, lens):
    g = W.geometry(name)
    geom = W.Geometry(g.n_head, g.d_nope, g.d_rope, g.d_v, g.kv_rank, t_q, g.dtype)
    wl = W.make_workload(name, seq_lens=lens, geom=geom)
    alg = bench.algorithmic(wl)
    assert alg["decode"] == brute_force(wl)
    e = 2 if g.dtype == "bf16" else 4
    rows = wl.batch * t_q
    H, R, Dn, Dv, P = g.n_head, g.kv_rank, g.d_nope, g.d_v, g.d_rope
    assert alg["absorb"] == (H * Dn * R * e + rows * H * (Dn + P) * e + rows * H * (R + P) * e,
                             2 * rows * H * Dn * R)
    assert alg["decompress"] == (H * Dv * R * e + rows * H * R * e + rows * H * Dv * e,
                                 2 * rows * H * R * Dv)


def test_first_chunk_flops_are_triangular():
    """A first prefill chunk (t_q == seq_len = n) sees 1 + 2 + ... + n keys."""
    n = 48
    g = W.geometry("glm52_decode")
    geom = W.Geometry(g.n_head, g.d_nope, g.d_rope, g.d_v, g.kv_rank, n, g.dtype)
    wl = W.make_workload("glm52_decode", seq_lens=[n], geom=geom)
    _, flops = bench.algorithmic(wl)["decode"]
    assert flops == 2 * g.n_head * (n * (n + 1) // 2) * (g.width + g.kv_rank)


def test_launches_per_step():
    """Three kernels per fused bf16 step (absorb, decode, merging decompress)
    up to 256 query rows per request; the combine is a fourth otherwise, and
    on the f32 path."""
    assert bench.LAUNCHES_PER_STEP(W.make_workload("glm52_decode", seq_lens=[5])) == 3
    assert bench.LAUNCHES_PER_STEP(W.make_workload("glm52_causal_t4", seq_lens=[5])) == 3
    assert bench.LAUNCHES_PER_STEP(W.make_workload("glm52_prefill_chunk")) == 4
    assert bench.LAUNCHES_PER_STEP(W.make_workload("tiny_f32")) == 4


def test_named_workload_work():
    """The bench's numbers for every named workload are the brute-force
    counts: the small ones at full size, the large ones on their first three
    requests (the recipe's lengths, seeded)."""
    large = ("deepseek_decode", "glm52_causal_t4", "glm53_flash_nope")
    for name in W.NAMES:
        lens = None if name not in large else \
            W.default_seq_lens(name, np.random.default_rng(0))[:3]
        wl = W.make_workload(name, seq_lens=lens)
        assert bench.algorithmic(wl)["decode"] == brute_force(wl), name


def test_stage_timing_replays_whole_passes():
    """The per-stage timing replays only the full-pass graph captured before
    its events: its step count is a whole number of passes over the layers."""
    for nl in (1, 2, 3, 12, 64):
        for steps in (1, 5, 8, 20, 100, 1000):
            n = bench.stage_steps(nl, steps)
            assert n % nl == 0 and n >= nl and n <= 20 * nl


def test_layer_count():
    """One layer when its operands alone exceed 4x L2; otherwise enough
    distinct layers to exceed it together (at least two, at most 64)."""
    l2 = 129 << 20
    assert bench.layer_count(4 * l2, l2) == 1
    assert bench.layer_count(10 * l2, l2) == 1
    assert bench.layer_count(l2, l2) == 4
    assert bench.layer_count(3 * l2, l2) == 2
    assert bench.layer_count(1, l2) == 64
    for per in (1 << 20, 20 << 20, 300 << 20):
        n = bench.layer_count(per, l2)
        assert n * per >= 4 * l2 or n == 64


def test_default_run_covers_every_workload_with_the_largest_as_headline():
    assert set(bench.ALL_CONFIGS) == {"tiny_f32", "glm52_decode", "deepseek_decode",
                                      "glm53_flash_nope", "glm52_causal_t4"}
    sizes = {}
    for name in bench.ALL_CONFIGS:
        lens = W.default_seq_lens(name, np.random.default_rng(W._SEEDS[name]))
        g = W.geometry(name)
        sizes[name] = int(lens.sum()) * g.width * (2 if g.dtype == "bf16" else 4)
    assert bench.HEADLINE == max(sizes, key=sizes.get)


def _kernel_tree(tmp_path, extra=""):
    """A copy of the pair decode kernel's sources under tmp_path (as bench.py
    finds them below its root), with `extra` appended to tc_decode.cu."""
    import os
    import shutil
    src = os.path.join(bench.ROOT, "mla_latent_cache_absorbed_gb300", "csrc")
    dst = tmp_path / "mla_latent_cache_absorbed_gb300" / "csrc"
    dst.mkdir(parents=True)
    for name in ("tc_decode.cu", "tc_split.cuh", "sm100.cuh"):
        shutil.copy(os.path.join(src, name), dst / name)
    with open(dst / "tc_decode.cu", "a") as f:
        f.write(extra)
    (tmp_path / "profiles").mkdir()
    return tmp_path


def test_fingerprint_ignores_comments_not_code(tmp_path, monkeypatch):
    """The decode kernel's fingerprint keys the committed ncu traffic: a
    comment or blank-line edit keeps it, a code edit changes it."""
    base = bench.kernel_fingerprint()
    monkeypatch.setattr(bench, "ROOT", str(_kernel_tree(tmp_path / "a", "\n// a comment\n\n")))
    assert bench.kernel_fingerprint() == base
    monkeypatch.setattr(bench, "ROOT", str(_kernel_tree(tmp_path / "b", "\nstatic int k_x;\n")))
    assert bench.kernel_fingerprint() != base


def test_profiled_traffic_only_for_the_captured_kernel(tmp_path, monkeypatch):
    """traffic is the summary's DRAM bytes while its recorded fingerprint is
    the kernel's own, and null once the kernel has changed."""
    root = _kernel_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    fp = bench.kernel_fingerprint()
    prof = root / "profiles" / "decode_pair_some_workload.md"
    prof.write_text(f"traffic_bytes_per_launch: 123456\nkernel_fingerprint: {fp[:12]}\n")
    assert bench.profiled_traffic("some_workload") == 123456
    prof.write_text("traffic_bytes_per_launch: 123456\nkernel_fingerprint: 000000000000\n")
    assert bench.profiled_traffic("some_workload") is None
    assert bench.profiled_traffic("no_such_workload") is None
