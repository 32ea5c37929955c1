"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Tolerances (the parity gates, tests/tolerances.py):
  f32 inputs   every output and LSE: max abs diff <= 1e-4
  bf16 inputs  outputs: |gpu - ref| <= 1e-2 + half a bf16 ulp of |ref| (the
               stated bound plus one rounding of the stored output); LSE (f32):
               max abs diff <= 1e-3; a -inf LSE must be -inf on both sides.
  f16 inputs   outputs: <= 2e-3 + half an f16 ulp of |ref| (the bf16 gate
               scaled by f16's finer quantum); LSE as for bf16.
The oracle runs on the same (bf16-rounded) values the GPU stage consumed: each
stage's input comes from the generator or from the oracle's previous stage,
never from the GPU.
"""
import numpy as np
import pytest

import oracle
from mla_latent_cache_absorbed_gb300 import _native as N
from mla_latent_cache_absorbed_gb300 import device as D
from mla_latent_cache_absorbed_gb300 import workloads as W
from tolerances import lse_bound, output_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    assert torch.cuda.is_available()
    N.load()


def assert_close(got, ref, dtype, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite GPU output"
    err = np.abs(got - ref)
    bound = output_bound(ref, dtype)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance, max err "
                             f"{err.max():.3e}; worst at {i}: ref {ref[i]:.6f} gpu {got[i]:.6f} "
                             f"bound {bound[i]:.3e}")


def assert_lse_close(got, ref, dtype, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    ninf_g, ninf_r = np.isneginf(got), np.isneginf(ref)
    assert np.array_equal(ninf_g, ninf_r), f"{what}: -inf rows differ"
    tol = lse_bound(dtype)
    err = np.abs(got[~ninf_r] - ref[~ninf_r])
    assert err.size == 0 or err.max() <= tol, f"{what}: max err {err.max():.3e}"


def rounded(x, dtype):
    return W.round_to(x, dtype)


def gpu_sides(wl):
    """(gpu cache, gpu q_pe): the workload's own, or, for interleaved-rope
    workloads, the permuted-NEOX copy built with the library's host
    permutation (what a loader does at load time)."""
    if wl.rope != "norm":
        return None, None
    P = wl.geom.d_rope
    k, q = W.neox_side_rope_columns(wl, lambda a: N.mla_permute_rope_cols(a, 0, P))
    return W.cache_with_rope_columns(wl, k), q


def run_stages(wl, rows=None):
    """Per-stage parity (absorb, decode, decompress) and the chained path.

    rows: None compares every query row of the decode; otherwise a list of
    flattened (b*t_q + t)*H + h ids whose decode the oracle computes alone.
    """
    import torch
    g = wl.geom
    dt = g.dtype
    H, R, T = g.n_head, g.kv_rank, g.t_q
    cache_gpu, q_pe_gpu = gpu_sides(wl)
    dc = D.upload(wl, kv_cache=cache_gpu, q_pe=q_pe_gpu)

    # --- absorb: oracle on the same inputs
    D.absorb(dc)
    torch.cuda.synchronize()
    q_abs_gpu = D.device_to_host_f32(dc.q_abs)
    q_abs_ref = oracle.absorb_q(wl.q_nope, wl.q_pe if q_pe_gpu is None else q_pe_gpu, wl.w_uk)
    assert_close(q_abs_gpu, q_abs_ref, dt, "absorb")

    # --- decode: both consume the oracle's absorb output, rounded to the dtype
    q_abs_oracle = (q_abs_ref if q_pe_gpu is None    # else the oracle's own rope layout
                    else oracle.absorb_q(wl.q_nope, wl.q_pe, wl.w_uk))
    q_in_ref = rounded(q_abs_oracle, dt)
    q_in_gpu = rounded(q_abs_ref, dt)
    dc.q_abs.copy_(D.host_to_device(q_in_gpu, dt, "cuda"))
    D.decode(dc)
    torch.cuda.synchronize()
    assert int(dc.dev_err.item()) == 0
    o_gpu = D.device_to_host_f32(dc.o_lat)
    lse_gpu = dc.lse.cpu().numpy()
    q4 = q_in_ref.reshape(wl.batch, T, H, -1)
    if rows is None:
        o_ref, lse_ref = oracle.decode_paged(q4, wl.kv_cache, wl.block_table, wl.seq_lens, T,
                                             R, wl.scale)
        o_ref = o_ref.reshape(-1, H, R)
        lse_ref = lse_ref.reshape(-1, H)
        assert_close(o_gpu, o_ref, dt, "decode out")
        assert_lse_close(lse_gpu, lse_ref, dt, "decode lse")
    else:
        ids = np.asarray(rows, np.int64)
        o_ref, lse_ref = oracle.decode_rows(q4, wl.kv_cache, wl.block_table, wl.seq_lens, T, R,
                                            wl.scale, ids)
        assert_close(o_gpu.reshape(-1, R)[ids], o_ref, dt, "decode out (sampled)")
        assert_lse_close(lse_gpu.reshape(-1)[ids], lse_ref, dt, "decode lse (sampled)")
        o_ref = None

    # --- decompress: both consume the same latent rows
    rng = np.random.default_rng(123)
    o_in = (o_ref if o_ref is not None else
            rng.standard_normal((wl.rows, H, R)).astype(np.float32) * 0.1)
    o_in = rounded(o_in, dt)
    dc.o_lat.copy_(D.host_to_device(o_in, dt, "cuda"))
    D.decompress(dc)
    torch.cuda.synchronize()
    dcp_ref = oracle.decompress(o_in, wl.w_uv)
    assert_close(D.device_to_host_f32(dc.out), dcp_ref, dt, "decompress")

    # --- the chained path, the oracle rounding at the same points
    D.full_step(dc)
    torch.cuda.synchronize()
    assert int(dc.dev_err.item()) == 0
    if rows is None:
        # the chain's decode input is q4 again and its decompress input the
        # rounded o_ref: the oracle results of the stage checks above are
        # the chain's
        assert_close(D.device_to_host_f32(dc.out), dcp_ref, dt, "full path out")
        assert_lse_close(dc.lse.cpu().numpy(), lse_ref, dt, "full path lse")
    return dc


def test_tiny_f32_full_path():
    wl = W.make_workload("tiny_f32")
    run_stages(wl)


def test_tiny_f32_nan_poison():
    wl = W.make_workload("tiny_f32", poison="nan")
    run_stages(wl)


def test_glm52_decode_full_size():
    run_stages(W.make_workload("glm52_decode"))


REDUCED = {
    "deepseek_decode": [8192, 1, 100, 16, 0, 2049],
    "glm53_flash_nope": [2048, 7, 0, 129, 31, 32768],
    "glm52_causal_t4": [4, 5, 100, 1000, 0, 4096],
}


@pytest.mark.parametrize("name", sorted(REDUCED))
def test_reduced_all_rows(name):
    run_stages(W.make_workload(name, seq_lens=REDUCED[name]))


def sample_rows(wl, n, seed):
    g = wl.geom
    rng = np.random.default_rng(seed)
    longest = int(np.argmax(wl.seq_lens))
    shortest = int(np.argmin(wl.seq_lens))
    bs = [longest, shortest, 0, wl.batch - 1] + list(rng.integers(0, wl.batch, n))
    ids = set()
    for i, b in enumerate(bs):
        t = int(rng.integers(0, g.t_q)) if i % 2 else g.t_q - 1
        h = int(rng.integers(0, g.n_head)) if i > 1 else (0 if i == 0 else g.n_head - 1)
        ids.add((b * g.t_q + t) * g.n_head + h)
    return sorted(ids)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["deepseek_decode", "glm53_flash_nope", "glm52_causal_t4"])
def test_full_size_sampled(name):
    wl = W.make_workload(name)
    run_stages(wl, rows=sample_rows(wl, 24, 7))


def test_poison_and_determinism():
    """NaN or 1e30 in rows no request may read changes no output bit, and
    two runs give identical bits."""
    import torch
    outs = []
    for poison in ("big", "nan", "nan"):
        wl = W.make_workload("glm52_causal_t4", seq_lens=[4, 33, 17, 64], poison=poison)
        cache_gpu, q_pe_gpu = gpu_sides(wl)
        dc = D.upload(wl, kv_cache=cache_gpu, q_pe=q_pe_gpu)
        D.full_step(dc)
        torch.cuda.synchronize()
        outs.append((dc.o_lat.view(torch.int16).cpu().numpy(), dc.lse.cpu().numpy(),
                     dc.out.view(torch.int16).cpu().numpy()))
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


def test_invalid_device_data_is_flagged():
    """A block id outside the pool, a seq_len beyond the table and a request
    shorter than t_q are caught on the device: the request's rows come back
    as zeros / -inf, the error word gets the bits, other rows are unaffected."""
    import torch
    wl = W.make_workload("glm52_causal_t4", seq_lens=[40, 40, 40, 2])
    wl.block_table[0, 1] = wl.num_blocks + 5      # out of the pool
    wl.seq_lens[1] = wl.max_blocks * 16 + 1        # beyond the table row
    dc = D.upload(wl)
    D.full_step(dc)
    torch.cuda.synchronize()
    err = int(dc.dev_err.item())
    assert err & N.DEVERR_BAD_BLOCK and err & N.DEVERR_SEQ_TOO_LONG and err & N.DEVERR_SEQ_SHORT
    H, T = wl.geom.n_head, wl.geom.t_q
    o = dc.o_lat.float().cpu().numpy().reshape(4, T, H, -1)
    lse = dc.lse.cpu().numpy().reshape(4, T, H)
    for b in (0, 1, 3):
        assert np.all(o[b] == 0) and np.all(np.isneginf(lse[b])), b
    assert np.all(np.isfinite(lse[2])) and np.abs(o[2]).max() > 0


def test_empty_requests_and_batch():
    import torch
    wl = W.make_workload("glm52_decode", seq_lens=[0, 0, 0])
    dc = D.upload(wl)
    D.full_step(dc)
    torch.cuda.synchronize()
    assert np.all(dc.o_lat.float().cpu().numpy() == 0)
    assert np.all(np.isneginf(dc.lse.cpu().numpy()))
    assert np.all(dc.out.float().cpu().numpy() == 0)
    # batch 0 is a no-op
    N.mla_decode_paged(0, 0, 0, 0, 0, 0, 0, 1, 1, dc.dims, 0.1, 0, 0, None)


@pytest.mark.parametrize("lens", [[1, 16, 32, 15, 17], [4096, 4095, 4097]])
def test_block_edges(lens):
    """Keys ending exactly on, just before and just after a block boundary."""
    run_stages(W.make_workload("glm52_decode", seq_lens=lens))


@pytest.mark.parametrize("name,lens", [
    ("glm52_decode", None),                                   # every request split over ~10 pairs
    ("deepseek_decode", [8192, 1, 100, 16, 0, 2049, 3000, 5000]),  # long and short mixed
])
def test_back_to_back_steps_are_identical_and_right(name, lens):
    """Twenty whole steps issued back to back on one stream, with no host
    synchronisation between them: the kernels of consecutive steps overlap
    (programmatic launches) and reuse the same buffers and workspace. Every
    step's latent output and LSE must be bit-identical to the first, and the
    first must match the oracle. A kernel that released a buffer too early
    shows here as a step that differs."""
    import torch
    wl = W.make_workload(name, seq_lens=lens)
    g = wl.geom
    dc = D.upload(wl)
    H, R, T = g.n_head, g.kv_rank, g.t_q
    snaps = []
    for _ in range(20):
        D.full_step(dc)
        snaps.append((dc.o_lat.clone(), dc.lse.clone(), dc.out.clone()))
    torch.cuda.synchronize()
    assert int(dc.dev_err.item()) == 0
    first = [t.view(torch.int16) if t.dtype == torch.bfloat16 else t for t in snaps[0]]
    for k, snap in enumerate(snaps[1:], 1):
        for a, b in zip(first, snap):
            b = b.view(torch.int16) if b.dtype == torch.bfloat16 else b
            assert torch.equal(a, b), f"step {k} differs from step 0"
    # the first step against the oracle (the chain rounds q_abs and o_lat to bf16)
    q_abs = W.round_bf16(oracle.absorb_q(wl.q_nope, wl.q_pe, wl.w_uk))
    o_ref, lse_ref = oracle.decode_paged(q_abs.reshape(wl.batch, T, H, -1), wl.kv_cache,
                                         wl.block_table, wl.seq_lens, T, R, wl.scale)
    assert_close(D.device_to_host_f32(snaps[0][0]), o_ref.reshape(-1, H, R), g.dtype,
                 "back-to-back decode out")
    assert_lse_close(snaps[0][1].cpu().numpy(), lse_ref.reshape(-1, H), g.dtype,
                     "back-to-back decode lse")


def oracle_decode_threaded(q4, wl, threads=None):
    """The oracle's decode of every (query row, head) pair, the pairs split
    over host threads (each call is the oracle's own decode_rows on disjoint
    pairs; the C code releases the GIL)."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    g = wl.geom
    n = wl.rows * g.n_head
    threads = threads or os.cpu_count() or 1
    parts = np.array_split(np.arange(n, dtype=np.int64), max(1, threads * 4))
    with ThreadPoolExecutor(threads) as ex:
        res = list(ex.map(lambda ids: oracle.decode_rows(
            q4, wl.kv_cache, wl.block_table, wl.seq_lens, g.t_q, g.kv_rank, wl.scale, ids),
            parts))
    return np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res])


@pytest.mark.slow
def test_deepseek_full_size_all_rows():
    """The whole DeepSeek-V3 geometry workload (64 requests of 8192 keys, 128
    heads): every query row of the decode against the oracle, so the full
    even split over all CTA pairs and its combine are compared row by row;
    then the fused step's output against the oracle's decompress."""
    import torch
    wl = W.make_workload("deepseek_decode")
    g = wl.geom
    H, R, T = g.n_head, g.kv_rank, g.t_q
    dc = D.upload(wl)
    q = rounded(oracle.absorb_q(wl.q_nope, wl.q_pe, wl.w_uk), g.dtype)
    dc.q_abs.copy_(D.host_to_device(q, g.dtype, "cuda"))
    D.decode(dc)
    torch.cuda.synchronize()
    assert int(dc.dev_err.item()) == 0
    o_ref, lse_ref = oracle_decode_threaded(q.reshape(wl.batch, T, H, -1), wl)
    assert_close(D.device_to_host_f32(dc.o_lat).reshape(-1, R), o_ref, g.dtype,
                 "deepseek decode out (all rows)")
    assert_lse_close(dc.lse.cpu().numpy().reshape(-1), lse_ref, g.dtype,
                     "deepseek decode lse (all rows)")
    D.attend(dc)
    torch.cuda.synchronize()
    assert int(dc.dev_err.item()) == 0
    out_ref = oracle.decompress(rounded(o_ref.reshape(-1, H, R), g.dtype), wl.w_uv)
    assert_close(D.device_to_host_f32(dc.out), out_ref, g.dtype, "deepseek fused step out")
