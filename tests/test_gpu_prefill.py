"""Chunked causal prefill in absorbed form: a block of t_q queries per request.

The queries of a chunk are the request's last t_q positions and query t sees
keys 0 .. seq_len - t_q + t; a first chunk has t_q == seq_len (query t sees
keys 0 .. t). The decode entry points take such blocks as they are: on the
tensor-core path the t_q * n_head query rows of a request form row groups of
128 and each row group gets a set of CTA pairs of its own; with more row
groups than the grid has pairs (more than 9728 query rows on 152 SMs) each
row group gets one pair and a pair walks several row groups in turn. Parity
is against the oracle on the same bf16 values, with the tolerances of
test_gpu_parity.py.
"""
import numpy as np
import pytest

import oracle
import test_gpu_attend as attend
import test_gpu_parity as parity
from mla_latent_cache_absorbed_gb300 import _native as N
from mla_latent_cache_absorbed_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    assert torch.cuda.is_available()
    N.load()


def chunk_workload(name, t_q, lens, seed=None):
    """The named workload's geometry and value recipe with t_q queries per
    request and the given seq_lens (the pool: the blocks needed and 8 spare)."""
    g = W.geometry(name)
    geom = W.Geometry(g.n_head, g.d_nope, g.d_rope, g.d_v, g.kv_rank, t_q, g.dtype)
    need = sum((int(s) + W.BLOCK - 1) // W.BLOCK for s in lens)
    return W.make_workload(name, seed=seed, seq_lens=lens, geom=geom, pool_blocks=need + 8)


def sampled_stages(wl, ids):
    """Per-stage parity on sampled query rows, for chunks too large for the
    oracle to compute whole. ids: flattened (b * t_q + t) * H + h.
      absorb      the oracle absorbs the sampled query rows (all heads);
      decode      those rows, rounded to bf16, replace the GPU's own absorbed
                  rows in q_abs, so both sides decode the same values; the
                  oracle decodes the sampled (row, head) pairs alone;
      decompress  a seeded random latent input for every row; the oracle
                  decompresses the sampled rows."""
    import torch
    from mla_latent_cache_absorbed_gb300 import device as D
    g = wl.geom
    H, R, T, dt = g.n_head, g.kv_rank, g.t_q, g.dtype
    ids = np.asarray(sorted(set(int(i) for i in ids)), np.int64)
    rs = np.unique(ids // H)
    dc = D.upload(wl)
    D.absorb(dc)
    torch.cuda.synchronize()
    q_abs_rows = oracle.absorb_q(wl.q_nope[rs], wl.q_pe[rs], wl.w_uk)
    parity.assert_close(D.device_to_host_f32(dc.q_abs)[rs], q_abs_rows, dt, "absorb (sampled)")

    q_in = parity.rounded(q_abs_rows, dt)
    dc.q_abs[torch.from_numpy(rs).cuda()] = D.host_to_device(q_in, dt, "cuda")
    D.decode(dc)
    torch.cuda.synchronize()
    assert int(dc.dev_err.item()) == 0
    q4 = np.zeros((wl.rows, H, g.width), np.float32)
    q4[rs] = q_in
    o_ref, lse_ref = oracle.decode_rows(q4.reshape(wl.batch, T, H, -1), wl.kv_cache,
                                        wl.block_table, wl.seq_lens, T, R, wl.scale, ids)
    parity.assert_close(D.device_to_host_f32(dc.o_lat).reshape(-1, R)[ids], o_ref, dt,
                        "decode out (sampled)")
    parity.assert_lse_close(dc.lse.cpu().numpy().reshape(-1)[ids], lse_ref, dt,
                            "decode lse (sampled)")

    rng = np.random.default_rng(123)
    o_in = parity.rounded(rng.standard_normal((wl.rows, H, R)).astype(np.float32) * 0.1, dt)
    dc.o_lat.copy_(D.host_to_device(o_in, dt, "cuda"))
    D.decompress(dc)
    torch.cuda.synchronize()
    parity.assert_close(D.device_to_host_f32(dc.out)[rs], oracle.decompress(o_in[rs], wl.w_uv),
                        dt, "decompress (sampled)")


CHUNKS = [
    # GLM-5.2 dims, 16 queries: 8 row groups; a first chunk, one row past it,
    # later chunks and an empty request
    ("glm52_decode", 16, [16, 17, 100, 0, 300]),
    # 128 queries, a first chunk: 64 row groups, one pair each on 152 SMs
    ("glm52_decode", 128, [128]),
    # DeepSeek geometry (128 heads), 32 queries: 32 row groups
    ("deepseek_decode", 32, [32, 200]),
    # NoPE rows (512 wide), 16 queries
    ("glm53_flash_nope", 16, [16, 300, 0]),
    # more row groups than the 76 pairs of 152 SMs: 80 row groups a request,
    # pairs 0-3 walk two of them (a first chunk and a later one)
    ("glm52_decode", 160, [160, 300]),
    # 160 row groups: pairs 0-7 walk three
    ("glm52_decode", 320, [320]),
    # DeepSeek geometry, 80 queries of 128 heads: 80 row groups
    ("deepseek_decode", 80, [80, 129]),
]


@pytest.mark.parametrize("name,t_q,lens", CHUNKS)
def test_chunk_all_rows(name, t_q, lens):
    """Every stage and the chained path against the oracle, every row."""
    parity.run_stages(chunk_workload(name, t_q, lens))


def test_chunk_beyond_row_group_limit_sampled():
    """160 queries of 64 heads are 80 row groups, more than the 76 pairs of
    the tensor-core grid on 152 SMs: pairs 0-3 walk two row groups each. A
    longer request than the all-rows case, on sampled rows."""
    wl = chunk_workload("glm52_decode", 160, [160, 500])
    sampled_stages(wl, parity.sample_rows(wl, 24, 5))


def test_prefill_chunk_workload_sampled():
    """The full glm52_prefill_chunk workload (t_q = 128, B = 4, a first chunk
    and three later ones up to 8192 rows) on sampled query rows."""
    wl = W.make_workload("glm52_prefill_chunk")
    sampled_stages(wl, parity.sample_rows(wl, 32, 11))


@pytest.mark.parametrize("name,t_q,lens", [("glm52_decode", 16, [16, 17, 100, 0, 1000]),
                                           ("glm52_prefill_chunk", 128, None)])
def test_fused_chunk_equals_three_calls(name, t_q, lens):
    """mla_attend_absorbed on a chunk gives the bits of absorb -> decode ->
    decompress. With more than 256 query rows per request the fused call runs
    those three calls itself (the merging decompress would look up the split
    parts of up to 128 row groups per CTA), so this pins that dispatch."""
    wl = (W.make_workload(name) if lens is None else chunk_workload(name, t_q, lens))
    _, ref, got = attend.three_then_fused(wl)
    assert ref[2] == 0
    attend.assert_same(ref, got, f"{name} t_q={t_q} {lens}")


def test_chunk_row_is_cut_decode():
    """Query t of a chunk equals a one-query decode of the same request whose
    seq_len is cut at that query's position (same cache, same block table).
    The two launches split the keys differently, so they agree to the bf16
    tolerance rather than bit for bit."""
    import torch
    from mla_latent_cache_absorbed_gb300 import device as D
    S = 700
    wl = chunk_workload("glm52_decode", 16, [S])
    g = wl.geom
    H, R, T = g.n_head, g.kv_rank, g.t_q
    dc = D.upload(wl)
    D.absorb(dc)
    D.decode(dc)
    torch.cuda.synchronize()
    assert int(dc.dev_err.item()) == 0
    o_chunk = D.device_to_host_f32(dc.o_lat).reshape(T, H, R)
    lse_chunk = dc.lse.cpu().numpy().reshape(T, H)
    dims1 = N.MlaDims.from_geometry(W.Geometry(g.n_head, g.d_nope, g.d_rope, g.d_v, g.kv_rank,
                                               1, g.dtype))
    ws1 = N.mla_decode_workspace_size(1, dc.max_blocks, dims1)
    work = torch.empty(max(ws1, 256), dtype=torch.uint8, device="cuda")
    for t in (0, 7, T - 1):
        q1 = dc.q_abs[t:t + 1].clone()          # query rows are b * t_q + t, here b = 0
        o1 = torch.empty((1, H, R), dtype=dc.o_lat.dtype, device="cuda")
        l1 = torch.empty((1, H), dtype=torch.float32, device="cuda")
        sl1 = torch.tensor([S - T + t + 1], dtype=torch.int32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        N.mla_decode_paged(o1, l1, q1, dc.kv_cache, dc.block_table, sl1, 1, dc.max_blocks,
                           dc.num_blocks, dims1, dc.scale, work, ws1, err, None)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        parity.assert_close(D.device_to_host_f32(o1).reshape(H, R), o_chunk[t], "bf16",
                            f"cut decode t={t}")
        assert np.abs(l1.cpu().numpy().reshape(H) - lse_chunk[t]).max() <= 1e-3
