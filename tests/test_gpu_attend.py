"""The fused call mla_attend_absorbed against the three calls it replaces.

mla_attend_absorbed runs absorb, decode and decompress as one chain; on the
bf16 tensor-core path the decompress merges the decode's split rows itself
(no combine kernel). Its contract is the same bits as mla_absorb_q ->
mla_decode_paged -> mla_decompress_out, whose parity with the oracle the
other GPU tests establish; one case here also checks the oracle directly.
"""
import numpy as np
import pytest

import oracle
from mla_latent_cache_absorbed_gb300 import _native as N
from mla_latent_cache_absorbed_gb300 import device as D
from mla_latent_cache_absorbed_gb300 import workloads as W

from tolerances import output_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    assert torch.cuda.is_available()
    N.load()


def bits(t):
    import torch
    return (t.view(torch.int16) if t.dtype == torch.bfloat16 else t).cpu().numpy()


def three_then_fused(wl, **upload_kw):
    """Outputs (out, lse, dev_err) of the three calls and of the fused call."""
    import torch
    dc = D.upload(wl, **upload_kw)
    D.full_step(dc)
    torch.cuda.synchronize()
    ref = (bits(dc.out), dc.lse.cpu().numpy().copy(), int(dc.dev_err.item()))
    dc.out.fill_(float("nan"))
    dc.lse.fill_(float("nan"))
    dc.dev_err.zero_()
    D.attend(dc)
    torch.cuda.synchronize()
    got = (bits(dc.out), dc.lse.cpu().numpy().copy(), int(dc.dev_err.item()))
    return dc, ref, got


def assert_same(ref, got, what):
    assert np.array_equal(ref[0].view(np.uint8), got[0].view(np.uint8)), f"{what}: out differs"
    assert np.array_equal(ref[1].view(np.uint8), got[1].view(np.uint8)), f"{what}: lse differs"
    assert ref[2] == got[2], f"{what}: dev_err {ref[2]} vs {got[2]}"


CASES = [
    ("tiny_f32", None),                                        # SIMT path, three calls inside
    ("glm52_decode", None),                                    # aligned split, ~10 parts a row
    ("glm52_decode", [1, 16, 32, 15, 17]),                      # block edges, one tile each
    ("glm52_decode", [0, 0, 0]),                               # every request empty
    ("deepseek_decode", [8192, 1, 100, 16, 0, 2049]),           # even split, mixed lengths
    ("deepseek_decode", [8192, 1, 100, 16, 0, 2049, 3000, 5000]),
    ("glm53_flash_nope", [2048, 7, 0, 129, 31, 32768]),         # NoPE rows, one long request
    ("glm52_causal_t4", [4, 5, 100, 1000, 0, 4096]),            # t_q = 4: two row groups
    ("glm52_decode", [32768]),       # one request on every pair: 76 parts a row
    ("glm52_decode", [5000]),        # batch of one: the cluster's second CTA owns no row
    ("deepseek_decode", [20000]),    # batch of one, 128 heads, one merge CTA per head
]


@pytest.mark.parametrize("name,lens", CASES)
def test_fused_equals_three_calls(name, lens):
    wl = W.make_workload(name, seq_lens=lens)
    _, ref, got = three_then_fused(wl)
    assert ref[2] == 0
    assert_same(ref, got, f"{name} {lens}")


def test_fused_flags_invalid_device_data_like_three_calls():
    """Bad block id, seq_len past the table, request shorter than t_q: the
    same rows are zero / -inf and the same error bits are set."""
    wl = W.make_workload("glm52_causal_t4", seq_lens=[40, 40, 40, 2])
    wl.block_table[0, 1] = wl.num_blocks + 5
    wl.seq_lens[1] = wl.max_blocks * 16 + 1
    _, ref, got = three_then_fused(wl)
    assert ref[2] & N.DEVERR_BAD_BLOCK and ref[2] & N.DEVERR_SEQ_TOO_LONG
    assert ref[2] & N.DEVERR_SEQ_SHORT
    assert_same(ref, got, "invalid data")


def test_fused_matches_oracle_glm52():
    """The fused step's output and LSE against the oracle (the chain rounds
    q_abs and o_lat to bf16 at the same points)."""
    import torch
    wl = W.make_workload("glm52_decode")
    g = wl.geom
    H, R, T = g.n_head, g.kv_rank, g.t_q
    dc = D.upload(wl)
    D.attend(dc)
    torch.cuda.synchronize()
    assert int(dc.dev_err.item()) == 0
    q_abs = W.round_bf16(oracle.absorb_q(wl.q_nope, wl.q_pe, wl.w_uk))
    o_ref, lse_ref = oracle.decode_paged(q_abs.reshape(wl.batch, T, H, -1), wl.kv_cache,
                                         wl.block_table, wl.seq_lens, T, R, wl.scale)
    out_ref = oracle.decompress(W.round_bf16(o_ref.reshape(-1, H, R)), wl.w_uv)
    got = dc.out.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - out_ref)
    assert np.all(err <= output_bound(out_ref, "bf16")), err.max()
    lse = dc.lse.cpu().numpy().astype(np.float64)
    lse_ref = lse_ref.reshape(-1, H).astype(np.float64)
    empty = np.isneginf(lse_ref)                     # the batch's empty request
    assert empty.any() and np.array_equal(np.isneginf(lse), empty)
    assert np.abs(lse[~empty] - lse_ref[~empty]).max() <= 1e-3


@pytest.mark.parametrize("name,lens", [("glm52_decode", None),
                                       ("deepseek_decode", [8192, 1, 100, 16, 0, 2049, 3000])])
def test_fused_back_to_back(name, lens):
    """Twenty fused steps with no host synchronisation: every step gives the
    bits of the three-call step (the chains of consecutive steps overlap)."""
    import torch
    wl = W.make_workload(name, seq_lens=lens)
    dc = D.upload(wl)
    D.full_step(dc)
    torch.cuda.synchronize()
    ref_out, ref_lse = bits(dc.out), dc.lse.cpu().numpy().copy()
    snaps = []
    for _ in range(20):
        D.attend(dc)
        snaps.append((dc.out.clone(), dc.lse.clone()))
    torch.cuda.synchronize()
    assert int(dc.dev_err.item()) == 0
    for k, (o, l) in enumerate(snaps):
        assert np.array_equal(bits(o).view(np.uint8), ref_out.view(np.uint8)), f"step {k}"
        assert np.array_equal(l.cpu().numpy().view(np.uint8), ref_lse.view(np.uint8)), f"step {k}"


def test_fused_workspace_and_validation():
    import torch
    wl = W.make_workload("glm52_decode", seq_lens=[100, 200])
    dc = D.upload(wl)
    need = N.mla_attend_workspace_size(dc.batch, dc.max_blocks, dc.dims)
    assert need >= N.mla_decode_workspace_size(dc.batch, dc.max_blocks, dc.dims)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(N.MlaError) as e:
        N.mla_attend_absorbed(dc.out, dc.lse, dc.q_nope, dc.q_pe, dc.w_uk, dc.w_uv, dc.kv_cache,
                              dc.block_table, dc.seq_lens, dc.batch, dc.max_blocks,
                              dc.num_blocks, dc.dims, dc.scale, ws, need - 1)
    assert "workspace" in str(e.value)
    # batch 0 is a no-op
    N.mla_attend_absorbed(0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 1, 1, dc.dims, 0.1, 0, 0)
