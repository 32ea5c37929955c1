"""mla_decode_paged_static: the decode for callers that cannot allocate.

Callers that record their work into CUDA graphs, or whose serving loop or
plugin host forbids device allocation, cannot provide mla_decode_paged's
workspace. This entry point keeps the split scratch in a static device array
inside the library instead. It runs the same kernels on the same inputs as
mla_decode_paged, so its results must be the same bits, call after call,
since every call reuses (and overwrites) the same array; one of the calls is
also checked against the oracle. The file is named to run last, after every
other test.
"""
import numpy as np
import pytest

import oracle
from mla_latent_cache_absorbed_gb300 import _native as N
from mla_latent_cache_absorbed_gb300 import device as D
from mla_latent_cache_absorbed_gb300 import workloads as W
from tolerances import lse_bound, output_bound

pytestmark = pytest.mark.gpu


def _oracle_queries(wl):
    """q_abs from the oracle's absorb, rounded to the workload's dtype."""
    q = oracle.absorb_q(wl.q_nope, wl.q_pe, wl.w_uk)
    return W.round_to(q, wl.geom.dtype) if wl.geom.dtype != "f32" else q


def _static_vs_workspace(wl, check_oracle):
    import torch
    g = wl.geom
    H, R, T = g.n_head, g.kv_rank, g.t_q
    dc = D.upload(wl)
    q = _oracle_queries(wl)
    dc.q_abs.copy_(D.host_to_device(q, g.dtype, "cuda"))
    D.decode(dc)  # the existing entry point, caller workspace
    torch.cuda.synchronize()
    assert int(dc.dev_err.item()) == 0
    o = torch.full_like(dc.o_lat, float("nan"))
    lse = torch.full_like(dc.lse, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    N.mla_decode_paged_static(o, lse, dc.q_abs, dc.kv_cache, dc.block_table, dc.seq_lens,
                              dc.batch, dc.max_blocks, dc.num_blocks, dc.dims, dc.scale, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # the same kernels on the same inputs: the same bits
    assert torch.equal(o.view(torch.int16), dc.o_lat.view(torch.int16)), "static-scratch output"
    assert torch.equal(lse, dc.lse), "static-scratch lse"
    if check_oracle:
        o_ref, lse_ref = oracle.decode_paged(q.reshape(wl.batch, T, H, -1), wl.kv_cache,
                                             wl.block_table, wl.seq_lens, T, R, wl.scale)
        got = D.device_to_host_f32(o).astype(np.float64)
        ref = o_ref.reshape(got.shape).astype(np.float64)
        assert np.all(np.abs(got - ref) <= output_bound(ref, g.dtype)), "output vs oracle"
        lg, lr = lse.cpu().numpy().reshape(-1), lse_ref.reshape(-1)
        assert np.array_equal(np.isneginf(lg), np.isneginf(lr))
        fin = ~np.isneginf(lr)
        assert np.abs(lg[fin] - lr[fin]).max() <= lse_bound(g.dtype), "lse vs oracle"


def test_static_scratch_matches_workspace_entry_point_twice():
    # two calls in a row on different batches: the second reuses the array
    # the first left filled (both split requests across several CTA pairs)
    _static_vs_workspace(W.make_workload("glm52_decode", seq_lens=[300, 0, 1, 1000]), True)
    _static_vs_workspace(W.make_workload("glm52_decode", seq_lens=[17, 64, 2048]), False)


def test_static_scratch_rejects_oversize_batches():
    """A batch whose split scratch exceeds the static array is refused with a
    clear message and nothing is launched (here the f32 path, whose scratch
    grows with the batch)."""
    d = N.MlaDims.from_geometry(W.geometry("tiny_f32"))
    need = N.mla_decode_workspace_size(100000, 64, d)
    assert need > (64 << 20)
    with pytest.raises(N.MlaError) as e:
        N.mla_decode_paged_static(256, 256, 256, 256, 256, 256, 100000, 64, 10, d, 0.1)
    assert "static scratch" in str(e.value)
