"""mla_decode_paged_static: the decode for callers that cannot allocate.

Callers that record their work into CUDA graphs, or whose serving loop or
plugin host forbids device allocation, cannot provide mla_decode_paged's
workspace. This entry point keeps the split scratch in a static device array
inside the library instead. Its results must match mla_decode_paged's, call
after call, since every call reuses (and overwrites) the same array. The file
is named to run last, after every other test.
"""
import numpy as np
import pytest

from mla_latent_cache_absorbed_gb300 import _native as N
from mla_latent_cache_absorbed_gb300 import device as D
from mla_latent_cache_absorbed_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ATOL_BF16, RTOL_BF16, ATOL_LSE = 1e-2, 2.0 ** -8, 1e-3


def _close(got, ref, atol, rtol, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    both_ninf = np.isneginf(got) & np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), what
    with np.errstate(invalid="ignore"):
        err = np.abs(np.where(both_ninf, 0.0, got - ref))
    assert np.all(err <= atol + rtol * np.abs(np.where(both_ninf, 0.0, ref))), \
        f"{what}: max err {err.max():.3e}"


def _static_vs_workspace(wl):
    import torch
    dc = D.upload(wl)
    D.absorb(dc)
    D.decode(dc)  # the existing entry point, caller workspace
    torch.cuda.synchronize()
    ref_o = dc.o_lat.float().cpu().numpy()
    ref_l = dc.lse.cpu().numpy()
    o = torch.full_like(dc.o_lat, float("nan"))
    lse = torch.full_like(dc.lse, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    N.mla_decode_paged_static(o, lse, dc.q_abs, dc.kv_cache, dc.block_table, dc.seq_lens,
                              dc.batch, dc.max_blocks, dc.num_blocks, dc.dims, dc.scale, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _close(o.float().cpu().numpy(), ref_o, ATOL_BF16, RTOL_BF16, "static-scratch output")
    _close(lse.cpu().numpy(), ref_l, ATOL_LSE, 0.0, "static-scratch lse")


def test_static_scratch_matches_workspace_entry_point_twice():
    # two calls in a row on different batches: the second reuses the array
    # the first left filled
    _static_vs_workspace(W.make_workload("glm52_decode", seq_lens=[300, 0, 1, 1000]))
    _static_vs_workspace(W.make_workload("glm52_decode", seq_lens=[17, 64, 2048]))


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
