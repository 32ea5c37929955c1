"""mla_absorb_q_rope (the absorb with the query's rope) against the oracle.

Tolerances, per part of each q_abs row:
  latent part   as the absorb's (test_gpu_parity.py): f32 max abs diff 1e-4;
                bf16 1e-2 plus half a bf16 ulp of |ref|;
  rope part     both sides turn the pair (a, b) by the same f32 theta (the same
                recurrence from the same f32 ratio), so they differ by their
                sin / cos (a few f32 ulps) and the products' rounding:
                1e-6 (|a| + |b|), plus 2^-8 |ref| for a bf16 result.
"""
import numpy as np
import pytest

import oracle
from mla_latent_cache_absorbed_gb300 import _native as N
from mla_latent_cache_absorbed_gb300 import device as D
from mla_latent_cache_absorbed_gb300 import workloads as W

from tolerances import output_bound

pytestmark = pytest.mark.gpu

BASE = 10000.0


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    assert torch.cuda.is_available()
    N.load()


def case(name, lens, seed=7):
    """The workload's q_nope and w_uk, a fresh pre-rope q_pe (seeded, rounded
    to the dtype) and each query row's position: the decode's
    seq_len - t_q + t, with a few far positions mixed in."""
    wl = W.make_workload(name, seq_lens=lens)
    g = wl.geom
    rng = np.random.default_rng(seed)
    q_pe = rng.standard_normal((wl.rows, g.n_head, g.d_rope)).astype(np.float32)
    if g.dtype == "bf16":
        q_pe = W.round_bf16(q_pe)
    pos = np.zeros(wl.rows, np.int64)
    for b, s in enumerate(wl.seq_lens):
        for t in range(g.t_q):
            pos[b * g.t_q + t] = max(int(s) - g.t_q + t, 0)
    far = [70000, 1 << 20, 16777215]
    pos[-min(len(far), wl.rows):] = far[:min(len(far), wl.rows)]
    return wl, q_pe, pos


def run_gpu(wl, q_pe, pos):
    import torch
    g = wl.geom
    dc = D.upload(wl, q_pe=q_pe)
    pos_d = torch.from_numpy(pos).cuda()
    N.mla_absorb_q_rope(dc.q_abs, dc.q_nope, dc.q_pe, dc.w_uk, pos_d, wl.rows, BASE, dc.dims)
    torch.cuda.synchronize()
    return dc, D.device_to_host_f32(dc.q_abs)


def check(wl, q_pe, pos, got):
    g = wl.geom
    R, P = g.kv_rank, g.d_rope
    ref = oracle.absorb_q_rope(wl.q_nope, q_pe, wl.w_uk, pos, BASE)
    err = np.abs(got.astype(np.float64) - ref)
    lat_ref = np.abs(ref[..., :R])
    lat_tol = output_bound(lat_ref, g.dtype)
    assert np.all(err[..., :R] <= lat_tol), f"latent part: max err {err[..., :R].max():.3e}"
    if P:
        h = P // 2
        ab = np.abs(q_pe[..., :h]).astype(np.float64) + np.abs(q_pe[..., h:])
        tol = 1e-6 * np.concatenate([ab, ab], axis=-1)
        if g.dtype == "bf16":
            tol = tol + 2.0 ** -8 * np.abs(ref[..., R:])
        bad = err[..., R:] > tol
        assert not bad.any(), f"rope part: {int(bad.sum())} outside, max err {err[..., R:].max():.3e}"


@pytest.mark.parametrize("name,lens", [
    ("tiny_f32", None),                           # f32: the SIMT absorb
    ("glm52_decode", None),                       # bf16: the tensor-core absorb
    ("glm52_causal_t4", [4, 5, 100, 1000]),       # four query rows per request
    ("glm52_prefill_chunk", None),                # 512 query rows, 4 M tiles
])
def test_absorb_q_rope_matches_oracle(name, lens):
    wl, q_pe, pos = case(name, lens)
    _, got = run_gpu(wl, q_pe, pos)
    check(wl, q_pe, pos, got)


def test_position_zero_is_the_plain_absorb():
    """At position 0 the rope turns nothing: the same bits as mla_absorb_q."""
    import torch
    wl, q_pe, pos = case("glm52_decode", None)
    pos[:] = 0
    dc, got = run_gpu(wl, q_pe, pos)
    plain = torch.empty_like(dc.q_abs)
    N.mla_absorb_q(plain, dc.q_nope, dc.q_pe, dc.w_uk, wl.rows, dc.dims)
    torch.cuda.synchronize()
    assert torch.equal(plain.view(torch.int16), dc.q_abs.view(torch.int16))


def test_nope_rows_are_the_plain_absorb():
    """With no rope columns the call is mla_absorb_q (positions unused)."""
    import torch
    wl = W.make_workload("glm53_flash_nope", seq_lens=[5, 9])
    dc = D.upload(wl)
    N.mla_absorb_q_rope(dc.q_abs, dc.q_nope, None, dc.w_uk, None, wl.rows, 0.0, dc.dims)
    torch.cuda.synchronize()
    got = dc.q_abs.clone()
    N.mla_absorb_q(dc.q_abs, dc.q_nope, None, dc.w_uk, wl.rows, dc.dims)
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), dc.q_abs.view(torch.int16))
