"""mla_prolog_q, the query half of the MLA prolog in one call ("aclnnMlaProlog",
computation formulas of the query), against the oracle.

The oracle composes its own pieces at the kernel's rounding points: the
RmsNorm of c_q (f64, stored f32), rounded to the path's 16-bit type; the
projections through W^UQ and W^QR (f32 sums); q^C rounded to the type; then
the absorb with the query's rope (oracle_absorb_q_rope). Tolerances: the
output gate of tests/tolerances.py on every element of q_abs.
"""
import numpy as np
import pytest

import oracle
from mla_latent_cache_absorbed_gb300 import _native as N
from mla_latent_cache_absorbed_gb300 import device as D
from mla_latent_cache_absorbed_gb300 import workloads as W
from tolerances import output_bound

pytestmark = pytest.mark.gpu


def oracle_q_abs(x: W.PrologQInputs):
    g = x.geom
    H, Dn, P = g.n_head, g.d_nope, g.d_rope
    cn = oracle.rmsnorm_rows(x.c_q, x.gamma_q, x.eps)
    cn = W.round_to(cn, g.dtype)
    qc = oracle.project(cn, x.w_uq).reshape(x.rows, H, Dn)
    qpe = (oracle.project(cn, x.w_qr).reshape(x.rows, H, P) if P
           else np.zeros((x.rows, H, 0), np.float32))
    qc = W.round_to(qc, g.dtype)
    return oracle.absorb_q_rope(qc, qpe, x.w_uk, x.positions, x.rope_base)


def run_gpu(x: W.PrologQInputs):
    import torch
    g = x.geom
    dt = g.dtype
    dev = "cuda"
    t = lambda a: D.host_to_device(a, dt, dev)
    q_abs = torch.full((x.rows, g.n_head, g.kv_rank + g.d_rope), float("nan"),
                       dtype={"bf16": torch.bfloat16, "f16": torch.float16}.get(dt, torch.float32),
                       device=dev)
    pos = torch.from_numpy(x.positions).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    w_qr = t(x.w_qr) if g.d_rope else None
    N.mla_prolog_q(q_abs, t(x.c_q), t(x.gamma_q), t(x.w_uq), w_qr, t(x.w_uk),
                   pos if g.d_rope else None, x.rows, x.q_rank, x.eps, x.rope_base,
                   N.MlaDims.from_geometry(g), err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return D.device_to_host_f32(q_abs)


def check(x):
    got = run_gpu(x).astype(np.float64)
    ref = oracle_q_abs(x).astype(np.float64)
    assert np.all(np.isfinite(got)), "non-finite output"
    err = np.abs(got - ref)
    bound = output_bound(ref, x.geom.dtype)
    bad = err > bound
    assert not bad.any(), (f"{int(bad.sum())} of {bad.size} outside, max err {err.max():.3e} "
                           f"at {np.unravel_index(np.argmax(err - bound), err.shape)}")


def geom(name, dtype=None, t_q=None):
    g = W.geometry(name)
    return W.Geometry(g.n_head, g.d_nope, g.d_rope, g.d_v, g.kv_rank,
                      g.t_q if t_q is None else t_q, dtype or g.dtype)


@pytest.mark.parametrize("name,rows,dtype", [
    ("glm52_decode", 8, None),          # GLM-5.2 decode rows (tensor cores, N = 192 + 64)
    ("deepseek_decode", 64, None),      # DeepSeek-V3 (N = 128 + 64)
    ("glm53_flash_nope", 128, None),    # NoPE (N = 256, no rope part)
    ("glm52_causal_t4", 130, None),     # two row tiles, the second with 2 rows
    ("glm52_prefill_chunk", 512, None), # four full row tiles
    ("glm52_decode", 8, "f16"),         # f16 operands
    ("deepseek_decode", 33, "f16"),
    ("deepseek_decode", 8, None),       # 128 heads: one CTA a head
    ("glm53_flash_nope", 24, None),     # a head over a CTA pair, no rope part
    ("glm52_decode", 40, None),         # a head over a CTA pair, 40-row tile
    ("glm52_decode", 47, None),         # ragged last 8-row group
])
def test_prolog_q_tensor_cores(name, rows, dtype):
    check(W.make_prolog_q(geom(name, dtype), rows))


def test_prolog_q_f32_simt():
    """The tiny f32 geometry (d_rope 8) goes through the SIMT form."""
    check(W.make_prolog_q(geom("tiny_f32"), 5, q_rank=48))


def test_prolog_q_bf16_simt_geometry():
    """A bf16 geometry outside the tensor-core kernel's (d_rope 32) takes the
    SIMT form with the same rounding points."""
    g = W.Geometry(4, 64, 32, 64, 512, 1, "bf16")
    check(W.make_prolog_q(g, 6, q_rank=256))


def test_prolog_q_position_zero_and_big_eps():
    """Position 0 turns nothing; a large eps dominates the norm."""
    x = W.make_prolog_q(geom("glm52_decode"), 8, eps=100.0)
    x.positions[:] = 0
    check(x)
