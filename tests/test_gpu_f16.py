"""The path with f16 queries, cache, weights and outputs, against the oracle.

f16 is one of the element types the vLLM CPU MLA backend lists. The tensor
cores take it as they take bf16 (kind::f16 MMAs, both operands f16, f32
accumulators), the SIMT kernels through their __half instances. The workloads
are the named ones with their values rounded to f16 (ties to even) instead of
bf16; the oracle consumes the same f16 values as f32. Tolerances:
test_gpu_parity.py's f16 gate.
"""
import numpy as np
import pytest

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


def f16_workload(name, lens=None, t_q=None, poison="big"):
    g = W.geometry(name)
    geom = W.Geometry(g.n_head, g.d_nope, g.d_rope, g.d_v, g.kv_rank,
                      g.t_q if t_q is None else t_q, "f16")
    return W.make_workload(name, seq_lens=lens, geom=geom, poison=poison)


@pytest.mark.parametrize("name,lens,t_q", [
    ("tiny_f32", None, None),                                # SIMT kernels (rank 32)
    ("glm52_decode", None, None),                            # tensor cores, full workload
    ("deepseek_decode", [8192, 1, 100, 16, 0, 2049], None),  # 128 heads
    ("glm53_flash_nope", [2048, 7, 0, 129, 31], None),       # 512-wide rows
    ("glm52_causal_t4", [4, 5, 100, 1000, 0], None),         # interleaved rope, t_q = 4
    ("glm52_decode", [16, 17, 300, 0], 16),                  # a prefill chunk
])
def test_f16_all_rows(name, lens, t_q):
    parity.run_stages(f16_workload(name, lens, t_q))


def test_f16_nan_poison():
    """NaN in rows no request may read changes nothing."""
    parity.run_stages(f16_workload("glm52_decode", [1, 16, 33, 500], poison="nan"))


@pytest.mark.parametrize("name,lens", [("glm52_decode", None),
                                       ("deepseek_decode", [8192, 1, 100, 16, 0, 2049, 3000]),
                                       ("glm52_causal_t4", [4, 5, 100, 1000, 0, 4096])])
def test_f16_fused_equals_three_calls(name, lens):
    wl = f16_workload(name, lens)
    _, ref, got = attend.three_then_fused(wl)
    assert ref[2] == 0
    attend.assert_same(ref, got, f"f16 {name} {lens}")

