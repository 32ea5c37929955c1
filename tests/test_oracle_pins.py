"""The oracle against its pins (no GPU): see tests/pins.py for what each pins."""
import pytest

import oracle
import pins


@pytest.mark.parametrize("check", pins.QUICK_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check(oracle.load())


def test_naive_equals_absorbed_full_dims():
    pins.check_naive_equals_absorbed_full_dims(oracle.load())


def test_nope_geometry_scale():
    """MlaDims::scale of mla.rs with no rope columns: the NoPE geometry's scale is
    1/sqrt(d_nope + d_rope) = 1/16, the same as GLM-5.2's, never 1/sqrt(512)."""
    from mla_latent_cache_absorbed_gb300 import workloads
    import math
    nope = workloads.geometry("glm53_flash_nope")
    glm = workloads.geometry("glm52_decode")
    s_nope = 1.0 / math.sqrt(nope.d_nope + nope.d_rope)
    s_glm = 1.0 / math.sqrt(glm.d_nope + glm.d_rope)
    assert nope.d_nope + nope.d_rope == 256
    assert abs(s_nope - 1.0 / 16.0) <= 1e-9 and abs(s_glm - s_nope) <= 1e-9
    assert abs(s_nope - 1.0 / math.sqrt(nope.kv_rank)) > 1e-3
