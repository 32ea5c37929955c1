"""The C-ABI library loads, exports every declared symbol, and its host-side
logic (validation, workspace sizing, the rope permutation) behaves, with no
GPU and no kernel launch."""
import ctypes
import os
import re

import numpy as np
import pytest

from mla_latent_cache_absorbed_gb300 import _native as N

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_symbols():
    text = open(os.path.join(ROOT, "include", "mla.h")).read()
    return sorted(set(re.findall(r"^\s*(?:mla_status|const char\*)\s+(mla_\w+)\s*\(", text,
                                 re.M)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(N.LIB_PATH):
        from mla_latent_cache_absorbed_gb300 import build
        build.build()
    return N.load()


def test_exports_every_header_symbol(lib):
    syms = header_symbols()
    assert len(syms) >= 9
    assert set(syms) == set(N.EXPORTS)
    for s in syms:
        assert getattr(lib, s) is not None


def test_status_strings(lib):
    for s in range(6):
        assert N.mla_status_str(s).startswith("MLA_")


def test_rope_perm_matches_definition(lib):
    assert list(N.mla_rope_norm_to_neox_perm(8)) == [0, 4, 1, 5, 2, 6, 3, 7]
    for n in (0, 2, 64):
        p = N.mla_rope_norm_to_neox_perm(n)
        assert sorted(p) == list(range(n))
        assert all(p[2 * j] == j and p[2 * j + 1] == j + n // 2 for j in range(n // 2))
    with pytest.raises(N.MlaError):
        N.mla_rope_norm_to_neox_perm(7)


def test_rope_perm_agrees_with_oracle(lib):
    import oracle
    for n in (2, 8, 64):
        assert np.array_equal(N.mla_rope_norm_to_neox_perm(n), oracle.norm_to_neox_perm(n))


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_permute_rope_cols(lib, dtype):
    x = np.arange(3 * 12).reshape(3, 12).astype(dtype)
    orig = x.copy()
    N.mla_permute_rope_cols(x, 4, 8)
    perm = N.mla_rope_norm_to_neox_perm(8)
    for r in range(3):
        assert np.array_equal(x[r, :4], orig[r, :4])
        for i in range(8):
            assert x[r, 4 + perm[i]] == orig[r, 4 + i]


def test_permute_rope_rows_matches_cols_on_transpose(lib):
    """Permuting the rope rows of a weight W equals permuting the rope
    columns of the activations x W^T it produces."""
    rng = np.random.default_rng(0)
    Wt = rng.standard_normal((10, 6)).astype(np.float32)  # [out_features, in]
    x = rng.standard_normal((4, 6)).astype(np.float32)
    y = x @ Wt.T
    N.mla_permute_rope_cols(y, 2, 8)
    W2 = Wt.copy()
    N.mla_permute_rope_rows(W2, 2, 8)
    assert np.allclose(x @ W2.T, y, atol=1e-6)


def test_validation_without_launch(lib):
    d = N.MlaDims(4, 16, 8, 16, 32, 1, 16, N.MLA_F32)
    bad = N.MlaDims(4, 16, 8, 16, 32, 1, 32, N.MLA_F32)  # block size 32
    with pytest.raises(N.MlaError) as e:
        N.mla_absorb_q(0, 0, 0, 0, 2, bad, 0)
    assert e.value.status == 1 and "block_size" in N.mla_last_error()
    with pytest.raises(N.MlaError):
        N.mla_absorb_q(0, 0, 0, 0, 2, d, 0)  # NULL buffers
    with pytest.raises(N.MlaError):
        N.mla_absorb_q(16, 16, 0, 16, 2, d, 0)  # q_pe NULL with d_rope > 0
    with pytest.raises(N.MlaError):
        N.mla_absorb_q(17, 16, 16, 16, 2, d, 0)  # misaligned
    N.mla_absorb_q(0, 0, 0, 0, 0, d, 0)  # zero rows: no-op
    odd = N.MlaDims(4, 16, 6, 16, 32, 1, 16, N.MLA_BF16)  # 12-byte rope rows
    with pytest.raises(N.MlaError):
        N.mla_decompress_out(16, 16, 16, 1, odd, 0)


def test_absorb_q_rope_validation(lib):
    """Argument checks of the absorb with the query's rope, before any launch."""
    d = N.MlaDims(4, 16, 8, 16, 32, 1, 16, N.MLA_BF16)
    f = N.mla_absorb_q_rope
    with pytest.raises(N.MlaError):
        f(256, 512, 768, 1024, 0, 2, 10000.0, d, 0)          # positions NULL with d_rope > 0
    with pytest.raises(N.MlaError):
        f(256, 512, 0, 1024, 1280, 2, 10000.0, d, 0)         # q_pe NULL with d_rope > 0
    with pytest.raises(N.MlaError):
        f(256, 512, 768, 1024, 1284, 2, 10000.0, d, 0)       # positions misaligned
    with pytest.raises(N.MlaError):
        f(256, 512, 768, 1024, 1280, 2, 0.0, d, 0)           # rope_base <= 0
    with pytest.raises(N.MlaError):
        f(256, 512, 768, 1024, 1280, 2, float("inf"), d, 0)  # rope_base not finite
    with pytest.raises(N.MlaError):
        f(256, 512, 768, 1024, 1280, -1, 10000.0, d, 0)      # negative rows
    f(0, 0, 0, 0, 0, 0, 10000.0, d, 0)                       # no rows: no-op


def test_decode_workspace_and_validation(lib):
    d = N.MlaDims(4, 16, 8, 16, 32, 1, 16, N.MLA_F32)
    n = N.mla_decode_workspace_size(2, 4, d)
    assert n > 0
    assert N.mla_decode_workspace_size(0, 4, d) >= 0
    with pytest.raises(N.MlaError):
        N.mla_decode_workspace_size(-1, 4, d)
    with pytest.raises(N.MlaError) as e:  # workspace too small
        N.mla_decode_paged(256, 0, 256, 256, 256, 256, 2, 4, 8, d, 0.2, 256, 16, None, 0)
    assert "workspace" in str(e.value)
    with pytest.raises(N.MlaError):  # misaligned workspace
        N.mla_decode_paged(256, 0, 256, 256, 256, 256, 2, 4, 8, d, 0.2, 272, n, None, 0)
    with pytest.raises(N.MlaError):  # NaN scale
        N.mla_decode_paged(256, 0, 256, 256, 256, 256, 2, 4, 8, d, float("nan"), 256, n,
                           None, 0)
    N.mla_decode_paged(0, 0, 0, 0, 0, 0, 0, 4, 8, d, 0.2, 0, 0, None, 0)  # empty batch
    # 32-bit index limits: query rows and cache positions
    big = N.MlaDims(4, 16, 8, 16, 32, 1 << 20, 16, N.MLA_F32)
    with pytest.raises(N.MlaError) as e:
        N.mla_decode_workspace_size(1024, 4, big)    # 2^32 query rows
    assert e.value.status == 2 and "query rows" in N.mla_last_error()
    with pytest.raises(N.MlaError) as e:
        N.mla_attend_workspace_size(1024, 4, big)
    assert e.value.status == 2
    with pytest.raises(N.MlaError) as e:
        N.mla_decode_workspace_size(2, 1 << 27, d)
    assert e.value.status == 2
    assert N.mla_decode_workspace_size(2, (1 << 27) - 1, d) > 0
    # the work split's 64-token tiles, batch * ceil(max_blocks / 4), are a
    # 32-bit count: 2^24 requests of 509 blocks (ceil(509 / 4) = 2^7 tiles
    # each) make 2^31 tiles, one too many, although batch * max_blocks is
    # below 2^33
    one_head = N.MlaDims(1, 16, 8, 16, 32, 1, 16, N.MLA_F32)
    with pytest.raises(N.MlaError) as e:
        N.mla_decode_workspace_size(1 << 24, 509, one_head)
    assert e.value.status == 2 and "cache tiles" in N.mla_last_error()
    with pytest.raises(N.MlaError):
        N.mla_attend_workspace_size(1 << 24, 512, one_head)
    assert N.mla_decode_workspace_size((1 << 24) - 1, 512, one_head) > 0


def test_f16_dims(lib):
    """f16 geometries pass validation (workspace sizes are computed without a
    GPU on the SIMT plan); the cache appends refuse an f16 cache before any
    launch."""
    d = N.MlaDims(4, 16, 8, 16, 32, 1, 16, N.MLA_F16)
    assert N.mla_decode_workspace_size(2, 4, d) > 0
    odd = N.MlaDims(4, 16, 4, 16, 32, 1, 16, N.MLA_F16)   # 8-byte rope rows
    with pytest.raises(N.MlaError):
        N.mla_absorb_q(16, 16, 16, 16, 1, odd, 0)
    with pytest.raises(N.MlaError) as e:
        N.mla_cache_append(256, 512, 768, 1024, 4, 2, N.MLA_F32, d, None, 0)
    assert e.value.status == 2 and "f16" in N.mla_last_error()
    with pytest.raises(N.MlaError) as e:
        N.mla_cache_append_rmsnorm_rope(256, 512, 768, 1024, 1280, 1536, 4, 2, N.MLA_F32,
                                        1e-6, 10000.0, d, None, 0)
    assert e.value.status == 2
    bad = N.MlaDims(4, 16, 8, 16, 32, 1, 16, 3)            # no such dtype
    with pytest.raises(N.MlaError):
        N.mla_decode_workspace_size(2, 4, bad)


def test_cache_append_rmsnorm_rope_validation(lib):
    """Argument checks of the fused append, all before any launch."""
    d = N.MlaDims(4, 16, 8, 16, 32, 1, 16, N.MLA_BF16)
    f = N.mla_cache_append_rmsnorm_rope
    ok = dict(eps=1e-6, rope_base=10000.0)
    # (cache, kv_c, k_pe, gamma, positions, slots): fake aligned addresses, never read
    a = (256, 512, 768, 1024, 1280, 1536)
    with pytest.raises(N.MlaError):
        f(*a, 4, 2, N.MLA_F32, -1.0, 10000.0, d, None, 0)             # eps < 0
    with pytest.raises(N.MlaError):
        f(*a, 4, 2, N.MLA_F32, float("nan"), 10000.0, d, None, 0)     # eps NaN
    with pytest.raises(N.MlaError):
        f(*a, 4, 2, N.MLA_F32, 1e-6, 0.0, d, None, 0)                 # rope_base <= 0
    with pytest.raises(N.MlaError):
        f(256, 512, 768, 0, 1280, 1536, 4, 2, N.MLA_F32, ok["eps"], ok["rope_base"], d, None, 0)  # gamma
    with pytest.raises(N.MlaError):
        f(256, 512, 768, 1024, 0, 1536, 4, 2, N.MLA_F32, ok["eps"], ok["rope_base"], d, None, 0)  # positions
    with pytest.raises(N.MlaError):
        f(256, 512, 768, 1032, 1280, 1536, 4, 2, N.MLA_F32, ok["eps"], ok["rope_base"], d, None, 0)  # gamma misaligned
    with pytest.raises(N.MlaError):
        f(256, 512, 768, 1024, 1284, 1536, 4, 2, N.MLA_F32, ok["eps"], ok["rope_base"], d, None, 0)  # positions misaligned
    odd = N.MlaDims(4, 16, 4, 16, 32, 1, 16, N.MLA_BF16)     # 4 rope elements: not a 16-byte row
    with pytest.raises(N.MlaError):
        f(*a, 4, 2, N.MLA_F32, ok["eps"], ok["rope_base"], odd, None, 0)
    f(0, 0, 0, 0, 0, 0, 0, 2, N.MLA_F32, ok["eps"], ok["rope_base"], d, None, 0)  # no tokens: no-op
    nope = N.MlaDims(4, 16, 0, 16, 32, 1, 16, N.MLA_BF16)
    f(0, 0, 0, 0, 0, 0, 0, 2, N.MLA_F32, ok["eps"], 0.0, nope, None, 0)  # rope_base unused without rope


def test_prolog_q_validation(lib):
    """Argument checks of the query prolog, all before any launch: the query
    rank, eps, the rope base and d_rope's parity, NULL and misaligned buffers;
    zero rows is a no-op."""
    d = N.MlaDims(4, 16, 8, 16, 32, 1, 16, N.MLA_BF16)
    f = N.mla_prolog_q
    ok = dict(q_abs=256, c_q=512, gamma_q=768, w_uq=1024, w_qr=1280, w_uk=1536, positions=1792)

    def call(rows=2, q_rank=64, eps=1e-6, rope_base=10000.0, dims=d, **kw):
        a = dict(ok, **kw)
        f(a["q_abs"], a["c_q"], a["gamma_q"], a["w_uq"], a["w_qr"], a["w_uk"], a["positions"],
          rows, q_rank, eps, rope_base, dims, None, 0)

    for bad in (dict(q_rank=0), dict(q_rank=12), dict(q_rank=16392), dict(rows=-1),
                dict(eps=-1.0), dict(eps=float("nan")), dict(rope_base=0.0),
                dict(rope_base=float("inf")), dict(q_abs=0), dict(w_uk=0), dict(positions=0),
                dict(w_qr=0), dict(c_q=520), dict(positions=1796)):
        with pytest.raises(N.MlaError) as e:
            call(**bad)
        assert e.value.status == 1, bad
    with pytest.raises(N.MlaError):
        call(dims=N.MlaDims(4, 16, 7, 16, 32, 1, 16, N.MLA_BF16))  # odd d_rope
    nope = N.MlaDims(4, 16, 0, 16, 32, 1, 16, N.MLA_BF16)
    call(rows=0, dims=nope, w_qr=0, positions=0)      # no rows, no rope: nothing to do
    call(rows=0)                                      # no rows: a no-op before the pointers


def test_static_decode_refuses_oversize_batch(lib):
    """mla_decode_paged_static compares the batch's scratch need with its
    fixed device array before touching the device: too large a batch is an
    argument error naming both sizes; an empty batch is a no-op."""
    d = N.MlaDims(4, 16, 8, 16, 32, 1, 16, N.MLA_F32)
    limit = 64 << 20  # MLA_STATIC_SCRATCH_BYTES
    batch = 4096
    while N.mla_decode_workspace_size(batch, 4096, d) <= limit:
        batch *= 2
    with pytest.raises(N.MlaError) as e:
        N.mla_decode_paged_static(256, 0, 256, 256, 256, 256, batch, 4096, 8, d, 0.2, None, 0)
    assert e.value.status == 1 and "static scratch" in N.mla_last_error()
    N.mla_decode_paged_static(0, 0, 0, 0, 0, 0, 0, 4, 8, d, 0.2, None, 0)


def test_attend_validation(lib):
    """Argument checks of the fused step, before any launch."""
    d = N.MlaDims(4, 16, 8, 16, 32, 1, 16, N.MLA_F32)
    n = N.mla_attend_workspace_size(2, 4, d)
    args = dict(out=256, lse=0, q_nope=512, q_pe=768, w_uk=1024, w_uv=1280, kv_cache=1536,
                block_table=1792, seq_lens=2048, workspace=4096)

    def call(batch=2, scale=0.2, nbytes=n, **kw):
        a = dict(args, **kw)
        N.mla_attend_absorbed(a["out"], a["lse"], a["q_nope"], a["q_pe"], a["w_uk"], a["w_uv"],
                              a["kv_cache"], a["block_table"], a["seq_lens"], batch, 4, 8, d,
                              scale, a["workspace"], nbytes, None, 0)

    for bad in (dict(batch=-1), dict(out=0), dict(q_pe=0), dict(workspace=0),
                dict(q_nope=520), dict(workspace=4112), dict(scale=float("nan")),
                dict(nbytes=n - 1)):
        with pytest.raises(N.MlaError) as e:
            call(**bad)
        assert e.value.status == 1, bad
    call(batch=0)  # empty batch: nothing to do
