"""Parity of mla_cache_append_rmsnorm_rope (through the C ABI) with the
oracle's restatement of the key formulas of the "aclnnMlaProlog" page:
c^KV = RmsNorm(latent) and k^R = ROPE(k_pe), stored by slot mapping.

The kernel computes in f32; the oracle takes the norm in f64 and the rope in
the mla.rs page's f32 (theta stepped from the position by the f32 factor
base^(-2/P), the same products on both sides). Tolerances, from that
arithmetic:
  * norm elements: the kernel's f32 error is below 2e-6 relative (a 16-term
    fma chain plus a 5-step butterfly for the sum of squares, then four
    roundings); f32 cache |got - ref| <= 4e-6 |ref|, bf16 cache adds the
    cast's half ulp: <= (2^-8 + 1e-5) |ref|;
  * rope elements: theta is the same f32 number on both sides, so the
    difference comes from sin/cos (a few f32 ulps each) and the roundings of
    the rotation: f32 cache |got - ref| <= 1e-6 (|a| + |b|) for the pair
    (a, b), bf16 cache adds 2^-8 |ref|.
Bytes of rows that no token writes (padding, unused slots) must keep their
poison pattern exactly.
"""
import numpy as np
import pytest

import oracle
from mla_latent_cache_absorbed_gb300 import _native as N

pytestmark = pytest.mark.gpu

F32, BF16 = 0, 1


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    assert torch.cuda.is_available()
    N.load()


def dims_for(R, P, cache_dtype):
    return N.MlaDims(1, 64, P, 64, R, 1, 16, cache_dtype)


def to_bits(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def from_bits(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


def dev(a):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16)
    return t.cuda()


def run_case(R, P, num_blocks, n, src_dtype, cache_dtype, seed, positions=None, pad_frac=0.2,
             bad_slot=False, eps=1e-6, base=10000.0, zero_rows=0):
    import torch
    rng = np.random.default_rng(seed)
    W = R + P
    kv = (rng.standard_normal((n, R)) * rng.uniform(0.1, 20.0, (n, 1))).astype(np.float32)
    kv[:zero_rows] = 0.0
    kp = (rng.standard_normal((n, P)) * 2).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, R).astype(np.float32)
    if positions is None:
        positions = rng.integers(0, 200000, size=n)
    positions = np.asarray(positions, np.int64)
    slots = rng.choice(num_blocks * 16, size=n, replace=False).astype(np.int64)
    slots[rng.random(n) < pad_frac] = -1
    if bad_slot:
        slots[n // 2] = num_blocks * 16 + 3
    if src_dtype == BF16:
        kv_h, kp_h, g_h = to_bits(kv), to_bits(kp), to_bits(gamma)
        kv_v, kp_v = from_bits(kv_h), from_bits(kp_h)
    else:
        kv_h, kp_h, g_h = kv, kp, gamma
        kv_v, kp_v = kv, kp
    if cache_dtype == BF16:
        cache_h = rng.integers(0, 2 ** 16, size=(num_blocks, 16, W), dtype=np.uint16) & 0x7f7f
    else:
        cache_h = rng.standard_normal((num_blocks, 16, W)).astype(np.float32)

    cache_d = dev(cache_h)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    N.mla_cache_append_rmsnorm_rope(cache_d, dev(kv_h), dev(kp_h) if P else None, dev(g_h),
                                    dev(positions) if P else None, dev(slots), n, num_blocks,
                                    src_dtype, eps, base, dims_for(R, P, cache_dtype), dev_err)
    torch.cuda.synchronize()
    got = cache_d.cpu().numpy()
    if cache_dtype == BF16:
        got = got.view(np.uint16)
    assert int(dev_err.item()) == (16 if bad_slot else 0)

    flat_got = got.reshape(-1, W)
    flat_poison = cache_h.reshape(-1, W)
    live = (slots >= 0) & (slots < num_blocks * 16)
    untouched = np.setdiff1d(np.arange(num_blocks * 16), slots[live])
    assert np.array_equal(flat_got[untouched].view(np.uint8), flat_poison[untouched].view(np.uint8))

    toks = np.nonzero(live)[0]
    rows = oracle.kv_prolog_rows(kv_h[toks], kp_h[toks] if P else None, g_h,
                                 positions[toks] if P else None, eps, base)
    out = flat_got[slots[toks]]
    out = from_bits(out).astype(np.float64) if cache_dtype == BF16 else out.astype(np.float64)
    cast = 2.0 ** -8 if cache_dtype == BF16 else 0.0
    ref_n = rows[:, :R]
    err_n = np.abs(out[:, :R] - ref_n)
    tol_n = (cast + (1e-5 if cast else 4e-6)) * np.abs(ref_n)
    assert np.all(err_n <= tol_n), f"norm: worst excess {(err_n - tol_n).max():.3e}"
    if zero_rows:
        assert np.all(out[np.isin(toks, np.arange(zero_rows)), :R] == 0.0)
    if P:
        h = P // 2
        pair = np.abs(kp_v[toks]).astype(np.float64)
        pair = np.concatenate([pair[:, :h] + pair[:, h:]] * 2, axis=1)
        ref_r = rows[:, R:]
        err_r = np.abs(out[:, R:] - ref_r)
        tol_r = cast * np.abs(ref_r) + (2e-6 if cast else 1e-6) * pair
        assert np.all(err_r <= tol_r), f"rope: worst excess {(err_r - tol_r).max():.3e}"
    return rows, out


@pytest.mark.parametrize("src_dtype,cache_dtype", [(F32, F32), (F32, BF16), (BF16, BF16), (BF16, F32)],
                         ids=["f32->f32", "f32->bf16", "bf16->bf16", "bf16->f32"])
def test_small_geometry(src_dtype, cache_dtype):
    run_case(32, 8, 7, 50, src_dtype, cache_dtype, seed=1, zero_rows=2)


@pytest.mark.parametrize("src_dtype", [F32, BF16], ids=["from f32", "from bf16"])
def test_glm_rows_decode_step(src_dtype):
    """One new token per request of a 64-request batch, 576-wide rows, long
    context positions (up to 200k)."""
    run_case(512, 64, 2000, 64, src_dtype, BF16, seed=2)


def test_glm_rows_prefill_chunk():
    """The benchmark's chunk launch: 32768 consecutive positions of one
    prefill chunk, bf16 in, bf16 cache."""
    run_case(512, 64, 2500, 32768, BF16, BF16, seed=3, positions=np.arange(32768) + 1000,
             pad_frac=0.02)


def test_position_extremes():
    """Positions 0 (the rope is the identity: rope elements equal the cast
    input), 1, and up to 2^24 - 1 (the largest exactly held in f32)."""
    pos = np.array([0, 0, 1, 2, 65535, 2 ** 20, 2 ** 24 - 1, 123457], np.int64)
    rows, out = run_case(512, 64, 10, 8, F32, F32, seed=5, positions=pos, pad_frac=0.0)
    rng = np.random.default_rng(5)   # the inputs run_case drew
    rng.standard_normal((8, 512))
    rng.uniform(0.1, 20.0, (8, 1))
    kp = (rng.standard_normal((8, 64)) * 2).astype(np.float32)
    assert np.array_equal(out[:2, 512:], kp[:2].astype(np.float64))


def test_nope_rows_no_rope_plane():
    """The NoPE geometry (P = 0): the norm alone, k_pe and positions NULL."""
    run_case(512, 0, 300, 1000, BF16, BF16, seed=6, pad_frac=0.1)


def test_eps_dominates_small_rows():
    """eps far above mean(x^2): the rows shrink by 1/sqrt(eps)."""
    run_case(64, 16, 5, 40, F32, F32, seed=7, eps=1e4)


def test_slot_past_cache_is_flagged_and_skipped():
    run_case(512, 64, 100, 40, F32, BF16, seed=8, bad_slot=True)


def test_no_tokens_is_a_no_op():
    import torch
    cache = torch.zeros(4, 16, 576, dtype=torch.bfloat16, device="cuda")
    N.mla_cache_append_rmsnorm_rope(cache, None, None, None, None, None, 0, 4, F32, 1e-6, 1e4,
                                    dims_for(512, 64, BF16))
    torch.cuda.synchronize()
    assert int(cache.abs().sum().item()) == 0
