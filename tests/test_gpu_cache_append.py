"""Parity of the cache append (mla_cache_append, through the C ABI) with the
oracle's restatement of the vLLM CPU MLA page's do_kv_cache_update.

This is byte work: every cache byte must equal the oracle's, bit for bit
(the f32 -> bf16 cast rounds to nearest, ties to even, on both sides). The
inputs are seeded and NaN-free; untouched cache rows hold a seeded poison
pattern that must survive.
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
    # n_head, d_nope, d_rope, d_v, kv_rank, t_q, block_size, dtype (only the
    # cache geometry matters to the append)
    return N.MlaDims(1, 64, P, 64, R, 1, 16, cache_dtype)


def to_bits(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def run_case(R, P, num_blocks, n, src_dtype, cache_dtype, seed, pad_frac=0.2, bad_slot=False):
    import torch
    rng = np.random.default_rng(seed)
    W = R + P
    kv = rng.standard_normal((n, R)).astype(np.float32) * 3
    kp = rng.standard_normal((n, P)).astype(np.float32) * 3
    # a few exact bf16 ties and signed zeros in the f32 sources
    if n > 2 and R >= 4:
        kv[0, :4] = np.array([0x3f808000, 0x3f818000, 0xbf808000, 0x80000000], np.uint32).view(np.float32)
    slots = rng.choice(num_blocks * 16, size=n, replace=False).astype(np.int64)
    slots[rng.random(n) < pad_frac] = -1
    if bad_slot:
        slots[n // 2] = num_blocks * 16 + 3
    if src_dtype == BF16:
        kv_h, kp_h = to_bits(kv), to_bits(kp)
    else:
        kv_h, kp_h = kv, kp
    if cache_dtype == BF16:
        cache_h = rng.integers(0, 2 ** 16, size=(num_blocks, 16, W), dtype=np.uint16)
        cache_h &= 0x7f7f  # keep the poison finite
    else:
        cache_h = rng.standard_normal((num_blocks, 16, W)).astype(np.float32)
    ref = oracle.cache_append(cache_h, kv_h, kp_h, slots, allow_errors=bad_slot)

    def dev(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.int16)
        return t.cuda()

    cache_d = dev(cache_h)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    N.mla_cache_append(cache_d, dev(kv_h), dev(kp_h) if P else None, dev(slots), n, num_blocks,
                       src_dtype, dims_for(R, P, cache_dtype), dev_err)
    torch.cuda.synchronize()
    got = cache_d.cpu().numpy()
    if cache_dtype == BF16:
        got = got.view(np.uint16)
    assert np.array_equal(got.view(np.uint8), ref.view(np.uint8)), \
        f"{int((got != ref).sum())} cache elements differ"
    assert int(dev_err.item()) == (16 if bad_slot else 0)


@pytest.mark.parametrize("src_dtype,cache_dtype", [(F32, F32), (F32, BF16), (BF16, BF16), (BF16, F32)],
                         ids=["f32->f32", "f32->bf16", "bf16->bf16", "bf16->f32"])
def test_small_geometry(src_dtype, cache_dtype):
    run_case(32, 8, 7, 50, src_dtype, cache_dtype, seed=1)


@pytest.mark.parametrize("src_dtype", [F32, BF16], ids=["from f32", "from bf16"])
def test_glm_rows_decode_step(src_dtype):
    """One new token per request of a 64-request batch, 576-wide rows."""
    run_case(512, 64, 2000, 64, src_dtype, BF16, seed=2)


def test_nope_rows_prefill_chunk():
    """A prefill-sized append: 32768 tokens of 512-wide rows (no rope plane)."""
    run_case(512, 0, 2500, 32768, F32, BF16, seed=3, pad_frac=0.05)


def test_slot_past_cache_is_flagged_and_skipped():
    run_case(512, 64, 100, 40, F32, BF16, seed=4, bad_slot=True)


def test_no_tokens_is_a_no_op():
    import torch
    cache = torch.zeros(4, 16, 576, dtype=torch.bfloat16, device="cuda")
    N.mla_cache_append(cache, None, None, None, 0, 4, F32, dims_for(512, 64, BF16))
    torch.cuda.synchronize()
    assert int(cache.abs().sum().item()) == 0
