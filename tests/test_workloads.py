"""Host-side checks of the seeded input generator (no GPU)."""
import numpy as np
import pytest

from mla_latent_cache_absorbed_gb300 import workloads as W


def test_tiny_workload_layout():
    wl = W.make_workload("tiny_f32")
    g = wl.geom
    assert list(wl.seq_lens) == [37, 64]
    assert wl.kv_cache.dtype == np.float32 and wl.kv_cache.shape[1:] == (16, g.width)
    assert abs(wl.scale - 1 / np.sqrt(24)) < 1e-12
    # every needed block is distinct and inside the pool; the rest is -1
    used = []
    for b, s in enumerate(wl.seq_lens):
        n = -(-int(s) // 16)
        assert np.all(wl.block_table[b, n:] == -1)
        used += list(wl.block_table[b, :n])
    assert len(set(used)) == len(used) and all(0 <= u < wl.num_blocks for u in used)
    # the tail of request 0's last block is poisoned, its live rows are not
    last = wl.block_table[0, 2]
    assert np.all(wl.kv_cache[last, 5:] == np.float32(1e30))
    assert np.all(np.abs(wl.kv_cache[last, :5]) < 1e3)
    # latent rows are RMS-normalised
    rows = wl.kv_cache[wl.block_table[0, 0], :, :g.kv_rank].astype(np.float64)
    assert np.allclose(np.mean(rows * rows, axis=1), 1.0, atol=1e-4)


def test_seeded_and_reproducible():
    a = W.make_workload("tiny_f32")
    b = W.make_workload("tiny_f32")
    assert np.array_equal(a.kv_cache, b.kv_cache) and np.array_equal(a.q_nope, b.q_nope)
    c = W.make_workload("tiny_f32", seed=5)
    assert not np.array_equal(a.q_nope, c.q_nope)


def test_bf16_values_are_exact_bf16():
    wl = W.make_workload("glm52_decode", seq_lens=[5, 0, 40])
    for a in (wl.q_nope, wl.q_pe, wl.w_uk, wl.w_uv):
        bits = a.view(np.uint32)
        assert np.all((bits & 0xFFFF) == 0)
    assert wl.kv_cache.dtype == np.uint16
    assert wl.block_table[1, 0] == -1


@pytest.mark.parametrize("name", ["glm52_decode", "glm52_causal_t4", "glm52_prefill_chunk"])
def test_rope_positions(name):
    """Roped query/key dot products depend only on the position difference."""
    wl = W.make_workload(name, seq_lens=[20, 33], poison="none")
    g = wl.geom
    P = g.d_rope
    rng = np.random.default_rng(0)
    x = rng.standard_normal(P)
    y = rng.standard_normal(P)
    rope = W.apply_rope_neox if wl.rope == "neox" else W.apply_rope_interleaved
    d1 = rope(x, np.array(7.0), 10000.0) @ rope(y, np.array(3.0), 10000.0)
    d2 = rope(x, np.array(104.0), 10000.0) @ rope(y, np.array(100.0), 10000.0)
    assert abs(d1 - d2) < 1e-9


def test_norm_workload_neox_side_keeps_dot_products():
    """The permuted-NEOX copy of the rope columns gives the same q.k dot
    products as the interleaved original (the load-time permutation fact)."""
    wl = W.make_workload("glm52_causal_t4", seq_lens=[9, 20], poison="none")
    P = wl.geom.d_rope
    perm = np.empty(P, np.int64)
    perm[0::2] = np.arange(P // 2)
    perm[1::2] = np.arange(P // 2) + P // 2

    def permute(a):
        tmp = a.copy()
        a[:, perm] = tmp

    k_neox, q_neox = W.neox_side_rope_columns(wl, permute)
    R = wl.geom.kv_rank
    k_norm = W.bits_to_f32(wl.kv_cache[..., R:]).astype(np.float64)
    b, t, h = 1, 3, 5
    q_norm = wl.q_pe[b * 4 + t, h].astype(np.float64)
    qn = q_neox[b * 4 + t, h].astype(np.float64)
    blk = wl.block_table[b, 0]
    for j in range(16):
        d_norm = q_norm @ k_norm[blk, j]
        d_neox = qn @ k_neox[blk, j].astype(np.float64)
        # both sides hold bf16-rounded values (relative error <= 2^-9 each)
        bound = 2 ** -7 * (np.abs(q_norm) @ np.abs(k_norm[blk, j]))
        assert abs(d_norm - d_neox) <= bound


def test_default_seq_len_recipes():
    rng = np.random.default_rng(1)
    s = W.default_seq_lens("glm52_decode", rng)
    assert s.shape == (8,) and s[3] == 0 and np.all(s[[0, 1, 2, 4, 5, 6, 7]] >= 1)
    s = W.default_seq_lens("glm53_flash_nope", np.random.default_rng(3))
    assert s.shape == (128,) and s.min() >= 1 and s.max() <= 32768
    assert 1000 < np.median(s) < 4000
    s = W.default_seq_lens("glm52_causal_t4", np.random.default_rng(4))
    assert s.min() >= 8192 and s.max() <= 65536
    s = W.default_seq_lens("glm52_prefill_chunk", np.random.default_rng(5))
    assert s.shape == (4,) and s[0] == 128 and s[1:].min() >= 129 and s.max() <= 8192
