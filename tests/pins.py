"""Pins that tie the CPU oracle to facts outside itself.

Each ``check_*`` function takes an oracle library handle (the real one, or a
deliberately broken copy built by ``test_oracle_mutants.py``) and raises
AssertionError when the oracle disagrees with:
  * the other of the two forms the memra mla.rs source proves equal
    (naive per-head decompression vs the absorbed form, fns mla_attend_naive
    and mla_attend_absorbed);
  * brute force in f64 on tiny inputs, and torch's scaled-dot-product
    attention (a library routine that the T=1 decode reduces to);
  * closed forms (empty request, one key, identical keys, zero scale, a
    hand-worked two-key example stored under tests/golden/);
  * structural invariants (split + LSE combine equals the unsplit result;
    paged equals contiguous; unused rows never read);
  * the rope facts of the mla.rs rope section (interleaved rope followed by
    the load-time permutation equals the permutation followed by NEOX rope,
    and roped dot products agree), and the scale of the NoPE geometry;
  * the cache append of the vLLM CPU MLA page (do_kv_cache_update): rows land
    at their slots unchanged (f32) or as torch's bf16 cast of them, padding
    slots are skipped, other rows keep their bits, a slot past the cache is
    reported;
  * the KV half of the MLA prolog of the "aclnnMlaProlog" page (RmsNorm of
    the latent, rope of k^R at each token's position, then the same scatter):
    closed forms of the norm and an f64 rotation for the rope;
  * the query half of the MLA prolog: the absorb with the query's rope at
    each row's position, the same rotation as the key half's;
  * chunked causal prefill: a block of queries per request is causal
    attention (torch's SDPA with a causal mask), and each of its queries the
    one-query decode of the request cut at that query's position.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------ helpers
def random_case(rng, H, Dn, P, Dv, R, t_q, t_kv):
    """Inputs with the workloads' value recipe: queries, latent rows and rope
    parts ~ N(0, 1), weights ~ N(0, sd = 1/sqrt(kv_rank)), as f32. Returns
    (q_nope [t_q,H,Dn], q_pe [t_q,H,P], c_kv [t_kv,R], k_pe [t_kv,P], w_uk, w_uv)."""
    g = lambda *shape, sd=1.0: (rng.standard_normal(shape) * sd).astype(np.float32)
    sd = 1.0 / math.sqrt(R)
    return (g(t_q, H, Dn), g(t_q, H, P), g(t_kv, R), g(t_kv, P), g(H, Dn, R, sd=sd),
            g(H, Dv, R, sd=sd))


def maxdiff(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))


def rel_ok(ref, got, tol):
    scale = max(float(np.max(np.abs(ref))), 1.0)
    return maxdiff(ref, got) <= tol * scale


def page(rows_f32, seq_lens, rng, bs=16, spare=3, poison=1e30):
    """Scatter per-request contiguous rows into a shuffled paged pool.

    rows_f32: list of [S_b, W] arrays. Returns (cache, block_table)."""
    nblk = [-(-r.shape[0] // bs) for r in rows_f32]
    W = rows_f32[0].shape[1] if rows_f32 else 1
    pool = sum(nblk) + spare
    perm = rng.permutation(pool).astype(np.int32)
    cache = np.full((pool, bs, W), poison, np.float32)
    bt = np.full((len(rows_f32), max(1, max(nblk) if nblk else 1)), -1, np.int32)
    k = 0
    for b, r in enumerate(rows_f32):
        for i in range(nblk[b]):
            blk = perm[k]
            k += 1
            bt[b, i] = blk
            chunk = r[i * bs:(i + 1) * bs]
            cache[blk, :chunk.shape[0]] = chunk
    return cache, bt


# ------------------------------------------------------------------ pins
# the two forms must agree relative to max(max |out|, 1): to 1e-5 on small
# shapes and to 1e-4 at full model dims, the two gates the mla.rs unit tests
# set for naive against absorbed (its small-shape cases and its full-dims
# cases respectively)
FORMS_RTOL = 1e-5
FORMS_RTOL_FULL_DIMS = 1e-4


def check_naive_equals_absorbed(lib):
    """Both forms of mla.rs (per-head decompression, then ordinary attention;
    the absorbed form) agree on small shapes chosen to vary the proportions:
    rope wider than nope, d_v above and below kv_rank, a single head, NoPE;
    for one query and for causal blocks of queries, including t_q == t_kv."""
    rng = np.random.default_rng(4242)
    shapes = [(5, 20, 12, 28, 56), (2, 8, 24, 8, 40), (3, 28, 4, 36, 24),
              (1, 12, 16, 12, 16), (4, 40, 0, 20, 72), (2, 24, 0, 48, 32)]
    for (H, Dn, P, Dv, R) in shapes:
        for (t_q, t_kv) in [(1, 23), (6, 14), (4, 4), (2, 31)]:
            args = random_case(rng, H, Dn, P, Dv, R, t_q, t_kv)
            scale = 1.0 / math.sqrt(Dn + P)
            a = oracle.attend_naive(*args, scale, lib=lib)
            b = oracle.attend_absorbed(*args, scale, lib=lib)
            assert np.all(np.isfinite(a)) and float(np.max(np.abs(a))) > 1e-6
            assert rel_ok(a, b, FORMS_RTOL), (H, Dn, P, Dv, R, t_q, t_kv, maxdiff(a, b))


def check_naive_equals_absorbed_full_dims(lib):
    """The same at the full GLM-5.2 (64 heads, 192/64/256, rank 512) and
    GLM-5.3-Flash NoPE (64 heads, 256/0/256, rank 512) geometries."""
    rng = np.random.default_rng(5150)
    for (H, Dn, P, Dv, R, t_q, t_kv) in [(64, 192, 64, 256, 512, 1, 12),
                                          (64, 192, 64, 256, 512, 3, 7),
                                          (64, 256, 0, 256, 512, 1, 10),
                                          (64, 256, 0, 256, 512, 5, 5)]:
        args = random_case(rng, H, Dn, P, Dv, R, t_q, t_kv)
        scale = 1.0 / math.sqrt(Dn + P)
        a = oracle.attend_naive(*args, scale, lib=lib)
        b = oracle.attend_absorbed(*args, scale, lib=lib)
        assert rel_ok(a, b, FORMS_RTOL_FULL_DIMS), (H, Dn, P, maxdiff(a, b))


def _chain(lib, q_nope, q_pe, w_uk, w_uv, cache, bt, seq_lens, t_q, R, scale):
    B = seq_lens.shape[0]
    H = q_nope.shape[1]
    q_abs = oracle.absorb_q(q_nope, q_pe, w_uk, lib=lib)
    o, lse = oracle.decode_paged(q_abs.reshape(B, t_q, H, -1), cache, bt, seq_lens, t_q,
                                 R, scale, lib=lib)
    out = oracle.decompress(o.reshape(B * t_q, H, R), w_uv, lib=lib)
    return q_abs, o, lse, out


def check_paged_chain_equals_naive(lib):
    """absorb -> paged decode (shuffled blocks, poisoned spare rows) ->
    decompress equals the naive form on each request's contiguous cache."""
    rng = np.random.default_rng(11)
    for (H, Dn, P, Dv, R, t_q, lens) in [(4, 16, 8, 16, 32, 1, [37, 64, 5]),
                                         (3, 20, 12, 28, 40, 3, [19, 3, 33]),
                                         (2, 16, 0, 24, 32, 2, [17, 40])]:
        W = R + P
        B = len(lens)
        scale = 1.0 / math.sqrt(Dn + P)
        per_req = [random_case(rng, H, Dn, P, Dv, R, t_q, s) for s in lens]
        w_uk, w_uv = per_req[0][4], per_req[0][5]
        rows = [np.concatenate([c[2], c[3]], axis=1) for c in per_req]
        cache, bt = page(rows, np.array(lens), rng)
        q_nope = np.concatenate([c[0] for c in per_req])
        q_pe = np.concatenate([c[1] for c in per_req])
        sl = np.array(lens, np.int32)
        _, _, _, out = _chain(lib, q_nope, q_pe, w_uk, w_uv, cache, bt, sl, t_q, R, scale)
        out = out.reshape(B, t_q, H, Dv)
        for b, c in enumerate(per_req):
            ref = oracle.attend_naive(c[0], c[1], c[2], c[3], w_uk, w_uv, scale, lib=lib)
            assert rel_ok(ref, out[b], 2e-5), (H, Dn, P, b, maxdiff(ref, out[b]))


def _bruteforce(q_abs_row, rows, R, scale):
    s = (rows.astype(np.float64) @ q_abs_row.astype(np.float64)) * scale
    m = s.max()
    e = np.exp(s - m)
    o = (e[:, None] * rows[:, :R].astype(np.float64)).sum(0) / e.sum()
    return o, m + math.log(e.sum())


def check_bruteforce_f64(lib):
    """Direct f64 softmax over every visible row agrees with the single-pass
    f32 decode, including causal rows and a request whose keys start in the
    middle of a block table."""
    rng = np.random.default_rng(3)
    H, R, P, t_q = 3, 32, 8, 3
    W = R + P
    lens = [1, 16, 17, 50]
    rows = [rng.standard_normal((s, W)).astype(np.float32) for s in lens]
    cache, bt = page(rows, lens, rng)
    q = rng.standard_normal((len(lens), t_q, H, W)).astype(np.float32)
    sl = np.array(lens, np.int32)
    scale = 0.3
    lens_ok = [s for s in lens if s >= t_q]
    o, lse, st = oracle.decode_paged(q, cache, bt, sl, t_q, R, scale, lib=lib,
                                     allow_errors=True)
    for b, s in enumerate(lens):
        for t in range(t_q):
            for h in range(H):
                if s < t_q:  # a request shorter than t_q is invalid: empty result
                    assert np.all(o[b, t, h] == 0) and lse[b, t, h] == -np.inf
                    continue
                vis = s - t_q + t + 1
                ro, rl = _bruteforce(q[b, t, h], rows[b][:vis], R, scale)
                assert maxdiff(ro, o[b, t, h]) <= 2e-6 * max(1.0, np.abs(ro).max())
                assert abs(rl - lse[b, t, h]) <= 2e-6 * max(1.0, abs(rl))
    assert st == -4  # the length-1 request is shorter than t_q
    assert lens_ok


def check_sdpa_reduction(lib):
    """For t_q = 1 the decode is ordinary attention with K = the whole row and
    V = its leading kv_rank columns: torch's SDPA (f64) on the gathered rows
    gives the same output, and logsumexp of the scaled scores the same LSE."""
    import torch
    rng = np.random.default_rng(5)
    H, R, P = 4, 32, 8
    W = R + P
    lens = [9, 40]
    rows = [rng.standard_normal((s, W)).astype(np.float32) for s in lens]
    cache, bt = page(rows, lens, rng)
    q = rng.standard_normal((len(lens), 1, H, W)).astype(np.float32)
    scale = 1.0 / math.sqrt(24)
    o, lse = oracle.decode_paged(q, cache, bt, np.array(lens, np.int32), 1, R, scale, lib=lib)
    for b, s in enumerate(lens):
        qt = torch.from_numpy(q[b, 0].astype(np.float64))[None, :, None, :]   # [1,H,1,W]
        kt = torch.from_numpy(rows[b].astype(np.float64))[None, None].expand(1, H, s, W)
        vt = kt[..., :R]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        ref = ref[0, :, 0, :].numpy()
        ref_lse = torch.logsumexp((qt @ kt.transpose(-1, -2))[0, :, 0, :] * scale, -1).numpy()
        assert maxdiff(ref, o[b, 0]) <= 3e-6, maxdiff(ref, o[b, 0])
        assert maxdiff(ref_lse, lse[b, 0]) <= 3e-6


def check_closed_forms(lib):
    """Empty request, one key, identical keys, zero scale, and the hand-worked
    two-key example in tests/golden/closed_form_decode.json."""
    rng = np.random.default_rng(9)
    R, P, H = 16, 4, 2
    W = R + P
    row = rng.standard_normal(W).astype(np.float32)
    one = [row[None, :]]
    same = [np.repeat(row[None, :], 23, 0)]
    mixed = [rng.standard_normal((29, W)).astype(np.float32)]
    q = rng.standard_normal((1, 1, H, W)).astype(np.float32)

    # empty request: zero row, -inf LSE
    cache, bt = page([np.zeros((0, W), np.float32)], [0], rng)
    o, lse = oracle.decode_paged(q, cache, np.full((1, 1), -1, np.int32),
                                 np.array([0], np.int32), 1, R, 0.5, lib=lib)
    assert np.all(o == 0) and np.all(lse == -np.inf)

    # one key: o = row[:R], lse = scale * q.row
    cache, bt = page(one, [1], rng)
    o, lse = oracle.decode_paged(q, cache, bt, np.array([1], np.int32), 1, R, 0.5, lib=lib)
    for h in range(H):
        assert maxdiff(o[0, 0, h], row[:R]) <= 1e-6
        s = 0.5 * float(np.dot(q[0, 0, h].astype(np.float64), row.astype(np.float64)))
        assert abs(lse[0, 0, h] - s) <= 1e-5 * max(1, abs(s))

    # identical keys: o = row[:R], lse = s + ln S
    cache, bt = page(same, [23], rng)
    o, lse = oracle.decode_paged(q, cache, bt, np.array([23], np.int32), 1, R, 0.5, lib=lib)
    for h in range(H):
        assert maxdiff(o[0, 0, h], row[:R]) <= 2e-6 * max(1, np.abs(row).max())
        s = 0.5 * float(np.dot(q[0, 0, h].astype(np.float64), row.astype(np.float64)))
        assert abs(lse[0, 0, h] - (s + math.log(23))) <= 2e-5 * max(1, abs(s))

    # zero scale: uniform weights, o = mean of rows, lse = ln S
    cache, bt = page(mixed, [29], rng)
    o, lse = oracle.decode_paged(q, cache, bt, np.array([29], np.int32), 1, R, 0.0, lib=lib)
    mean = mixed[0][:, :R].astype(np.float64).mean(0)
    for h in range(H):
        assert maxdiff(o[0, 0, h], mean) <= 2e-6
        assert abs(lse[0, 0, h] - math.log(29)) <= 1e-6

    # hand-worked example
    with open(os.path.join(GOLDEN, "closed_form_decode.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        rows = np.array(case["rows"], np.float32)
        Rc = case["kv_rank"]
        qq = np.array(case["q"], np.float32).reshape(1, 1, 1, -1)
        cache, bt = page([rows], [rows.shape[0]], rng, bs=case["block_size"])
        o, lse = oracle.decode_paged(qq, cache, bt, np.array([rows.shape[0]], np.int32), 1,
                                     Rc, case["scale"], lib=lib)
        assert maxdiff(o[0, 0, 0], case["o"]) <= 1e-6, (case["name"], o[0, 0, 0])
        assert abs(lse[0, 0, 0] - case["lse"]) <= 1e-6, (case["name"], lse[0, 0, 0])


def check_split_combine(lib):
    """Any split of the visible keys, merged by LSE, equals the unsplit
    decode; an empty split carries no weight; all-empty gives 0 and -inf."""
    rng = np.random.default_rng(21)
    R, P = 32, 8
    W = R + P
    S = 70
    rows = [rng.standard_normal((S, W)).astype(np.float32)]
    cache, bt = page(rows, [S], rng)
    q = rng.standard_normal(W).astype(np.float32)
    full_o, full_l = oracle.decode_range(q, cache, bt[0], S, 1, 0, R, 0.4, 0, S, lib=lib)
    for cuts in ([0, 35, 70], [0, 1, 2, 70], [0, 16, 16, 48, 70], [0, 69, 70]):
        parts = [oracle.decode_range(q, cache, bt[0], S, 1, 0, R, 0.4, a, b, lib=lib)
                 for a, b in zip(cuts[:-1], cuts[1:])]
        o, l = oracle.combine(np.stack([p[0] for p in parts]),
                              np.array([p[1] for p in parts], np.float32), lib=lib)
        assert maxdiff(o, full_o) <= 2e-6 * max(1, np.abs(full_o).max()), cuts
        assert abs(l - full_l) <= 2e-6 * max(1, abs(full_l)), cuts
    o, l = oracle.combine(np.zeros((2, R), np.float32),
                          np.array([-np.inf, -np.inf], np.float32), lib=lib)
    assert np.all(o == 0) and l == -np.inf


def check_paged_equals_contiguous(lib):
    """The same rows under two different block layouts give bit-identical
    results (same summation order), and unused rows are never read (poison
    1e30 or NaN leaves every bit unchanged)."""
    rng = np.random.default_rng(33)
    R, P, H, t_q = 32, 8, 3, 2
    W = R + P
    lens = [33, 16, 2]
    rows = [rng.standard_normal((s, W)).astype(np.float32) for s in lens]
    q = rng.standard_normal((3, t_q, H, W)).astype(np.float32)
    sl = np.array(lens, np.int32)
    c1, bt1 = page(rows, lens, np.random.default_rng(1), poison=1e30)
    c2, bt2 = page(rows, lens, np.random.default_rng(2), poison=np.nan, spare=9)
    # identity layout: request b's blocks are consecutive
    nb = [-(-s // 16) for s in lens]
    c3 = np.full((sum(nb), 16, W), np.nan, np.float32)
    bt3 = np.full((3, max(nb)), -1, np.int32)
    k = 0
    for b, r in enumerate(rows):
        for i in range(nb[b]):
            ch = r[i * 16:(i + 1) * 16]
            c3[k, :ch.shape[0]] = ch
            bt3[b, i] = k
            k += 1
    outs = [oracle.decode_paged(q, c, bt, sl, t_q, R, 0.25, lib=lib)
            for c, bt in ((c1, bt1), (c2, bt2), (c3, bt3))]
    for o, l in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0][0].view(np.uint32))
        assert np.array_equal(l.view(np.uint32), outs[0][1].view(np.uint32))


def check_decode_rows_consistent(lib):
    """Sampled-row decode returns exactly the rows of the full decode, for
    f32 inputs and for bf16 patterns (whose f32 values are the upper half)."""
    rng = np.random.default_rng(44)
    R, P, H, t_q = 32, 8, 4, 2
    W = R + P
    lens = [20, 7]
    rows = [rng.standard_normal((s, W)).astype(np.float32) for s in lens]
    cache, bt = page(rows, lens, rng)
    q = rng.standard_normal((2, t_q, H, W)).astype(np.float32)
    sl = np.array(lens, np.int32)
    o, l = oracle.decode_paged(q, cache, bt, sl, t_q, R, 0.2, lib=lib)
    ids = np.array([0, 5, 9, 15], np.int64)
    so, sl_ = oracle.decode_rows(q, cache, bt, sl, t_q, R, 0.2, ids, lib=lib)
    assert np.array_equal(so, o.reshape(-1, R)[ids])
    assert np.array_equal(sl_, l.reshape(-1)[ids])
    # bf16 patterns: truncating to the upper half gives exact bf16 values
    qb = (q.view(np.uint32) >> 16).astype(np.uint16)
    cb = (cache.view(np.uint32) >> 16).astype(np.uint16)
    qf = (qb.astype(np.uint32) << 16).view(np.float32)
    cf = (cb.astype(np.uint32) << 16).view(np.float32)
    ob, lb = oracle.decode_paged(qb, cb, bt, sl, t_q, R, 0.2, lib=lib)
    of, lf = oracle.decode_paged(qf, cf, bt, sl, t_q, R, 0.2, lib=lib)
    assert np.array_equal(ob, of) and np.array_equal(lb, lf)


def check_invalid_requests(lib):
    """Out-of-range block ids, a seq_len beyond the block-table row and a
    non-empty request shorter than t_q are reported and give empty rows."""
    rng = np.random.default_rng(55)
    R, P = 16, 0
    rows = [rng.standard_normal((20, R)).astype(np.float32)]
    cache, bt = page(rows, [20], rng)
    q = rng.standard_normal((1, 1, 1, R)).astype(np.float32)
    bad = bt.copy()
    bad[0, 1] = cache.shape[0]  # one past the pool
    o, l, st = oracle.decode_paged(q, cache, bad, np.array([20], np.int32), 1, R, 1.0,
                                   lib=lib, allow_errors=True)
    assert st == -2 and np.all(o == 0) and l[0, 0, 0] == -np.inf
    o, l, st = oracle.decode_paged(q, cache, bt, np.array([33], np.int32), 1, R, 1.0,
                                   lib=lib, allow_errors=True)
    assert st == -3 and np.all(o == 0)
    q2 = rng.standard_normal((1, 4, 1, R)).astype(np.float32)
    o, l, st = oracle.decode_paged(q2, cache, bt, np.array([3], np.int32), 4, R, 1.0,
                                   lib=lib, allow_errors=True)
    assert st == -4 and np.all(o == 0)


def check_absorb_decompress_unit_weights(lib):
    """With unit-vector weights the absorb copies q_nope into rank space and
    the decompress picks single latent coordinates; the rope tail of q_abs is
    q_pe itself."""
    rng = np.random.default_rng(66)
    H, Dn, R, P, Dv, rows = 3, 8, 12, 4, 5, 2
    perm = [rng.permutation(R)[:Dn] for _ in range(H)]
    w_uk = np.zeros((H, Dn, R), np.float32)
    for h in range(H):
        w_uk[h, np.arange(Dn), perm[h]] = 1.0
    q_nope = rng.standard_normal((rows, H, Dn)).astype(np.float32)
    q_pe = rng.standard_normal((rows, H, P)).astype(np.float32)
    qa = oracle.absorb_q(q_nope, q_pe, w_uk, lib=lib)
    for h in range(H):
        expect = np.zeros((rows, R), np.float32)
        expect[:, perm[h]] = q_nope[:, h]
        assert np.array_equal(qa[:, h, :R], expect)
        assert np.array_equal(qa[:, h, R:], q_pe[:, h])
    sel = [rng.integers(0, R, size=Dv) for _ in range(H)]
    w_uv = np.zeros((H, Dv, R), np.float32)
    for h in range(H):
        w_uv[h, np.arange(Dv), sel[h]] = 2.0
    o_lat = rng.standard_normal((rows, H, R)).astype(np.float32)
    out = oracle.decompress(o_lat, w_uv, lib=lib)
    for h in range(H):
        assert np.array_equal(out[:, h], 2.0 * o_lat[:, h][:, sel[h]])


def check_rope_permutation(lib):
    """The load-time permutation of the mla.rs rope section, pi(2j) = j and
    pi(2j+1) = j + n/2, and what it is for:
      * for n = 6 the map is [0, 3, 1, 4, 2, 5], and for every even n it is a
        bijection whose first half of images comes from the even entries;
      * moving the entries of an interleaved-roped vector by pi gives the NEOX
        rope of the moved vector bit for bit: both layouts turn plane k by the
        same f32 angle with the same products, so this holds exactly; checked
        on each plane's unit vectors and on random vectors at positions
        spread from 0 to 2^21, for two bases;
      * hence the dot products attention takes are the same in both layouts."""
    assert list(oracle.norm_to_neox_perm(6, lib=lib)) == [0, 3, 1, 4, 2, 5]
    for n in (2, 10, 32, 128):
        pi = np.asarray(oracle.norm_to_neox_perm(n, lib=lib))
        assert sorted(pi) == list(range(n))
        assert np.array_equal(pi[0::2], np.arange(n // 2))
        assert np.array_equal(pi[1::2], np.arange(n // 2) + n // 2)
    rng = np.random.default_rng(2718)

    def moved(v, pi):
        out = np.empty_like(v)
        out[pi] = v
        return out

    for n, base in ((32, 10000.0), (64, 8_000_000.0)):
        pi = np.asarray(oracle.norm_to_neox_perm(n, lib=lib))
        positions = [0.0, 2.0, 255.0, 31337.0, float(2 ** 21)] + \
            list(np.round(np.exp(rng.uniform(0.0, math.log(2.0 ** 21), 6))))
        for pos in positions:
            basis = [np.eye(n, dtype=np.float32)[i] for i in range(n)]
            probes = basis + [rng.standard_normal(n).astype(np.float32) for _ in range(3)]
            for v in probes:
                a = moved(oracle.rope_interleaved(v, pos, base, lib=lib), pi)
                b = oracle.rope_neox(moved(v, pi), pos, base, lib=lib)
                assert np.array_equal(a, b), (n, base, pos)
            # the same products in another order: equal to f64 rounding
            u, w = probes[-2], probes[-1]
            pu = oracle.rope_interleaved(u, pos, base, lib=lib).astype(np.float64)
            pw = oracle.rope_interleaved(w, pos + 3.0, base, lib=lib).astype(np.float64)
            qu = oracle.rope_neox(moved(u, pi), pos, base, lib=lib).astype(np.float64)
            qw = oracle.rope_neox(moved(w, pi), pos + 3.0, base, lib=lib).astype(np.float64)
            bound = n * 2.0 ** -52 * float(np.abs(pu * pw).sum())
            assert abs(np.dot(pu, pw) - np.dot(qu, qw)) <= bound, (n, base, pos)


def check_rope_against_rotation(lib):
    """Each rope pairing is a rotation of its pairs by theta_j = pos *
    base^(-2j/n): compared with an f64 rotation at small positions, and the
    identity at position 0."""
    from mla_latent_cache_absorbed_gb300 import workloads as wlmod
    rng = np.random.default_rng(12)
    n, base = 16, 10000.0
    x = rng.standard_normal(n).astype(np.float32)
    assert np.array_equal(oracle.rope_neox(x, 0.0, base, lib=lib), x)
    assert np.array_equal(oracle.rope_interleaved(x, 0.0, base, lib=lib), x)
    for pos in (1.0, 3.0, 40.0):
        a = oracle.rope_neox(x, pos, base, lib=lib)
        b = wlmod.apply_rope_neox(x, np.array(pos), base)
        assert maxdiff(a, b) <= 2e-5, pos
        a = oracle.rope_interleaved(x, pos, base, lib=lib)
        b = wlmod.apply_rope_interleaved(x, np.array(pos), base)
        assert maxdiff(a, b) <= 2e-5, pos


def check_cache_append(lib):
    """do_kv_cache_update (vLLM CPU MLA page): flat[slot] = [kv_c | k_pe] cast
    to the cache type; slots < 0 skipped. The bf16 cast is torch's (round to
    nearest, ties to even), checked on values that sit exactly on a tie."""
    import oracle as O
    import torch
    rng = np.random.default_rng(11)
    R, P, nb, bs = 32, 8, 5, 16
    n = 9
    kv = rng.standard_normal((n, R)).astype(np.float32)
    kp = rng.standard_normal((n, P)).astype(np.float32)
    # exact ties for the bf16 cast: the 16 dropped bits are 0x8000
    ties = np.array([0x3f808000, 0x3f818000, 0xbf808000, 0x40008000], np.uint32).view(np.float32)
    kv[0, :4] = ties
    kv[1, :3] = [np.inf, -0.0, 3.0e38]
    slots = np.array([7, -1, 79, 0, -5, 40, 41, 12, 3], np.int64)
    poison = np.full((nb, bs, R + P), -7.25, np.float32)
    out = O.cache_append(poison, kv, kp, slots, lib=lib).reshape(-1, R + P)
    rows = np.concatenate([kv, kp], 1)
    written = set()
    for k, s_ in enumerate(slots):
        if s_ >= 0:
            assert np.array_equal(out[s_], rows[k]), k
            written.add(int(s_))
    for r in range(nb * bs):
        if r not in written:
            assert np.all(out[r] == -7.25), r
    # bf16 cache: torch's cast of the same rows, bit for bit
    pb = np.full((nb, bs, R + P), 0x1234, np.uint16)
    outb = O.cache_append(pb, kv, kp, slots, lib=lib).reshape(-1, R + P)
    ref = torch.from_numpy(rows).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for k, s_ in enumerate(slots):
        if s_ >= 0:
            assert np.array_equal(outb[s_], ref[k]), k
    assert np.all(outb[1] == 0x1234)
    # bf16 sources copy exactly
    kvb = torch.from_numpy(kv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    kpb = torch.from_numpy(kp).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    outc = O.cache_append(pb, kvb, kpb, slots, lib=lib).reshape(-1, R + P)
    assert np.array_equal(outc[7], np.concatenate([kvb[0], kpb[0]]))
    # a slot past the cache is reported and writes nothing
    bad = O.cache_append(poison, kv[:1], kp[:1], np.array([nb * bs]), allow_errors=True, lib=lib)
    assert np.all(bad == -7.25)
    try:
        O.cache_append(poison, kv[:1], kp[:1], np.array([nb * bs]), lib=lib)
        raise AssertionError("a slot past the cache must be reported")
    except O.OracleError:
        pass


def _rotation_f64(k_pe_row, pos, base):
    """NEOX rope written as the rotation it is: pair (j, j + n/2) turned by
    theta_j = pos * base^(-2j/n), in f64."""
    n = k_pe_row.size
    half = n // 2
    th = float(pos) * float(base) ** (-2.0 * np.arange(half) / n)
    a = k_pe_row[:half].astype(np.float64)
    b = k_pe_row[half:].astype(np.float64)
    return np.concatenate([a * np.cos(th) - b * np.sin(th), a * np.sin(th) + b * np.cos(th)])


def check_kv_prolog(lib):
    """KV half of the MLA prolog ("aclnnMlaProlog" page, key formulas): the
    RmsNorm of the latent against closed forms (a constant row c gives
    gamma sign(c) with eps = 0 and gamma c / sqrt(c^2 + eps) otherwise; unit
    mean square; scale invariance; a zero row stays zero), the rope of k^R
    against an f64 rotation at each token's own position (identity at 0,
    pair norms kept at large positions), and the scatter of
    do_kv_cache_update (padding skipped, other rows untouched, f32 rows
    exact, bf16 rows torch's cast of them, a slot past the cache reported)."""
    import oracle as O
    import torch
    rng = np.random.default_rng(13)
    R, P, base = 32, 8, 10000.0
    gamma = rng.uniform(0.5, 1.5, R).astype(np.float32)
    kv = np.array([[3.0] * R, [-0.5] * R], np.float32)
    kp = np.zeros((2, P), np.float32)
    rows = O.kv_prolog_rows(kv, kp, gamma, [0, 0], 0.0, base, lib=lib)
    assert maxdiff(rows[0, :R], gamma) <= 1e-12 and maxdiff(rows[1, :R], -gamma) <= 1e-12
    for c, eps in ((3.0, 27.0), (-0.5, 0.75)):   # eps = 3 c^2: gamma sign(c) / 2
        row = O.kv_prolog_rows(np.full((1, R), c, np.float32), kp[:1], gamma, [0], eps, base,
                               lib=lib)[0]
        assert maxdiff(row[:R], gamma * math.copysign(0.5, c)) <= 1e-12, (c, eps)
    x = rng.standard_normal((3, R)).astype(np.float32)
    ones = np.ones(R, np.float32)
    y = O.kv_prolog_rows(x, np.zeros((3, P), np.float32), ones, [0, 0, 0], 0.0, base, lib=lib)
    assert np.all(np.abs((y[:, :R] ** 2).mean(1) - 1.0) <= 1e-12)
    y4 = O.kv_prolog_rows(4 * x, np.zeros((3, P), np.float32), ones, [0] * 3, 0.0, base, lib=lib)
    assert maxdiff(y4[:, :R], y[:, :R]) <= 1e-14
    yg = O.kv_prolog_rows(x, np.zeros((3, P), np.float32), gamma, [0] * 3, 0.0, base, lib=lib)
    assert maxdiff(yg[:, :R], y[:, :R] * gamma) <= 1e-12
    z = O.kv_prolog_rows(np.zeros((1, R), np.float32), kp[:1], gamma, [0], 1e-6, base, lib=lib)
    assert np.all(z == 0.0)
    # rope: each token at its own position
    kpe = rng.standard_normal((5, P)).astype(np.float32)
    pos = np.array([0, 1, 3, 40, 17], np.int64)
    rows = O.kv_prolog_rows(x[np.arange(5) % 3], kpe, gamma, pos, 1e-6, base, lib=lib)
    assert np.array_equal(rows[0, R:], kpe[0].astype(np.float64))
    for t in range(1, 5):
        assert maxdiff(rows[t, R:], _rotation_f64(kpe[t], pos[t], base)) <= 2e-5, t
    far = O.kv_prolog_rows(x[:1], kpe[:1], gamma, [100000], 1e-6, base, lib=lib)[0, R:]
    h = P // 2
    n0 = np.hypot(kpe[0, :h].astype(np.float64), kpe[0, h:])
    n1 = np.hypot(far[:h], far[h:])
    assert np.all(np.abs(n1 - n0) <= 1e-5 * n0)
    # scatter by slot mapping
    nb, bs = 4, 16
    slots = np.array([7, -1, 63, 2, 20], np.int64)   # row 0 is nobody's
    kvs = x[np.arange(5) % 3]
    poison = np.full((nb, bs, R + P), -7.25, np.float32)
    out = O.cache_append_rmsnorm_rope(poison, kvs, kpe, gamma, pos, slots, 1e-6, base,
                                      lib=lib).reshape(-1, R + P)
    rows32 = rows.astype(np.float32)
    for t, s_ in enumerate(slots):
        if s_ >= 0:
            assert np.array_equal(out[s_], rows32[t]), t
            assert maxdiff(out[s_, R:], _rotation_f64(kpe[t], pos[t], base)) <= 2e-5, t
    untouched = np.setdiff1d(np.arange(nb * bs), slots[slots >= 0])
    assert np.all(out[untouched] == -7.25)
    pb = np.full((nb, bs, R + P), 0x1234, np.uint16)
    outb = O.cache_append_rmsnorm_rope(pb, kvs, kpe, gamma, pos, slots, 1e-6, base,
                                       lib=lib).reshape(-1, R + P)
    ref = torch.from_numpy(rows32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for t, s_ in enumerate(slots):
        if s_ >= 0:
            assert np.array_equal(outb[s_], ref[t]), t
    assert np.all(outb.reshape(-1, R + P)[untouched] == 0x1234)
    bad = O.cache_append_rmsnorm_rope(poison, kvs[:1], kpe[:1], gamma, [5], [nb * bs], 1e-6, base,
                                      allow_errors=True, lib=lib)
    assert np.all(bad == -7.25)
    try:
        O.cache_append_rmsnorm_rope(poison, kvs[:1], kpe[:1], gamma, [5], [nb * bs], 1e-6, base,
                                    lib=lib)
        raise AssertionError("a slot past the cache must be reported")
    except O.OracleError:
        pass


def check_causal_prefill(lib):
    """A chunk of t_q queries per request (chunked prefill in absorbed form,
    the queries being the request's last t_q positions):
      * a first chunk (t_q == t_kv) is ordinary causal self-attention over the
        whole rows: torch's SDPA with is_causal (f64) on the gathered rows
        gives the output, and logsumexp of the causally masked scaled scores
        the LSE;
      * a later chunk (t_q < t_kv): the same with the mask aligned to the
        chunk's end (query t sees keys 0 .. t_kv - t_q + t), built from
        torch.tril with a diagonal offset;
      * query t of a chunk is the one-query decode of the same request cut to
        its first t_kv - t_q + t + 1 rows, bit for bit."""
    import torch
    rng = np.random.default_rng(21)
    H, R, P = 2, 32, 8
    W = R + P
    scale = 1.0 / math.sqrt(24)
    for T, lens in [(24, [24, 24]), (20, [45, 20, 33])]:
        rows = [rng.standard_normal((s, W)).astype(np.float32) for s in lens]
        cache, bt = page(rows, lens, rng)
        sl = np.array(lens, np.int32)
        q = rng.standard_normal((len(lens), T, H, W)).astype(np.float32)
        o, lse = oracle.decode_paged(q, cache, bt, sl, T, R, scale, lib=lib)
        for b, S in enumerate(lens):
            qt = torch.from_numpy(q[b].astype(np.float64)).permute(1, 0, 2)[None]   # [1,H,T,W]
            kt = torch.from_numpy(rows[b].astype(np.float64))[None, None].expand(1, H, S, W)
            vt = kt[..., :R]
            if S == T:
                ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale,
                                                                       is_causal=True)
            mask = torch.tril(torch.ones(T, S, dtype=torch.bool), diagonal=S - T)
            if S != T:
                ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale,
                                                                       attn_mask=mask)
            sc = (qt @ kt.transpose(-1, -2)) * scale
            ref_lse = torch.logsumexp(sc.masked_fill(~mask, float("-inf")), -1)
            ref = ref[0].permute(1, 0, 2).numpy()          # [T,H,R]
            ref_lse = ref_lse[0].permute(1, 0).numpy()     # [T,H]
            assert maxdiff(ref, o[b]) <= 3e-6, (T, S, maxdiff(ref, o[b]))
            assert maxdiff(ref_lse, lse[b]) <= 3e-6, (T, S, maxdiff(ref_lse, lse[b]))
            for t in (0, T // 2, T - 1):
                cut = np.array([S - T + t + 1], np.int32)
                o1, l1 = oracle.decode_paged(q[b:b + 1, t:t + 1], cache, bt[b:b + 1], cut, 1, R,
                                             scale, lib=lib)
                assert np.array_equal(o1[0, 0], o[b, t]) and np.array_equal(l1[0, 0], lse[b, t]), \
                    (T, S, t)


def check_q_prolog(lib):
    """Query half of the MLA prolog ("aclnnMlaProlog" page, query formulas)
    as the decode consumes it, q_abs = [q^C W^UK | ROPE(c^Q W^QR)]:
      * the latent part is the absorb of q^C, bit for bit, and a head whose
        W^UK is the identity on its first d_nope columns returns q^C there;
      * the rope part is the f64 rotation of each row at its own position
        (identity at position 0), per head;
      * q^R . k^R with the key half's rope (oracle_kv_prolog_row) depends
        only on the distance of the two positions: the query and the key
        are turned by the same convention;
      * with no rope columns it is the absorb."""
    import oracle as O
    rng = np.random.default_rng(31)
    rows, H, Dn, P, R = 5, 3, 8, 16, 24
    base = 10000.0
    qn = rng.standard_normal((rows, H, Dn)).astype(np.float32)
    qp = rng.standard_normal((rows, H, P)).astype(np.float32)
    w = (rng.standard_normal((H, Dn, R)) / math.sqrt(R)).astype(np.float32)
    w[1] = 0.0
    w[1][np.arange(Dn), np.arange(Dn)] = 1.0                  # head 1: W^UK = [I | 0]
    pos = np.array([0, 1, 17, 4095, 70000], np.int64)
    out = O.absorb_q_rope(qn, qp, w, pos, base, lib=lib)
    plain = O.absorb_q(qn, qp, w, lib=lib)
    assert np.array_equal(out[:, :, :R], plain[:, :, :R])
    assert np.array_equal(out[:, 1, :Dn], qn[:, 1]) and np.all(out[:, 1, Dn:R] == 0)
    assert np.array_equal(out[0, :, R:], qp[0])                # position 0: no turn
    # the rope takes theta_j = pos * base^(-2j/P) by j f32 multiplications of
    # the f32 ratio: |theta error| <= theta_j (j + 2) 2^-23; with sin/cos and
    # the rotation's own f32 rounding, a pair (a, b) is off by at most
    # (|a| + |b|) (theta error + 1e-6)
    h2 = P // 2
    j = np.arange(h2)
    for r in range(rows):
        th = float(pos[r]) * base ** (-2.0 * j / P)
        dth = th * (j + 2) * 2.0 ** -23
        for h in range(H):
            ref = _rotation_f64(qp[r, h], pos[r], base)
            ab = np.abs(qp[r, h, :h2]).astype(np.float64) + np.abs(qp[r, h, h2:])
            bound = np.tile(ab * (dth + 1e-6), 2)
            assert np.all(np.abs(out[r, h, R:] - ref) <= bound), (r, h)
    # relative positions: (query at p + d) . (key at p) is the same for every p
    k = rng.standard_normal((1, P)).astype(np.float32)
    ones = np.ones(R, np.float32)
    kv = np.ones((1, R), np.float32)
    dots = []
    for p0 in (0, 5, 300):
        q_at = O.absorb_q_rope(qn[:1, :1], qp[:1, :1], w[:1], [p0 + 7], base, lib=lib)[0, 0, R:]
        k_at = O.kv_prolog_rows(kv, k, ones, [p0], 0.0, base, lib=lib)[0, R:]
        dots.append(float(np.dot(q_at.astype(np.float64), k_at)))
    assert max(dots) - min(dots) <= 1e-4 * max(1.0, abs(dots[0])), dots
    nope = O.absorb_q_rope(qn, qp[:, :, :0], w, pos, base, lib=lib)
    assert np.array_equal(nope, O.absorb_q(qn, qp[:, :, :0], w, lib=lib))


def check_q_prolog_full(lib):
    """The query half of the MLA prolog from c^Q's row before the norm
    ("aclnnMlaProlog" page, query formulas: c^Q = RmsNorm(x W^DQ),
    q^C = c^Q W^UQ, q^N = q^C W^UK, q^R = ROPE(c^Q W^QR)):
      * RmsNorm against closed forms: a constant row c gives gamma c /
        sqrt(c^2 + eps); with gamma = 1 and eps = 0 every row has unit mean
        square; scaling a row by 3.5 changes nothing (eps = 0); a zero row
        stays zero;
      * the projection against an f64 matmul within the bound of a sequential
        f32 sum (k 2^-24 sum |x_k w_kj| plus rounding of the result), and an
        identity weight returns its input exactly;
      * norm, both projections, the absorb and the rope composed by the oracle
        against the whole formula restated in f64 (numpy, the rope as a
        rotation), relative 1e-4."""
    import oracle as O
    rng = np.random.default_rng(77)
    # --- RmsNorm closed forms
    n = 48
    g = (rng.random(n) + 0.5).astype(np.float32)
    for c, eps in ((2.5, 0.0), (-0.75, 1e-2), (3.0, 9.0)):
        out = O.rmsnorm_rows(np.full((1, n), c, np.float32), g, eps, lib=lib)[0]
        ref = g.astype(np.float64) * c / math.sqrt(c * c + eps)
        assert np.all(np.abs(out - ref) <= 2e-7 * np.abs(ref) + 1e-30), (c, eps)
    x = rng.standard_normal((6, n)).astype(np.float32)
    ones = np.ones(n, np.float32)
    unit = O.rmsnorm_rows(x, ones, 0.0, lib=lib).astype(np.float64)
    assert np.all(np.abs(np.mean(unit * unit, axis=1) - 1.0) <= 1e-6)
    a = O.rmsnorm_rows(x, g, 0.0, lib=lib)
    b = O.rmsnorm_rows((x * 3.5).astype(np.float32), g, 0.0, lib=lib)
    assert np.all(np.abs(a - b) <= 2e-7 * np.abs(a) + 1e-30)
    assert np.all(O.rmsnorm_rows(np.zeros((2, n), np.float32), g, 1e-6, lib=lib) == 0)
    # --- projection
    k, m = 40, 24
    xs = rng.standard_normal((5, k)).astype(np.float32)
    w = (rng.standard_normal((k, m)) / math.sqrt(k)).astype(np.float32)
    y = O.project(xs, w, lib=lib).astype(np.float64)
    ref = xs.astype(np.float64) @ w.astype(np.float64)
    bound = k * 2.0 ** -24 * (np.abs(xs).astype(np.float64) @ np.abs(w).astype(np.float64)) \
        + 2.0 ** -24 * np.abs(ref)
    assert np.all(np.abs(y - ref) <= bound)
    eye = np.eye(k, dtype=np.float32)
    assert np.array_equal(O.project(xs, eye, lib=lib), xs)
    # --- the whole query half against f64
    rows, H, Dn, P, R, qr = 5, 3, 8, 16, 24, 40
    base, eps = 10000.0, 1e-6
    cq = rng.standard_normal((rows, qr)).astype(np.float32)
    gq = (rng.random(qr) + 0.5).astype(np.float32)
    w_uq = (rng.standard_normal((qr, H * Dn)) / math.sqrt(qr)).astype(np.float32)
    w_qr = (rng.standard_normal((qr, H * P)) / math.sqrt(qr)).astype(np.float32)
    w_uk = (rng.standard_normal((H, Dn, R)) / math.sqrt(R)).astype(np.float32)
    pos = np.array([0, 3, 77, 4095, 12345], np.int64)
    cn = O.rmsnorm_rows(cq, gq, eps, lib=lib)
    qc = O.project(cn, w_uq, lib=lib).reshape(rows, H, Dn)
    qpe = O.project(cn, w_qr, lib=lib).reshape(rows, H, P)
    got = O.absorb_q_rope(qc, qpe, w_uk, pos, base, lib=lib).astype(np.float64)
    c64 = cq.astype(np.float64)
    cn64 = gq.astype(np.float64) * c64 / np.sqrt(np.mean(c64 * c64, axis=1, keepdims=True) + eps)
    qc64 = (cn64 @ w_uq.astype(np.float64)).reshape(rows, H, Dn)
    qpe64 = (cn64 @ w_qr.astype(np.float64)).reshape(rows, H, P)
    lat64 = np.einsum("rhd,hdl->rhl", qc64, w_uk.astype(np.float64))
    rope64 = np.stack([np.stack([_rotation_f64(qpe64[r, h], pos[r], base) for h in range(H)])
                       for r in range(rows)])
    want = np.concatenate([lat64, rope64], axis=2)
    assert rel_ok(want, got, 1e-4), maxdiff(want, got)


QUICK_CHECKS = [check_naive_equals_absorbed, check_paged_chain_equals_naive,
                check_bruteforce_f64, check_sdpa_reduction, check_closed_forms,
                check_split_combine, check_paged_equals_contiguous,
                check_decode_rows_consistent, check_invalid_requests,
                check_absorb_decompress_unit_weights, check_rope_permutation,
                check_rope_against_rotation, check_cache_append, check_kv_prolog,
                check_causal_prefill, check_q_prolog, check_q_prolog_full]
