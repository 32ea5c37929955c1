"""Seeded synthetic workloads for absorbed MLA decode.

This module generates inputs only. It holds none of the attention arithmetic:
it draws random numbers, prepares them the way the upstream model would
(RMS-norm of the latent rows, rotary embedding of the rope columns, bf16
rounding), lays them out in a paged cache and builds block tables. Both the
CUDA path and the CPU oracle consume what it returns.

The five named workloads follow the decode configurations this library is
measured on:

  tiny_f32           B=2, t_q=1, H=4, d_nope=16, d_rope=8, d_v=16, kv_rank=32,
                     seq_lens [37, 64], f32, no rope, seed 0
  glm52_decode       GLM-5.2 dims (H=64, 192/64/256, rank 512), bf16, B=8,
                     seq_lens U[1, 4096] with seq_lens[3] = 0, NEOX rope base
                     10000, seed 1
  deepseek_decode    DeepSeek-V3 geometry (H=128, 128/64/128, rank 512), bf16,
                     B=64, every seq_len 8192, 40,000-block pool, seed 2
  glm53_flash_nope   GLM-5.3-Flash NoPE geometry (H=64, 256/0/256, rank 512),
                     bf16, B=128, seq_lens lognormal(median 2048, sigma 1)
                     rounded and clipped to [1, 32768], seed 3
  glm52_causal_t4    GLM-5.2 dims, bf16, t_q=4, B=32, seq_lens U[8192, 65536],
                     interleaved (NORM) rope base 10000 whose columns the
                     library's load-time permutation maps to NEOX, seed 4

A sixth workload is the chunked causal prefill in absorbed form, the same
attention with a block of queries per request:

  glm52_prefill_chunk  GLM-5.2 dims, bf16, t_q=128 (a prompt chunk of 128
                     tokens, the last 128 positions of each request), B=4,
                     seq_lens U[129, 8192] with seq_lens[0] = 128 (a first
                     chunk: t_q == t_kv, query t sees keys 0..t), NEOX rope
                     base 10000, seed 5

Value recipe (all workloads): q_nope, q_pe, k_pe ~ N(0, 1); c_kv rows ~ N(0, 1)
then x / sqrt(mean(x^2) + 1e-6) computed in f64; w_uk, w_uv ~ N(0, sd =
1/sqrt(kv_rank)). Rope angles theta_j = pos * base^(-2j/n) are computed
directly in f64; key row j sits at position j, query t of t_q at position
seq_len - t_q + t (0 for an empty request). bf16 values are f32 values rounded
to nearest-even by torch.

Paging: block size 16. Each request needs ceil(seq_len/16) blocks, drawn
without replacement from a random permutation of the pool. Block-table entries
past a request's last block are -1. Rows past seq_len in a request's last
block, and every pool block no request uses, are poisoned ("big": 1e30, or
"nan") so that any read of them shows in the result.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK = 16


@dataclass(frozen=True)
class Geometry:
    n_head: int
    d_nope: int
    d_rope: int
    d_v: int
    kv_rank: int
    t_q: int
    dtype: str  # "f32", "bf16" or "f16"
    block_size: int = BLOCK

    @property
    def width(self) -> int:
        """Cache row width: kv_rank + d_rope."""
        return self.kv_rank + self.d_rope


@dataclass
class Workload:
    name: str
    geom: Geometry
    scale: float
    seq_lens: np.ndarray            # int32 [B]
    block_table: np.ndarray         # int32 [B, max_blocks]
    num_blocks: int
    kv_cache: np.ndarray            # [num_blocks, bs, W]; float32 (f16-exact for f16),
                                    # or uint16 bf16 bits
    q_nope: np.ndarray              # float32 [B*t_q, H, d_nope] (bf16-exact when bf16)
    q_pe: np.ndarray                # float32 [B*t_q, H, d_rope]
    w_uk: np.ndarray                # float32 [H, d_nope, kv_rank]
    w_uv: np.ndarray                # float32 [H, d_v, kv_rank]
    rope: str                       # "none", "neox" or "norm"
    rope_base: float = 10000.0
    # "norm" workloads only: the pre-rope rope columns and their positions, from
    # which the consumer of the permuted layout builds its own copy.
    k_pe_raw: np.ndarray | None = None   # float32 [num_blocks, bs, d_rope]
    q_pe_raw: np.ndarray | None = None   # float32 [B*t_q, H, d_rope]
    q_pos: np.ndarray | None = None      # float64 [B*t_q]
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def rows(self) -> int:
        """Query rows: batch * t_q."""
        return self.batch * self.geom.t_q


NAMES = ("tiny_f32", "glm52_decode", "deepseek_decode", "glm53_flash_nope",
         "glm52_causal_t4", "glm52_prefill_chunk")

_GEOMS = {
    "tiny_f32": Geometry(4, 16, 8, 16, 32, 1, "f32"),
    "glm52_decode": Geometry(64, 192, 64, 256, 512, 1, "bf16"),
    "deepseek_decode": Geometry(128, 128, 64, 128, 512, 1, "bf16"),
    "glm53_flash_nope": Geometry(64, 256, 0, 256, 512, 1, "bf16"),
    "glm52_causal_t4": Geometry(64, 192, 64, 256, 512, 4, "bf16"),
    "glm52_prefill_chunk": Geometry(64, 192, 64, 256, 512, 128, "bf16"),
}
_SEEDS = {n: i for i, n in enumerate(NAMES)}
_ROPE = {"tiny_f32": "none", "glm52_decode": "neox", "deepseek_decode": "none",
         "glm53_flash_nope": "none", "glm52_causal_t4": "norm",
         "glm52_prefill_chunk": "neox"}


def geometry(name: str) -> Geometry:
    return _GEOMS[name]


def default_seq_lens(name: str, rng: np.random.Generator) -> np.ndarray:
    if name == "tiny_f32":
        s = np.array([37, 64])
    elif name == "glm52_decode":
        s = rng.integers(1, 4097, size=8)
        s[3] = 0
    elif name == "deepseek_decode":
        s = np.full(64, 8192)
    elif name == "glm53_flash_nope":
        s = np.rint(np.exp(rng.normal(math.log(2048.0), 1.0, size=128)))
        s = np.clip(s, 1, 32768)
    elif name == "glm52_causal_t4":
        s = rng.integers(8192, 65537, size=32)
    elif name == "glm52_prefill_chunk":
        s = rng.integers(129, 8193, size=4)
        s[0] = 128
    else:
        raise KeyError(name)
    return s.astype(np.int32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round f32 values to the nearest bf16 (ties to even); return f32 values."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round f32 values to bf16 and return the raw uint16 patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def round_f16(x: np.ndarray) -> np.ndarray:
    """Round f32 values to the nearest f16 (ties to even, numpy's cast);
    return f32 values."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).astype(np.float32)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Values rounded to a 16-bit dtype ("bf16", "f16") as f32; f32 unchanged."""
    if dtype == "bf16":
        return round_bf16(x)
    if dtype == "f16":
        return round_f16(x)
    return np.asarray(x, np.float32)


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 patterns (uint16) to their exact f32 values."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def rope_angles(pos: np.ndarray, n_dims: int, base: float) -> np.ndarray:
    """theta[..., j] = pos * base^(-2j/n), f64."""
    j = np.arange(n_dims // 2, dtype=np.float64)
    inv = base ** (-2.0 * j / n_dims)
    return np.asarray(pos, np.float64)[..., None] * inv


def apply_rope_neox(x: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """Rotate pairs (x[j], x[j+n/2]) by theta_j(pos); x [..., n], pos [...]. f64."""
    n = x.shape[-1]
    if n == 0:
        return np.asarray(x, np.float64)
    th = rope_angles(pos, n, base)
    c, s = np.cos(th), np.sin(th)
    a, b = x[..., : n // 2].astype(np.float64), x[..., n // 2:].astype(np.float64)
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def apply_rope_interleaved(x: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """Rotate pairs (x[2j], x[2j+1]) by theta_j(pos); x [..., n], pos [...]. f64."""
    n = x.shape[-1]
    if n == 0:
        return np.asarray(x, np.float64)
    th = rope_angles(pos, n, base)
    c, s = np.cos(th), np.sin(th)
    a, b = x[..., 0::2].astype(np.float64), x[..., 1::2].astype(np.float64)
    y = np.empty(x.shape, np.float64)
    y[..., 0::2] = a * c - b * s
    y[..., 1::2] = a * s + b * c
    return y


def rms_norm_rows(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) per row, computed in f64, returned as f32."""
    x64 = x.astype(np.float64)
    return (x64 / np.sqrt(np.mean(x64 * x64, axis=-1, keepdims=True) + eps)).astype(np.float32)


def make_workload(name: str, seed: int | None = None, seq_lens=None,
                  poison: str = "big", pool_blocks: int | None = None,
                  geom: Geometry | None = None) -> Workload:
    """Build a named workload (optionally with other seq_lens or geometry).

    seq_lens overrides the drawn lengths (the rest of the recipe is unchanged);
    pool_blocks overrides the pool size (default: the blocks needed plus
    max(4, 1/8) spare, or 40,000 for deepseek_decode).
    """
    g = geom or _GEOMS[name]
    rng = np.random.default_rng(_SEEDS[name] if seed is None else seed)
    sl = default_seq_lens(name, rng) if seq_lens is None else np.asarray(seq_lens, np.int32)
    B, T, H, bs = sl.shape[0], g.t_q, g.n_head, g.block_size
    W, R, P = g.width, g.kv_rank, g.d_rope
    rope = _ROPE.get(name, "none")
    if g.d_rope == 0:
        rope = "none"

    nblk = (sl.astype(np.int64) + bs - 1) // bs
    need = int(nblk.sum())
    max_blocks = max(1, int(nblk.max()) if B else 1)
    if pool_blocks is None:
        pool_blocks = 40000 if name == "deepseek_decode" else need + max(4, need // 8)
    if pool_blocks < need:
        raise ValueError("pool smaller than the blocks the requests need")
    order = rng.permutation(pool_blocks).astype(np.int32)
    bt = np.full((B, max_blocks), -1, np.int32)
    used = np.zeros(pool_blocks, bool)
    k = 0
    for b in range(B):
        n = int(nblk[b])
        bt[b, :n] = order[k:k + n]
        used[order[k:k + n]] = True
        k += n

    # queries and weights
    rows = B * T
    q_nope = rng.standard_normal((rows, H, g.d_nope), dtype=np.float32)
    q_pe_raw = rng.standard_normal((rows, H, P), dtype=np.float32)
    ws = 1.0 / math.sqrt(R)
    w_uk = (rng.standard_normal((H, g.d_nope, R), dtype=np.float32) * ws).astype(np.float32)
    w_uv = (rng.standard_normal((H, g.d_v, R), dtype=np.float32) * ws).astype(np.float32)

    # query positions: the last t_q positions of each request
    q_pos = np.zeros(rows, np.float64)
    for b in range(B):
        for t in range(T):
            q_pos[b * T + t] = max(int(sl[b]) - T + t, 0)

    # position of every pool row: its index within its request (unused rows: 0)
    row_pos = np.zeros((pool_blocks, bs), np.float64)
    for b in range(B):
        n = int(nblk[b])
        if n:
            row_pos[bt[b, :n]] = np.arange(n * bs, dtype=np.float64).reshape(n, bs)

    bf16 = g.dtype == "bf16"
    cache = np.empty((pool_blocks, bs, W), np.uint16 if bf16 else np.float32)
    k_pe_raw_all = np.empty((pool_blocks, bs, P), np.float32) if rope == "norm" else None
    chunk = max(1, (1 << 22) // max(1, bs * W))
    for c0 in range(0, pool_blocks, chunk):
        c1 = min(pool_blocks, c0 + chunk)
        n = (c1 - c0) * bs
        ckv = rms_norm_rows(rng.standard_normal((n, R), dtype=np.float32))
        kpe = rng.standard_normal((n, P), dtype=np.float32)
        pos = row_pos[c0:c1].reshape(n)
        if rope == "norm":
            k_pe_raw_all[c0:c1] = kpe.reshape(c1 - c0, bs, P)
            kpe = apply_rope_interleaved(kpe, pos, 10000.0).astype(np.float32)
        elif rope == "neox":
            kpe = apply_rope_neox(kpe, pos, 10000.0).astype(np.float32)
        rowsv = np.concatenate([ckv, kpe], axis=1) if P else ckv
        if g.dtype == "f16":
            rowsv = round_f16(rowsv)
        cache[c0:c1] = (bf16_bits(rowsv) if bf16 else rowsv).reshape(c1 - c0, bs, W)

    if rope == "norm":
        q_pe = apply_rope_interleaved(q_pe_raw, q_pos[:, None], 10000.0).astype(np.float32)
    elif rope == "neox":
        q_pe = apply_rope_neox(q_pe_raw, q_pos[:, None], 10000.0).astype(np.float32)
    else:
        q_pe = q_pe_raw

    if g.dtype != "f32":
        q_nope, q_pe = round_to(q_nope, g.dtype), round_to(q_pe, g.dtype)
        w_uk, w_uv = round_to(w_uk, g.dtype), round_to(w_uv, g.dtype)

    poison_rows(cache, sl, bt, used, poison, bf16, g.dtype == "f16")
    return Workload(name=name, geom=g, scale=1.0 / math.sqrt(g.d_nope + g.d_rope),
                    seq_lens=sl, block_table=bt, num_blocks=pool_blocks,
                    kv_cache=cache, q_nope=q_nope, q_pe=q_pe, w_uk=w_uk, w_uv=w_uv,
                    rope=rope, k_pe_raw=k_pe_raw_all,
                    q_pe_raw=q_pe_raw if rope == "norm" else None,
                    q_pos=q_pos if rope == "norm" else None,
                    meta={"seed": _SEEDS[name] if seed is None else seed,
                          "poison": poison, "blocks_needed": need})


def poison_value(poison: str, bf16: bool, f16: bool = False):
    """A finite huge value (1e30; 60000 for f16, whose largest is 65504) or NaN."""
    big = 60000.0 if f16 else 1e30
    v = np.float32(big) if poison == "big" else np.float32(np.nan)
    return bf16_bits(np.array([v]))[0] if bf16 else v


def poison_rows(cache, seq_lens, block_table, used, poison, bf16, f16=False):
    """Overwrite every row no request may read with the poison value."""
    if poison == "none":
        return
    val = poison_value(poison, bf16, f16)
    cache[~used] = val
    bs = cache.shape[1]
    for b in range(seq_lens.shape[0]):
        s = int(seq_lens[b])
        if s % bs:
            cache[block_table[b, s // bs], s % bs:] = val


def neox_side_rope_columns(wl: Workload, permute_cols) -> tuple[np.ndarray, np.ndarray]:
    """For a "norm" workload, build the rope columns in the permuted layout.

    permute_cols(x2d) must permute the last axis of a float32 [rows, d_rope]
    array in place with the NORM->NEOX load-time permutation. The permuted
    pre-rope values are then rotated with NEOX pairing at the same positions.
    Returns (k_pe [num_blocks, bs, P] float32, q_pe [B*t_q, H, P] float32),
    rounded to the workload's 16-bit type; unused cache rows keep the poison.
    """
    assert wl.rope == "norm"
    g = wl.geom
    P, bs = g.d_rope, g.block_size
    kraw = np.ascontiguousarray(wl.k_pe_raw.reshape(-1, P)).copy()
    qraw = np.ascontiguousarray(wl.q_pe_raw.reshape(-1, P)).copy()
    permute_cols(kraw)
    permute_cols(qraw)
    row_pos = np.zeros((wl.num_blocks, bs), np.float64)
    for b in range(wl.batch):
        n = -(-int(wl.seq_lens[b]) // bs)
        if n:
            row_pos[wl.block_table[b, :n]] = np.arange(n * bs, dtype=np.float64).reshape(n, bs)
    k = apply_rope_neox(kraw, row_pos.reshape(-1), wl.rope_base).astype(np.float32)
    qpos = np.repeat(wl.q_pos, g.n_head)
    q = apply_rope_neox(qraw, qpos, wl.rope_base).astype(np.float32)
    k, q = round_to(k, g.dtype), round_to(q, g.dtype)
    return k.reshape(wl.num_blocks, bs, P), q.reshape(wl.rows, g.n_head, P)


def cache_with_rope_columns(wl: Workload, k_pe: np.ndarray) -> np.ndarray:
    """A copy of the workload's cache whose rope columns are replaced by k_pe
    (poisoned rows stay poisoned)."""
    g = wl.geom
    R = g.kv_rank
    cache = wl.kv_cache.copy()
    if g.dtype == "bf16":
        cache[:, :, R:] = bf16_bits(k_pe)
    else:
        cache[:, :, R:] = k_pe
    used = np.zeros(wl.num_blocks, bool)
    for b in range(wl.batch):
        n = -(-int(wl.seq_lens[b]) // g.block_size)
        used[wl.block_table[b, :n]] = True
    poison_rows(cache, wl.seq_lens, wl.block_table, used, wl.meta["poison"],
                g.dtype == "bf16", g.dtype == "f16")
    return cache


# --------------------------------------------------------------------------
# inputs of the query half of the prolog
# --------------------------------------------------------------------------
@dataclass
class PrologQInputs:
    """Inputs of the query half of the MLA prolog for one geometry: each query
    row's x W^DQ before its norm (c_q), the norm's gamma, the projection
    weights W^UQ [q_rank][H*d_nope] and W^QR [q_rank][H*d_rope] in the page's
    (k, n) layout, W^UK [H][d_nope][kv_rank] and each row's position. Values
    are f32, already rounded to the geometry's dtype."""
    geom: Geometry
    c_q: np.ndarray
    gamma_q: np.ndarray
    w_uq: np.ndarray
    w_qr: np.ndarray
    w_uk: np.ndarray
    positions: np.ndarray
    q_rank: int
    eps: float
    rope_base: float

    @property
    def rows(self) -> int:
        return self.c_q.shape[0]


def make_prolog_q(geom: Geometry, rows: int, q_rank: int = 1536, seed: int = 11,
                  eps: float = 1e-6, rope_base: float = 10000.0) -> PrologQInputs:
    """Seeded inputs of the query half of the prolog. The pages give no query
    rank; 1536 is the default. c_q ~ 3 N(0, 1) (a down-projection's output,
    not yet normed); gamma ~ U(0.5, 1.5); W^UQ, W^QR ~ N(0, sd = 1/sqrt(q_rank));
    W^UK ~ N(0, sd = 1/sqrt(kv_rank)); positions U[0, 65536)."""
    rng = np.random.default_rng(seed)
    H, Dn, P, R = geom.n_head, geom.d_nope, geom.d_rope, geom.kv_rank
    c_q = (3.0 * rng.standard_normal((rows, q_rank))).astype(np.float32)
    gamma = (rng.random(q_rank) + 0.5).astype(np.float32)
    s = 1.0 / math.sqrt(q_rank)
    w_uq = (rng.standard_normal((q_rank, H * Dn)) * s).astype(np.float32)
    w_qr = (rng.standard_normal((q_rank, H * P)) * s).astype(np.float32)
    w_uk = (rng.standard_normal((H, Dn, R)) / math.sqrt(R)).astype(np.float32)
    positions = rng.integers(0, 65536, rows).astype(np.int64)
    if geom.dtype != "f32":
        c_q, gamma = round_to(c_q, geom.dtype), round_to(gamma, geom.dtype)
        w_uq, w_qr, w_uk = round_to(w_uq, geom.dtype), round_to(w_qr, geom.dtype), \
            round_to(w_uk, geom.dtype)
    return PrologQInputs(geom, c_q, gamma, w_uq, w_qr, w_uk, positions, q_rank, eps, rope_base)
