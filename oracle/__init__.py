"""Plain CPU oracle for absorbed MLA decode over a paged latent cache.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The product path (``mla_latent_cache_absorbed_gb300``) never does, and
the two share no code: the arithmetic lives in ``mla_oracle.c`` (plain C, f32,
sequential sums, built with ``-ffp-contract=off``), and this module only
marshals numpy arrays into it.

Each wrapper names the passage its C function restates (see the header of
``mla_oracle.c``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_mla.so")

F32 = 0
BF16 = 1

_lib = None
_lock = threading.Lock()


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle with gcc into a shared library and return its path."""
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _stale() -> bool:
    return (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))


def load(path: str | None = None):
    """Load (building first if missing or older than the source) the oracle."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _stale():
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_I64 = ctypes.c_int64
_D = ctypes.c_double


def _declare(lib):
    lib.oracle_absorb_q.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I]
    lib.oracle_absorb_q_rope.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F]
    lib.oracle_decode_range.argtypes = [_P, _P, _P, _I, _P, _I, _P, _I, _I, _I,
                                        _I, _I, _I, _I, _I, _F, _I, _I, _P, _P]
    lib.oracle_decode_rows.argtypes = [_P, _P, _P, _I, _P, _I, _P, _P, _I, _I, _I,
                                       _I, _I, _I, _I, _I, _F, _P, _I64, _P]
    lib.oracle_decode_paged.argtypes = [_P, _P, _P, _I, _P, _I, _P, _P, _I, _I, _I,
                                        _I, _I, _I, _I, _I, _F, _P]
    lib.oracle_combine.argtypes = [_P, _P, _P, _P, _I, _I]
    lib.oracle_decompress.argtypes = [_P, _P, _P, _I, _I, _I, _I]
    lib.oracle_attend_naive.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                        _I, _I, _I, _F, _P, _P, _P]
    lib.oracle_attend_absorbed.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I,
                                           _I, _I, _I, _I, _F, _P, _P, _P]
    lib.oracle_rope_interleaved.argtypes = [_P, _I, _F, _F]
    lib.oracle_rope_neox.argtypes = [_P, _I, _F, _F]
    lib.oracle_norm_to_neox_perm.argtypes = [_I, _P]
    lib.oracle_cache_append.argtypes = [_P, _I, _P, _P, _I, _P, _I, _I64, _I, _I]
    lib.oracle_kv_prolog_row.argtypes = [_P, _P, _P, _P, _I, _I64, _I64, _I, _I, _D, _F]
    lib.oracle_rmsnorm_rows.argtypes = [_P, _P, _P, _I, _I, _I, _D]
    lib.oracle_project.argtypes = [_P, _P, _P, _I, _I, _I]
    lib.oracle_cache_append_rmsnorm_rope.argtypes = [_P, _I, _P, _P, _P, _I, _P, _P, _I, _I64,
                                                     _I, _I, _D, _F]
    for name in ("oracle_absorb_q", "oracle_decode_range", "oracle_decode_rows",
                 "oracle_decode_paged", "oracle_combine", "oracle_decompress",
                 "oracle_attend_naive", "oracle_attend_absorbed",
                 "oracle_norm_to_neox_perm", "oracle_cache_append", "oracle_kv_prolog_row",
                 "oracle_cache_append_rmsnorm_rope"):
        getattr(lib, name).restype = _I
    lib.oracle_rope_interleaved.restype = None
    lib.oracle_rope_neox.restype = None
    return lib


class OracleError(RuntimeError):
    """Raised when the oracle reports an invalid request (status < 0)."""

    def __init__(self, status: int):
        super().__init__(f"oracle status {status}")
        self.status = status


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _elem(a: np.ndarray) -> tuple[np.ndarray, int]:
    """f32 arrays pass as f32, uint16 arrays as raw bf16 patterns."""
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a), BF16
    return _f32(a), F32


def _check(status: int, allow_errors: bool):
    if status != 0 and not allow_errors:
        raise OracleError(status)
    return status


# --------------------------------------------------------------------------
# stage functions
# --------------------------------------------------------------------------
def absorb_q(q_nope, q_pe, w_uk, lib=None) -> np.ndarray:
    """q_abs[r,h] = [w_uk[h]^T q_nope[r,h] | q_pe[r,h]] (mla.rs absorb step).

    q_nope [rows, H, Dn], q_pe [rows, H, P], w_uk [H, Dn, R] -> [rows, H, R+P].
    """
    lib = lib or load()
    q_nope, q_pe, w_uk = _f32(q_nope), _f32(q_pe), _f32(w_uk)
    rows, H, Dn = q_nope.shape
    P = q_pe.shape[2]
    R = w_uk.shape[2]
    out = np.empty((rows, H, R + P), np.float32)
    _check(lib.oracle_absorb_q(_ptr(out), _ptr(q_nope), _ptr(q_pe), _ptr(w_uk),
                               rows, H, Dn, P, R), False)
    return out


def absorb_q_rope(q_nope, q_pe, w_uk, positions, rope_base, lib=None) -> np.ndarray:
    """The query half of the "aclnnMlaProlog" page as the decode consumes it:
    q_abs[r,h] = [w_uk[h]^T q_nope[r,h] | NEOX rope of q_pe[r,h] at
    positions[r]] (mla.rs rope_neox, f32).

    q_nope [rows, H, Dn], q_pe [rows, H, P] (before the rope), w_uk [H, Dn, R],
    positions [rows] int -> [rows, H, R+P].
    """
    lib = lib or load()
    q_nope, q_pe, w_uk = _f32(q_nope), _f32(q_pe), _f32(w_uk)
    rows, H, Dn = q_nope.shape
    P = q_pe.shape[2]
    R = w_uk.shape[2]
    pos = np.ascontiguousarray(np.asarray(positions, np.int64).reshape(rows))
    out = np.empty((rows, H, R + P), np.float32)
    _check(lib.oracle_absorb_q_rope(_ptr(out), _ptr(q_nope), _ptr(q_pe), _ptr(w_uk), _ptr(pos),
                                    rows, H, Dn, P, R, float(rope_base)), False)
    return out


def rmsnorm_rows(x, gamma, eps, lib=None) -> np.ndarray:
    """c^Q = RmsNorm(x) per row (the "aclnnMlaProlog" page's RmsNorm formula,
    f64 arithmetic, f32 result). x [rows, n] and gamma [n] are f32 arrays, or
    uint16 arrays of bf16 bit patterns (both the same kind)."""
    lib = lib or load()
    xa, dt = _elem(np.asarray(x))
    ga, gdt = _elem(np.asarray(gamma))
    assert dt == gdt, "x and gamma must be of one element type"
    rows, n = xa.shape
    out = np.empty((rows, n), np.float32)
    _check(lib.oracle_rmsnorm_rows(_ptr(out), _ptr(xa), _ptr(ga), dt, rows, n, float(eps)), False)
    return out


def project(x, w, lib=None) -> np.ndarray:
    """y = x W for x [rows, k] and a projection weight W [k, n] (f32 sums in
    k order): q^C = c^Q W^UQ or c^Q W^QR of the "aclnnMlaProlog" page."""
    lib = lib or load()
    xa, wa = _f32(x), _f32(w)
    rows, k = xa.shape
    n = wa.shape[1]
    assert wa.shape[0] == k
    y = np.empty((rows, n), np.float32)
    _check(lib.oracle_project(_ptr(y), _ptr(xa), _ptr(wa), rows, k, n), False)
    return y


def decode_rows(q_abs, kv_cache, block_table, seq_lens, t_q, kv_rank, scale,
                rows, allow_errors=False, lib=None):
    """Paged single-pass decode (cpu_mla_attn.cpp) of selected query rows.

    q_abs [B, t_q, H, W] (or [B*t_q, H, W]); kv_cache [num_blocks, bs, W];
    block_table [B, max_blocks] int32; seq_lens [B] int32; rows: flattened
    (b*t_q + t)*H + h ids. Returns (o [n, R], lse [n]) and, when
    allow_errors, the status as a third value.
    """
    lib = lib or load()
    q, q_dt = _elem(np.asarray(q_abs))
    kv, kv_dt = _elem(np.asarray(kv_cache))
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    ids = np.ascontiguousarray(rows, dtype=np.int64)
    num_blocks, bs, W = kv.shape
    B, max_blocks = bt.shape
    H = q.shape[-2]
    P = W - kv_rank
    o = np.empty((ids.size, kv_rank), np.float32)
    lse = np.empty(ids.size, np.float32)
    scratch = np.empty(2 * kv_rank + P, np.float32)
    st = lib.oracle_decode_rows(_ptr(o), _ptr(lse), _ptr(q), q_dt, _ptr(kv), kv_dt,
                                _ptr(bt), _ptr(sl), B, t_q, H, kv_rank, P, bs,
                                max_blocks, num_blocks, float(scale), _ptr(ids),
                                ids.size, _ptr(scratch))
    _check(st, allow_errors)
    return (o, lse, st) if allow_errors else (o, lse)


def decode_paged(q_abs, kv_cache, block_table, seq_lens, t_q, kv_rank, scale,
                 allow_errors=False, lib=None):
    """All rows of the paged decode: o [B, t_q, H, R], lse [B, t_q, H]."""
    lib = lib or load()
    q, q_dt = _elem(np.asarray(q_abs))
    kv, kv_dt = _elem(np.asarray(kv_cache))
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    num_blocks, bs, W = kv.shape
    B, max_blocks = bt.shape
    H = q.shape[-2]
    P = W - kv_rank
    o = np.empty((B, t_q, H, kv_rank), np.float32)
    lse = np.empty((B, t_q, H), np.float32)
    scratch = np.empty(2 * kv_rank + P, np.float32)
    st = lib.oracle_decode_paged(_ptr(o), _ptr(lse), _ptr(q), q_dt, _ptr(kv), kv_dt,
                                 _ptr(bt), _ptr(sl), B, t_q, H, kv_rank, P, bs,
                                 max_blocks, num_blocks, float(scale), _ptr(scratch))
    _check(st, allow_errors)
    return (o, lse, st) if allow_errors else (o, lse)


def decode_range(q_row, kv_cache, bt_row, seq_len, t_q, t, kv_rank, scale,
                 j_begin, j_end, lib=None):
    """One query row over the visible keys in [j_begin, j_end): (o [R], lse)."""
    lib = lib or load()
    q, q_dt = _elem(np.asarray(q_row))
    kv, kv_dt = _elem(np.asarray(kv_cache))
    bt = np.ascontiguousarray(bt_row, dtype=np.int32)
    num_blocks, bs, W = kv.shape
    P = W - kv_rank
    o = np.empty(kv_rank, np.float32)
    lse = np.empty(1, np.float32)
    acc = np.empty(kv_rank, np.float32)
    qf = np.empty(W, np.float32)
    _check(lib.oracle_decode_range(_ptr(o), _ptr(lse), _ptr(q), q_dt, _ptr(kv), kv_dt,
                                   _ptr(bt), int(seq_len), t_q, t, kv_rank, P, bs,
                                   bt.size, num_blocks, float(scale), int(j_begin),
                                   int(j_end), _ptr(acc), _ptr(qf)), False)
    return o, float(lse[0])


def combine(o_parts, lse_parts, lib=None):
    """LSE-weighted merge of partial results: (o [R], lse)."""
    lib = lib or load()
    o_parts = _f32(o_parts)
    lse_parts = _f32(lse_parts)
    n, R = o_parts.shape
    o = np.empty(R, np.float32)
    lse = np.empty(1, np.float32)
    _check(lib.oracle_combine(_ptr(o), _ptr(lse), _ptr(o_parts), _ptr(lse_parts), n, R),
           False)
    return o, float(lse[0])


def decompress(o_lat, w_uv, lib=None) -> np.ndarray:
    """out[r,h,j] = sum_l w_uv[h,j,l] o_lat[r,h,l] (mla.rs decompress step)."""
    lib = lib or load()
    o_lat, w_uv = _f32(o_lat), _f32(w_uv)
    rows, H, R = o_lat.shape
    Dv = w_uv.shape[1]
    out = np.empty((rows, H, Dv), np.float32)
    _check(lib.oracle_decompress(_ptr(out), _ptr(o_lat), _ptr(w_uv), rows, H, Dv, R),
           False)
    return out


def attend_naive(q_nope, q_pe, c_kv, k_pe, w_uk, w_uv, scale, lib=None):
    """mla.rs mla_attend_naive over a contiguous cache: out [t_q, H, Dv]."""
    lib = lib or load()
    args = [_f32(a) for a in (q_nope, q_pe, c_kv, k_pe, w_uk, w_uv)]
    q_nope, q_pe, c_kv, k_pe, w_uk, w_uv = args
    t_q, H, Dn = q_nope.shape
    P = q_pe.shape[2]
    t_kv, R = c_kv.shape
    Dv = w_uv.shape[1]
    out = np.empty((t_q, H, Dv), np.float32)
    k_nope = np.empty(t_kv * Dn, np.float32)
    v = np.empty(t_kv * Dv, np.float32)
    scores = np.empty(t_kv, np.float32)
    _check(lib.oracle_attend_naive(_ptr(out), *[_ptr(a) for a in args], t_q, t_kv, H,
                                   Dn, P, Dv, R, float(scale), _ptr(k_nope), _ptr(v),
                                   _ptr(scores)), False)
    return out


def attend_absorbed(q_nope, q_pe, c_kv, k_pe, w_uk, w_uv, scale, lib=None):
    """mla.rs mla_attend_absorbed over a contiguous cache: out [t_q, H, Dv]."""
    lib = lib or load()
    args = [_f32(a) for a in (q_nope, q_pe, c_kv, k_pe, w_uk, w_uv)]
    q_nope, q_pe, c_kv, k_pe, w_uk, w_uv = args
    t_q, H, Dn = q_nope.shape
    P = q_pe.shape[2]
    t_kv, R = c_kv.shape
    Dv = w_uv.shape[1]
    out = np.empty((t_q, H, Dv), np.float32)
    q_lat = np.empty(R, np.float32)
    o_lat = np.empty(R, np.float32)
    scores = np.empty(t_kv, np.float32)
    _check(lib.oracle_attend_absorbed(_ptr(out), *[_ptr(a) for a in args], t_q, t_kv,
                                      H, Dn, P, Dv, R, float(scale), _ptr(q_lat),
                                      _ptr(o_lat), _ptr(scores)), False)
    return out


def rope_interleaved(x, pos, base, lib=None) -> np.ndarray:
    """mla.rs rope_interleaved on a copy of x (all of x is the rope span)."""
    lib = lib or load()
    y = _f32(x).copy()
    lib.oracle_rope_interleaved(_ptr(y), y.size, float(pos), float(base))
    return y


def rope_neox(x, pos, base, lib=None) -> np.ndarray:
    """mla.rs rope_neox on a copy of x (all of x is the rope span)."""
    lib = lib or load()
    y = _f32(x).copy()
    lib.oracle_rope_neox(_ptr(y), y.size, float(pos), float(base))
    return y


def norm_to_neox_perm(n_dims: int, lib=None) -> np.ndarray:
    """mla.rs norm_to_neox_perm: source index -> NEOX index."""
    lib = lib or load()
    p = np.empty(n_dims, np.int32)
    _check(lib.oracle_norm_to_neox_perm(n_dims, _ptr(p)), False)
    return p


def cache_append(kv_cache, kv_c, k_pe, slot_mapping, allow_errors=False, lib=None):
    """The page's do_kv_cache_update: writes [kv_c[n] | k_pe[n]] into flat
    cache row slot_mapping[n] (cast to the cache's type, round to nearest
    even for bf16), skipping slots < 0. kv_cache is [num_blocks, bs, W]
    float32 or uint16 (bf16 bits) and is updated in place on a copy that is
    returned; kv_c [n, R] and k_pe [n, P] are float32 or uint16 (bf16)."""
    lib = lib or load()
    cache = np.array(kv_cache, copy=True, order="C")
    if cache.dtype not in (np.float32, np.uint16):
        raise TypeError("cache must be float32 or bf16 bits (uint16)")
    cdt = BF16 if cache.dtype == np.uint16 else F32
    kv_c_a, sdt = _elem(np.asarray(kv_c))
    k_pe_a, sdt2 = _elem(np.asarray(k_pe))
    if sdt != sdt2:
        raise TypeError("kv_c and k_pe must share an element type")
    n, R = kv_c_a.shape
    P = k_pe_a.shape[1] if k_pe_a.ndim == 2 else 0
    if cache.shape[-1] != R + P:
        raise ValueError("cache row width must be kv_rank + d_rope")
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    num_slots = int(np.prod(cache.shape[:-1]))
    st = lib.oracle_cache_append(_ptr(cache), cdt, _ptr(kv_c_a), _ptr(k_pe_a), sdt, _ptr(slots), n,
                                 num_slots, R, P)
    _check(st, allow_errors)
    return cache


def _prolog_inputs(kv_c, k_pe, gamma, positions):
    kv_c_a, sdt = _elem(np.asarray(kv_c))
    n, R = kv_c_a.shape
    if k_pe is None:
        k_pe_a, sdt2, P = np.zeros((n, 0), kv_c_a.dtype), sdt, 0
    else:
        k_pe_a, sdt2 = _elem(np.asarray(k_pe))
        P = k_pe_a.shape[1]
    g_a, sdt3 = _elem(np.asarray(gamma))
    if not (sdt == sdt2 == sdt3):
        raise TypeError("kv_c, k_pe and gamma must share an element type")
    if g_a.shape != (R,):
        raise ValueError("gamma must have kv_rank elements")
    pos = np.ascontiguousarray(np.zeros(n) if positions is None else positions, dtype=np.int64)
    return kv_c_a, k_pe_a, g_a, pos, sdt, n, R, P


def kv_prolog_rows(kv_c, k_pe, gamma, positions, eps, rope_base, lib=None) -> np.ndarray:
    """The cache rows [RmsNorm(kv_c[n]) | rope_neox(k_pe[n], positions[n])]
    before any cast, as float64 [n, R + P] (the norm in f64, the rope in the
    mla.rs page's f32); the "aclnnMlaProlog" page's key formulas."""
    lib = lib or load()
    kv_c_a, k_pe_a, g_a, pos, sdt, n, R, P = _prolog_inputs(kv_c, k_pe, gamma, positions)
    rows = np.empty((n, R + P), np.float64)
    for t in range(n):
        _check(lib.oracle_kv_prolog_row(_ptr(rows[t]), _ptr(kv_c_a), _ptr(k_pe_a), _ptr(g_a), sdt,
                                        t, int(pos[t]), R, P, float(eps), float(rope_base)), False)
    return rows


def cache_append_rmsnorm_rope(kv_cache, kv_c, k_pe, gamma, positions, slot_mapping, eps,
                              rope_base, allow_errors=False, lib=None):
    """cache_append of the rows kv_prolog_rows gives (rounded to f32, then
    cast to the cache's type), on a copy of kv_cache that is returned."""
    lib = lib or load()
    cache = np.array(kv_cache, copy=True, order="C")
    if cache.dtype not in (np.float32, np.uint16):
        raise TypeError("cache must be float32 or bf16 bits (uint16)")
    cdt = BF16 if cache.dtype == np.uint16 else F32
    kv_c_a, k_pe_a, g_a, pos, sdt, n, R, P = _prolog_inputs(kv_c, k_pe, gamma, positions)
    if cache.shape[-1] != R + P:
        raise ValueError("cache row width must be kv_rank + d_rope")
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    num_slots = int(np.prod(cache.shape[:-1]))
    st = lib.oracle_cache_append_rmsnorm_rope(_ptr(cache), cdt, _ptr(kv_c_a), _ptr(k_pe_a),
                                              _ptr(g_a), sdt, _ptr(pos), _ptr(slots), n,
                                              num_slots, R, P, float(eps), float(rope_base))
    _check(st, allow_errors)
    return cache
