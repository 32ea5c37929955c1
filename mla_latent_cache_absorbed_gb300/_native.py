"""Thin ctypes binding of libmla_gb300 (include/mla.h).

Each function carries the name of the C entry point it calls and only
marshals arguments: torch tensors become device pointers, the current torch
stream becomes the cudaStream_t, and a non-OK status becomes MlaError. All
computation happens in the library's kernels. Loading fails loudly when the
library has not been built; there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla_gb300.so")

MLA_F32 = 0
MLA_BF16 = 1
MLA_F16 = 2

DEVERR_BAD_BLOCK = 1
DEVERR_SEQ_TOO_LONG = 2
DEVERR_SEQ_SHORT = 4
DEVERR_TIMEOUT = 8

# Every exported symbol of include/mla.h.
EXPORTS = ("mla_absorb_q", "mla_absorb_q_rope", "mla_prolog_q", "mla_decode_workspace_size",
           "mla_decode_paged",
           "mla_decode_paged_static", "mla_decompress_out", "mla_cache_append",
           "mla_cache_append_rmsnorm_rope", "mla_attend_workspace_size", "mla_attend_absorbed",
           "mla_rope_norm_to_neox_perm",
           "mla_permute_rope_cols", "mla_permute_rope_rows", "mla_debug_decode_wait_test",
           "mla_status_str", "mla_last_error")


class MlaDims(ctypes.Structure):
    _fields_ = [("n_head", ctypes.c_int32), ("d_nope", ctypes.c_int32),
                ("d_rope", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("kv_rank", ctypes.c_int32), ("t_q", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("dtype", ctypes.c_int32)]

    @classmethod
    def from_geometry(cls, g) -> "MlaDims":
        """From a workloads.Geometry (or anything with the same fields)."""
        return cls(g.n_head, g.d_nope, g.d_rope, g.d_v, g.kv_rank, g.t_q, g.block_size,
                   {"bf16": MLA_BF16, "f16": MLA_F16}.get(g.dtype, MLA_F32))


class MlaError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} -> {status}: {message}")
        self.status = status


_lib = None


def load(path: str = LIB_PATH):
    """Load the library (raises if it is missing: build it with build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m mla_latent_cache_absorbed_gb300.build`")
    lib = ctypes.CDLL(path)
    P, I32, I64, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    D = ctypes.POINTER(MlaDims)
    lib.mla_absorb_q.argtypes = [P, P, P, P, I32, D, P]
    lib.mla_absorb_q_rope.argtypes = [P, P, P, P, P, I32, F, D, P]
    lib.mla_prolog_q.argtypes = [P, P, P, P, P, P, P, I32, I32, F, F, D, P, P]
    lib.mla_decode_workspace_size.argtypes = [I32, I32, D, ctypes.POINTER(ctypes.c_size_t)]
    lib.mla_decode_paged.argtypes = [P, P, P, P, P, P, I32, I32, I32, D, F, P,
                                     ctypes.c_size_t, P, P]
    lib.mla_decode_paged_static.argtypes = [P, P, P, P, P, P, I32, I32, I32, D, F, P, P]
    lib.mla_decompress_out.argtypes = [P, P, P, I32, D, P]
    lib.mla_cache_append.argtypes = [P, P, P, P, I32, I32, I32, D, P, P]
    lib.mla_cache_append_rmsnorm_rope.argtypes = [P, P, P, P, P, P, I32, I32, I32, F, F, D, P, P]
    lib.mla_attend_workspace_size.argtypes = [I32, I32, D, ctypes.POINTER(ctypes.c_size_t)]
    lib.mla_attend_absorbed.argtypes = [P, P, P, P, P, P, P, P, P, I32, I32, I32, D, F, P,
                                        ctypes.c_size_t, P, P]
    lib.mla_rope_norm_to_neox_perm.argtypes = [I32, P]
    lib.mla_permute_rope_cols.argtypes = [P, I32, I64, I64, I32, I32]
    lib.mla_permute_rope_rows.argtypes = [P, I32, I64, I32, I32]
    lib.mla_debug_decode_wait_test.argtypes = [ctypes.c_uint64, I32]
    lib.mla_status_str.argtypes = [ctypes.c_int]
    lib.mla_status_str.restype = ctypes.c_char_p
    lib.mla_last_error.argtypes = []
    lib.mla_last_error.restype = ctypes.c_char_p
    for name in ("mla_absorb_q", "mla_absorb_q_rope", "mla_decode_workspace_size",
                 "mla_decode_paged",
                 "mla_decode_paged_static", "mla_decompress_out", "mla_cache_append",
                 "mla_cache_append_rmsnorm_rope", "mla_attend_workspace_size",
                 "mla_attend_absorbed",
                 "mla_rope_norm_to_neox_perm", "mla_permute_rope_cols",
                 "mla_permute_rope_rows"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != 0:
        lib = load()
        raise MlaError(fn, status, lib.mla_last_error().decode() or
                       lib.mla_status_str(status).decode())


def _ptr(x) -> int | None:
    """Device pointer of a torch tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def mla_absorb_q(q_abs, q_nope, q_pe, w_uk, rows: int, dims: MlaDims, stream=None):
    _check("mla_absorb_q", load().mla_absorb_q(_ptr(q_abs), _ptr(q_nope), _ptr(q_pe),
                                               _ptr(w_uk), rows, ctypes.byref(dims),
                                               _stream(stream)))


def mla_absorb_q_rope(q_abs, q_nope, q_pe, w_uk, positions, rows: int, rope_base: float,
                      dims: MlaDims, stream=None):
    """mla_absorb_q with the query's NEOX rope at each row's position."""
    _check("mla_absorb_q_rope",
           load().mla_absorb_q_rope(_ptr(q_abs), _ptr(q_nope), _ptr(q_pe), _ptr(w_uk),
                                    _ptr(positions), rows, float(rope_base), ctypes.byref(dims),
                                    _stream(stream)))


def mla_prolog_q(q_abs, c_q, gamma_q, w_uq, w_qr, w_uk, positions, rows: int, q_rank: int,
                 eps: float, rope_base: float, dims: MlaDims, dev_err=None, stream=None):
    """The query half of the prolog: RmsNorm of c_q, W^UQ / W^QR, absorb, rope."""
    _check("mla_prolog_q",
           load().mla_prolog_q(_ptr(q_abs), _ptr(c_q), _ptr(gamma_q), _ptr(w_uq), _ptr(w_qr),
                               _ptr(w_uk), _ptr(positions), rows, q_rank, float(eps),
                               float(rope_base), ctypes.byref(dims), _ptr(dev_err),
                               _stream(stream)))


def mla_decode_workspace_size(batch: int, max_blocks: int, dims: MlaDims) -> int:
    n = ctypes.c_size_t(0)
    _check("mla_decode_workspace_size",
           load().mla_decode_workspace_size(batch, max_blocks, ctypes.byref(dims),
                                            ctypes.byref(n)))
    return n.value


def mla_decode_paged(out, lse, q_abs, kv_cache, block_table, seq_lens, batch: int,
                     max_blocks: int, num_blocks: int, dims: MlaDims, scale: float,
                     workspace, workspace_bytes: int, dev_err=None, stream=None):
    _check("mla_decode_paged",
           load().mla_decode_paged(_ptr(out), _ptr(lse), _ptr(q_abs), _ptr(kv_cache),
                                   _ptr(block_table), _ptr(seq_lens), batch, max_blocks,
                                   num_blocks, ctypes.byref(dims), float(scale),
                                   _ptr(workspace), workspace_bytes, _ptr(dev_err),
                                   _stream(stream)))


def mla_decode_paged_static(out, lse, q_abs, kv_cache, block_table, seq_lens, batch: int,
                            max_blocks: int, num_blocks: int, dims: MlaDims, scale: float,
                            dev_err=None, stream=None):
    """mla_decode_paged with the library's static scratch (allocates nothing)."""
    _check("mla_decode_paged_static",
           load().mla_decode_paged_static(_ptr(out), _ptr(lse), _ptr(q_abs), _ptr(kv_cache),
                                          _ptr(block_table), _ptr(seq_lens), batch, max_blocks,
                                          num_blocks, ctypes.byref(dims), float(scale),
                                          _ptr(dev_err), _stream(stream)))


def mla_decompress_out(out, o_lat, w_uv, rows: int, dims: MlaDims, stream=None):
    _check("mla_decompress_out", load().mla_decompress_out(_ptr(out), _ptr(o_lat), _ptr(w_uv),
                                                           rows, ctypes.byref(dims),
                                                           _stream(stream)))


def mla_cache_append(kv_cache, kv_c, k_pe, slot_mapping, n_tokens: int, num_blocks: int,
                     src_dtype: int, dims: MlaDims, dev_err=None, stream=None):
    _check("mla_cache_append",
           load().mla_cache_append(_ptr(kv_cache), _ptr(kv_c), _ptr(k_pe), _ptr(slot_mapping),
                                   n_tokens, num_blocks, src_dtype, ctypes.byref(dims),
                                   _ptr(dev_err), _stream(stream)))


def mla_cache_append_rmsnorm_rope(kv_cache, kv_c, k_pe, gamma, positions, slot_mapping,
                                  n_tokens: int, num_blocks: int, src_dtype: int, eps: float,
                                  rope_base: float, dims: MlaDims, dev_err=None, stream=None):
    _check("mla_cache_append_rmsnorm_rope",
           load().mla_cache_append_rmsnorm_rope(_ptr(kv_cache), _ptr(kv_c), _ptr(k_pe),
                                                _ptr(gamma), _ptr(positions), _ptr(slot_mapping),
                                                n_tokens, num_blocks, src_dtype, eps, rope_base,
                                                ctypes.byref(dims), _ptr(dev_err),
                                                _stream(stream)))


def mla_attend_workspace_size(batch: int, max_blocks: int, dims: MlaDims) -> int:
    n = ctypes.c_size_t(0)
    _check("mla_attend_workspace_size",
           load().mla_attend_workspace_size(batch, max_blocks, ctypes.byref(dims),
                                            ctypes.byref(n)))
    return n.value


def mla_attend_absorbed(out, lse, q_nope, q_pe, w_uk, w_uv, kv_cache, block_table, seq_lens,
                        batch: int, max_blocks: int, num_blocks: int, dims: MlaDims,
                        scale: float, workspace, workspace_bytes: int, dev_err=None,
                        stream=None):
    _check("mla_attend_absorbed",
           load().mla_attend_absorbed(_ptr(out), _ptr(lse), _ptr(q_nope), _ptr(q_pe), _ptr(w_uk),
                                      _ptr(w_uv), _ptr(kv_cache), _ptr(block_table),
                                      _ptr(seq_lens), batch, max_blocks, num_blocks,
                                      ctypes.byref(dims), float(scale), _ptr(workspace),
                                      workspace_bytes, _ptr(dev_err), _stream(stream)))


def mla_rope_norm_to_neox_perm(n_dims: int) -> np.ndarray:
    perm = np.empty(max(n_dims, 1), np.int32)
    _check("mla_rope_norm_to_neox_perm",
           load().mla_rope_norm_to_neox_perm(n_dims, perm.ctypes.data_as(ctypes.c_void_p)))
    return perm[:n_dims]


def _host_elem_bytes(a: np.ndarray) -> int:
    if a.dtype in (np.float32, np.int32, np.uint32):
        return 4
    if a.dtype in (np.uint16, np.int16, np.float16):
        return 2
    raise TypeError(f"unsupported host dtype {a.dtype}")


def mla_permute_rope_cols(x: np.ndarray, col0: int, n_dims: int):
    """In place on a C-contiguous host array viewed as [rows, last_dim]."""
    assert x.flags.c_contiguous
    stride = x.shape[-1]
    rows = x.size // stride if stride else 0
    _check("mla_permute_rope_cols",
           load().mla_permute_rope_cols(x.ctypes.data_as(ctypes.c_void_p), _host_elem_bytes(x),
                                        rows, stride, col0, n_dims))


def mla_permute_rope_rows(w: np.ndarray, row0: int, n_dims: int):
    """In place on a C-contiguous host matrix [n_rows, row_len]."""
    assert w.flags.c_contiguous and w.ndim == 2
    _check("mla_permute_rope_rows",
           load().mla_permute_rope_rows(w.ctypes.data_as(ctypes.c_void_p), _host_elem_bytes(w),
                                        w.shape[1], row0, n_dims))


def mla_debug_decode_wait_test(limit_ns: int, stall: bool):
    """Timeout-path test switch of the tensor-core decode (see include/mla.h)."""
    _check("mla_debug_decode_wait_test",
           load().mla_debug_decode_wait_test(int(limit_ns), 1 if stall else 0))


def mla_status_str(status: int) -> str:
    return load().mla_status_str(status).decode()


def mla_last_error() -> str:
    return load().mla_last_error().decode()
