"""Device-side plumbing around the C ABI: upload a workload, run the path.

PyTorch supplies device memory and streams; every step of the path runs in
libmla_gb300's kernels through the `_native` binding.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import _native as N


def _torch():
    import torch
    return torch


def host_to_device(a: np.ndarray, dtype: str, device):
    """Upload a host array. bf16 data may be given as f32 values (exact bf16)
    or as uint16 bit patterns; f16 data as f32 values (exact f16)."""
    torch = _torch()
    if dtype == "bf16":
        if a.dtype == np.uint16:
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)
    elif dtype == "f16":
        t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.float16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, np.float32))
    return t.to(device)


def device_to_host_f32(t) -> np.ndarray:
    return t.float().cpu().numpy()


@dataclass
class DeviceCase:
    dims: N.MlaDims
    batch: int
    max_blocks: int
    num_blocks: int
    scale: float
    q_nope: object
    q_pe: object
    w_uk: object
    w_uv: object
    kv_cache: object
    block_table: object
    seq_lens: object
    # outputs / scratch
    q_abs: object
    o_lat: object
    lse: object
    out: object
    workspace: object
    ws_bytes: int
    dev_err: object

    @property
    def rows(self) -> int:
        return self.batch * self.dims.t_q


def upload(wl, device="cuda", kv_cache=None, q_pe=None) -> DeviceCase:
    """Upload a workloads.Workload; kv_cache / q_pe override the workload's
    (used for the permuted-rope layout)."""
    torch = _torch()
    g = wl.geom
    dims = N.MlaDims.from_geometry(g)
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16}.get(g.dtype, torch.float32)
    rows = wl.rows
    H, R, W = g.n_head, g.kv_rank, g.width
    ws = N.mla_decode_workspace_size(wl.batch, wl.max_blocks, dims)
    return DeviceCase(
        dims=dims, batch=wl.batch, max_blocks=wl.max_blocks, num_blocks=wl.num_blocks,
        scale=wl.scale,
        q_nope=host_to_device(wl.q_nope, g.dtype, device),
        q_pe=host_to_device(wl.q_pe if q_pe is None else q_pe, g.dtype, device),
        w_uk=host_to_device(wl.w_uk, g.dtype, device),
        w_uv=host_to_device(wl.w_uv, g.dtype, device),
        kv_cache=host_to_device(wl.kv_cache if kv_cache is None else kv_cache, g.dtype, device),
        block_table=torch.from_numpy(wl.block_table).to(device),
        seq_lens=torch.from_numpy(wl.seq_lens).to(device),
        q_abs=torch.empty((rows, H, W), dtype=tdt, device=device),
        o_lat=torch.empty((rows, H, R), dtype=tdt, device=device),
        lse=torch.empty((rows, H), dtype=torch.float32, device=device),
        out=torch.empty((rows, H, g.d_v), dtype=tdt, device=device),
        workspace=torch.empty(max(ws, 256), dtype=torch.uint8, device=device),
        ws_bytes=ws,
        dev_err=torch.zeros(1, dtype=torch.int32, device=device),
    )


def absorb(dc: DeviceCase, stream=None):
    N.mla_absorb_q(dc.q_abs, dc.q_nope, dc.q_pe, dc.w_uk, dc.rows, dc.dims, stream)


def decode(dc: DeviceCase, stream=None, q_abs=None, out=None, lse=None):
    N.mla_decode_paged(dc.o_lat if out is None else out, dc.lse if lse is None else lse,
                       dc.q_abs if q_abs is None else q_abs, dc.kv_cache, dc.block_table,
                       dc.seq_lens, dc.batch, dc.max_blocks, dc.num_blocks, dc.dims, dc.scale,
                       dc.workspace, dc.ws_bytes, dc.dev_err, stream)


def decompress(dc: DeviceCase, stream=None, o_lat=None, out=None):
    N.mla_decompress_out(dc.out if out is None else out, dc.o_lat if o_lat is None else o_lat,
                         dc.w_uv, dc.rows, dc.dims, stream)


def full_step(dc: DeviceCase, stream=None):
    """One pass of the hot path: absorb -> paged decode -> decompress, as three
    calls (o_lat and q_abs land in the case's buffers)."""
    absorb(dc, stream)
    decode(dc, stream)
    decompress(dc, stream)


def attend_workspace(dc: DeviceCase):
    """The fused call's scratch (allocated once per case)."""
    ws = getattr(dc, "_attend_ws", None)
    if ws is None:
        torch = _torch()
        n = N.mla_attend_workspace_size(dc.batch, dc.max_blocks, dc.dims)
        ws = (torch.empty(max(n, 256), dtype=torch.uint8, device=dc.out.device), n)
        dc._attend_ws = ws
    return ws


def attend(dc: DeviceCase, stream=None, out=None, lse=None):
    """One pass of the hot path as one call (mla_attend_absorbed)."""
    ws, n = attend_workspace(dc)
    N.mla_attend_absorbed(dc.out if out is None else out, dc.lse if lse is None else lse,
                          dc.q_nope, dc.q_pe, dc.w_uk, dc.w_uv, dc.kv_cache, dc.block_table,
                          dc.seq_lens, dc.batch, dc.max_blocks, dc.num_blocks, dc.dims,
                          dc.scale, ws, n, dc.dev_err, stream)
