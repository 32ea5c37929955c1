"""The decode's timeout path, made to run on purpose without a fault.

Every wait inside the tensor-core decode has a time limit; a wait that gives
up records MLA_DEVERR_TIMEOUT in the caller's error word, and the kernel
drains the copies it issued, frees its tensor memory and returns, so the
stream stays usable (where the CPU kernel of "vllm.cpp cpu_mla_attn.cpp"
aborts the process). The test switch shortens the limit to 1 ms and makes the
score MMA warp wait on a barrier nothing arrives on: every pair's waits then
give up. The call after it, with the switch off, must be right again.
"""
import numpy as np
import pytest

import oracle
from mla_latent_cache_absorbed_gb300 import _native as N
from mla_latent_cache_absorbed_gb300 import device as D
from mla_latent_cache_absorbed_gb300 import workloads as W
from tolerances import lse_bound, output_bound

pytestmark = pytest.mark.gpu


def test_a_wait_that_gives_up_is_reported_and_the_stream_stays_usable():
    import torch
    wl = W.make_workload("glm52_decode", seq_lens=[300, 0, 1, 1000])
    g = wl.geom
    H, R, T = g.n_head, g.kv_rank, g.t_q
    dc = D.upload(wl)
    q = W.round_to(oracle.absorb_q(wl.q_nope, wl.q_pe, wl.w_uk), g.dtype)
    dc.q_abs.copy_(D.host_to_device(q, g.dtype, "cuda"))
    torch.cuda.synchronize()
    try:
        N.mla_debug_decode_wait_test(1_000_000, True)   # 1 ms limit, one barrier never completes
        D.decode(dc)
        torch.cuda.synchronize()
    finally:
        N.mla_debug_decode_wait_test(0, False)
    err = int(dc.dev_err.item())
    assert err & N.DEVERR_TIMEOUT, err
    # the same stream, the same buffers: the next call is right again
    dc.dev_err.zero_()
    D.decode(dc)
    torch.cuda.synchronize()
    assert int(dc.dev_err.item()) == 0
    o_ref, lse_ref = oracle.decode_paged(q.reshape(wl.batch, T, H, -1), wl.kv_cache,
                                         wl.block_table, wl.seq_lens, T, R, wl.scale)
    got = D.device_to_host_f32(dc.o_lat).astype(np.float64)
    ref = o_ref.reshape(got.shape).astype(np.float64)
    assert np.all(np.abs(got - ref) <= output_bound(ref, g.dtype))
    lg, lr = dc.lse.cpu().numpy().reshape(-1), lse_ref.reshape(-1)
    assert np.array_equal(np.isneginf(lg), np.isneginf(lr))
    fin = ~np.isneginf(lr)
    assert np.abs(lg[fin] - lr[fin]).max() <= lse_bound(g.dtype)
