"""Absorbed multi-head latent attention (MLA) decode over a paged latent KV
cache, as a C-ABI library of hand-written sm_103a CUDA kernels.

The compute lives in ``libmla_gb300.so`` (sources under ``csrc/``, public
header ``include/mla.h`` at the repository root). ``_native`` is the thin
ctypes binding whose functions carry the C entry points' names;
``workloads`` generates the seeded synthetic inputs.
"""
__all__ = ["workloads"]
