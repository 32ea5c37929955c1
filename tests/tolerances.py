"""The parity gates the GPU tests use, in one place.

The stated gates are a max abs diff of 1e-4 for f32 inputs and of 1e-2 on
outputs (1e-3 on the f32 LSE) for bf16 inputs, against the oracle run on the
bf16-rounded values. A bf16 output is itself a rounding of its f32 value: where
one such rounding (half a bf16 ulp of the reference) fits under 1e-2, i.e.
|ref| < 4, the gate is the flat 1e-2; above that the flat bound is smaller
than the storage error alone, and the gate is one bf16 ulp of the reference.

f16 is not among the stated gates. Its gate is the bf16 one scaled by f16's
finer quantum (3 more mantissa bits, so its roundings of P and of the output
are 8x smaller): a flat 2e-3 wherever half an f16 ulp fits under it (|ref| < 8),
one f16 ulp of the reference above that.
"""
import numpy as np

ATOL_F32 = 1e-4
ATOL_BF16 = 1e-2
ATOL_F16 = 2e-3
ATOL_LSE_BF16 = 1e-3


def ulp(ref, mantissa_bits):
    """Spacing of the 16-bit float grid (mantissa_bits stored bits) at |ref|."""
    _, e = np.frexp(np.abs(np.asarray(ref, np.float64)))
    return np.ldexp(1.0, e - 1 - mantissa_bits)


def output_bound(ref, dtype):
    """Per-element bound on |gpu - ref| for a stage output of this dtype."""
    ref = np.asarray(ref, np.float64)
    if dtype == "f32":
        return np.full(ref.shape, ATOL_F32)
    atol, bits = (ATOL_BF16, 7) if dtype == "bf16" else (ATOL_F16, 10)
    u = ulp(ref, bits)
    return np.where(u / 2 <= atol, atol, u)


def lse_bound(dtype):
    return ATOL_F32 if dtype == "f32" else ATOL_LSE_BF16
