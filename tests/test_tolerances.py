"""The parity gates themselves, on CPU: the stated absolute bound plus one
rounding of the 16-bit output (half an ulp of the reference)."""
import numpy as np

from tolerances import output_bound, ulp


def test_bf16_gate():
    assert ulp(1.0, 7) == 2.0 ** -7 and ulp(1.99, 7) == 2.0 ** -7 and ulp(0.5, 7) == 2.0 ** -8
    assert output_bound(0.0, "bf16") <= 1e-2 + 1e-30
    assert output_bound(1.0, "bf16") == 1e-2 + 2.0 ** -8
    assert output_bound(3.99, "bf16") == 1e-2 + 2.0 ** -7
    assert output_bound(-4.0, "bf16") == 1e-2 + 2.0 ** -6
    # never looser than 1e-2 + 2^-8 |ref|, the earlier form
    r = np.linspace(-40, 40, 100001)
    assert np.all(output_bound(r, "bf16") <= 1e-2 + 2.0 ** -8 * np.abs(r) + 1e-15)


def test_f16_and_f32_gates():
    assert output_bound(7.99, "f16") == 2e-3 + 2.0 ** -9
    assert output_bound(1.0, "f16") == 2e-3 + 2.0 ** -11
    assert np.all(output_bound(np.array([0.0, 100.0]), "f32") == 1e-4)
