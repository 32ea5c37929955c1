"""The parity gates themselves, on CPU: flat where one rounding of the output
fits under the stated absolute bound, one ulp of the reference above."""
import numpy as np

from tolerances import output_bound, ulp


def test_bf16_gate():
    assert output_bound(0.0, "bf16") == 1e-2
    assert output_bound(1.0, "bf16") == 1e-2           # half ulp 2^-8 fits
    assert output_bound(3.99, "bf16") == 1e-2          # half ulp 2^-7 = 0.0078 fits
    assert output_bound(4.0, "bf16") == 2.0 ** -5      # half ulp 2^-6 = 0.0156 does not
    assert output_bound(-7.9, "bf16") == 2.0 ** -5
    assert output_bound(8.0, "bf16") == 2.0 ** -4
    assert ulp(1.0, 7) == 2.0 ** -7 and ulp(1.99, 7) == 2.0 ** -7


def test_f16_and_f32_gates():
    assert output_bound(7.99, "f16") == 2e-3           # half ulp 2^-9 fits
    assert output_bound(8.0, "f16") == 2.0 ** -7
    assert np.all(output_bound(np.array([0.0, 100.0]), "f32") == 1e-4)
