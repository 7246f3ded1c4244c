"""The error metrics the parity tests use (no GPU)."""
import numpy as np
import torch

from case_io import bf16_half_ulp, bf16_out_err, bf16_pair_err, normwise_err


def test_half_ulp_matches_bf16_spacing():
    x = np.array([1.0, 1.5, 2.0, 3.99, 0.25, 1e-3, 300.0])
    spacing = np.array([2.0 ** -7, 2.0 ** -7, 2.0 ** -6, 2.0 ** -6, 2.0 ** -9, 2.0 ** -17, 2.0])
    np.testing.assert_array_equal(bf16_half_ulp(x), spacing / 2)
    np.testing.assert_array_equal(bf16_half_ulp(-x), spacing / 2)


def test_bf16_rounding_of_exact_values_has_no_excess():
    rng = np.random.default_rng(0)
    ref = (rng.standard_normal(100000) * 3).astype(np.float32).astype(np.float64)  # one rounding to BF16
    x = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    assert normwise_err(x, ref) > 1e-3          # the raw metric sees the rounding
    assert bf16_out_err(x, ref) == 0.0          # the BF16-aware metric does not
    y = torch.from_numpy(ref * (1 + 1e-6)).to(torch.bfloat16).double().numpy()
    assert bf16_pair_err(x, y) == 0.0


def test_bf16_out_err_sees_real_errors():
    ref = np.linspace(-4, 4, 1001)
    x = torch.from_numpy(ref + 0.05).to(torch.bfloat16).double().numpy()
    assert bf16_out_err(x, ref) > 5e-3
