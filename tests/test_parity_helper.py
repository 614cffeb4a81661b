"""CPU checks of the parity helper's bf16 storage allowance: exactly one bf16 rounding of the
reference passes with a zero max-abs budget, and an error beyond it still fails."""
import numpy as np
import pytest
import torch

from tests.parity import assert_close, bf16_half_ulp


def test_half_ulp_matches_bf16_spacing():
    x = torch.tensor([1.0, 1.5, 3.0, -0.75, 1e-3, 300.0], dtype=torch.float32)
    up = torch.nextafter(x.to(torch.bfloat16), torch.full_like(x, np.inf).to(torch.bfloat16))
    spacing = (up.double() - x.to(torch.bfloat16).double()).abs().numpy()
    assert np.array_equal(bf16_half_ulp(x.numpy()), spacing / 2)


def test_storage_rounding_alone_passes_and_more_fails():
    gen = torch.Generator().manual_seed(0)
    ref = torch.randn(4096, generator=gen, dtype=torch.float64)
    ref[7] = 40.0 + 2 ** -7  # about 40 times the RMS: its bf16 rounding alone is ~0.04 of it
    stored = ref.to(torch.bfloat16)
    rel, mx = assert_close("rounded", stored, ref.numpy(), max_tol=0.0)  # nothing beyond storage
    assert mx > 0  # the literal max-abs figure still sees the rounding
    bad = stored.clone()
    bad[100] = (ref[100] + 0.06 * ref.pow(2).mean().sqrt() + 0.05).to(torch.bfloat16)
    with pytest.raises(AssertionError):
        assert_close("beyond", bad, ref.numpy())
    # fp32 results get no allowance
    with pytest.raises(AssertionError):
        assert_close("fp32", stored.float(), ref.numpy(), max_tol=0.0)
