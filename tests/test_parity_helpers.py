"""The tolerance helpers of the GPU parity tests, pinned on the CPU: half a
bf16 ulp of a stored value agrees with the spacing of torch's bfloat16 grid,
and the rounding excess of a correctly rounded value is zero while a value
one ulp off keeps half an ulp of excess."""
import numpy as np
import torch

from _parity import half_ulp_bf16, rounding_excess


def _bf16_values(n=200_000, seed=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, generator=g) * torch.exp(torch.randn(n, generator=g) * 8)
    return x.to(torch.bfloat16)


def test_half_ulp_matches_bf16_grid_spacing():
    b = _bf16_values()
    b = b[b != 0]
    bits = b.view(torch.int16).to(torch.int32) & 0x7FFF
    # the next representable magnitude up: one more in the low mantissa bit
    nxt = (bits + 1).to(torch.int16).view(torch.bfloat16).to(torch.float64).numpy()
    mag = b.abs().to(torch.float64).numpy()
    ok = np.isfinite(nxt)
    assert np.array_equal(half_ulp_bf16(mag)[ok], (nxt - mag)[ok] / 2)
    assert np.array_equal(half_ulp_bf16(-mag), half_ulp_bf16(mag))
    assert half_ulp_bf16(np.array([0.0]))[0] == 0.0
    assert half_ulp_bf16(np.array([1.0]))[0] == 2.0 ** -8


def test_rounding_excess_of_correct_and_wrong_roundings():
    g = torch.Generator().manual_seed(1)
    # fp32 values (torch rounds fp32 -> bf16 once, to nearest even)
    exact = torch.randn(100_000, generator=g, dtype=torch.float32) * 3
    rounded = exact.to(torch.bfloat16).to(torch.float64).numpy()
    ex = exact.to(torch.float64).numpy()
    # round-to-nearest never moves a value by more than half an ulp of its result
    assert rounding_excess(rounded, ex).max() == 0.0
    # one ulp further away from the exact value leaves at least half an ulp of excess
    hu = half_ulp_bf16(rounded)
    step = np.where(rounded >= ex, 1.0, -1.0)
    off = rounded + step * 2 * hu
    keep = half_ulp_bf16(off) == hu            # the same binade as the correct rounding
    assert keep.mean() > 0.99
    assert (rounding_excess(off, ex)[keep] >= hu[keep]).all()
