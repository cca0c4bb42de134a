"""The per-element max-abs bar of the GPU parity tests: 1e-2, or one step of
the 16-bit output grid where that step is coarser.  The grid step is checked
here against the formats themselves: the next representable value above |x|,
found by incrementing the bit pattern."""
import numpy as np
import torch

from gpu_helpers import grid_spacing, max_abs_bound


def _next_up_gap(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    t = torch.from_numpy(np.abs(x)).to(dtype)
    bits = t.view(torch.int16)
    up = (bits + 1).view(dtype)
    return (up.double() - t.double()).numpy()


def test_grid_spacing_matches_the_formats():
    rng = np.random.default_rng(3)
    for dtype, fmt, lo, hi in ((torch.bfloat16, "bf16", -30, 30), (torch.float16, "f16", -13, 15)):
        x = np.ldexp(rng.uniform(1.0, 2.0, 20000), rng.integers(lo, hi, 20000)) * rng.choice([-1, 1], 20000)
        x = torch.from_numpy(x).to(dtype).double().numpy()          # values on the grid
        assert np.array_equal(grid_spacing(x, fmt), _next_up_gap(x, dtype))


def test_bar_is_flat_where_the_grid_is_fine():
    x = np.array([0.0, 0.1, -0.7, 1.0, 1.999])
    assert np.all(max_abs_bound(x) == 1e-2)
    assert np.all(max_abs_bound(np.array([2.0, 3.9, -15.0]), "f16") == 1e-2)
    assert np.all(max_abs_bound(np.array([2.0, -3.9])) == 2.0 ** -6)
    assert np.all(max_abs_bound(np.array([4.0, 7.5])) == 2.0 ** -5)
