"""The per-element bound the GPU parity tests apply (gpu_util.bound): the
stated max-abs bound wherever the output type can meet it, and otherwise
half an ulp of the output type at the exact value plus a fifth of the stated
bound.  Pinned here against the types' own rounding (torch's conversions)."""
import numpy as np
import pytest
import torch

from gpu_util import TOL, bound


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_stated_bound_wherever_rounding_leaves_room(dtype):
    # below 4 in magnitude half an ulp plus the arithmetic share stays under
    # the stated bound, which then applies unchanged
    x = np.linspace(-3.999, 3.999, 20001)
    assert np.all(bound(x, dtype) == TOL[dtype])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_bound_covers_correct_rounding(dtype):
    # the exact value rounded to the output type (round to nearest even) is
    # always within the bound, and never with less than a fifth of the
    # stated bound to spare where the bound exceeds the stated one
    rng = np.random.default_rng(5)
    x = rng.normal(0.0, 3.0, 200000) * np.exp2(rng.integers(-4, 5, 200000))
    # fp32 values (what the kernels round), so that the conversion rounds once
    x = x[np.abs(x) < 60000].astype(np.float32).astype(np.float64)
    r = torch.from_numpy(x).float().to(dtype).double().numpy()
    err = np.abs(r - x)
    b = bound(x, dtype)
    assert np.all(err <= b)
    wide = b > TOL[dtype]
    assert np.all(err[wide] <= b[wide] - TOL[dtype] / 5 + 1e-15)


def test_values_from_the_failing_case():
    # bf16: -4.0787841... lies between -4.0625 and -4.09375 (ulp 1/32 on
    # [4, 8)); round to nearest gives -4.09375, 0.01497 away
    x = -4.078784141252045
    r = float(torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).double())
    assert r == -4.09375 and abs(r - x) > TOL[torch.bfloat16]
    assert abs(bound(np.array(x), torch.bfloat16) - (2.0 ** -6 + 2e-3)) < 1e-15
    # fp16 at 5.0: half an ulp is 2^-9
    assert abs(bound(np.array(5.0), torch.float16) - (2.0 ** -9 + 4e-4)) < 1e-15
