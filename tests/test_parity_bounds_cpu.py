"""The in-dtype parity bound itself: the correctly rounded oracle value always passes
it, and a value one unit in the last place off (at magnitudes where the absolute term
does not hide it) fails it -- so the bound is as tight as rounding allows."""
import numpy as np
import pytest
import torch

from parity_bounds import check_in_dtype


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_rounded_oracle_values_pass(dtype):
    g = torch.Generator().manual_seed(7)
    ref = (torch.randn(20000, generator=g, dtype=torch.float64) * torch.logspace(-4, 1, 20000, dtype=torch.float64))
    check_in_dtype(ref.to(dtype), ref.numpy())  # round-to-nearest-even of the exact value


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_one_ulp_off_fails(dtype):
    ref = torch.tensor([0.7, -1.3, 2.9, 3.6], dtype=torch.float64)
    for i in range(len(ref)):
        low = ref.to(dtype)
        bits = low.view(torch.int16).clone()
        # the next representable value on the far side of the rounded one from the
        # exact value: at least one ulp off, and an ulp exceeds |ref| * 2^-p + 1e-4 here
        away = (low[i].double() - ref[i]).abs() > 0 and (low[i].double().abs() > ref[i].abs())
        bits[i] += 1 if (away or low[i].double() == ref[i]) else -1
        off = bits.view(dtype)
        assert (off[i].double() - ref[i]).abs() >= (low[i].double() - ref[i]).abs()
        with pytest.raises(AssertionError):
            check_in_dtype(off, ref.numpy())


def test_non_finite_fails():
    ref = np.array([0.5, 0.25])
    with pytest.raises(AssertionError):
        check_in_dtype(torch.tensor([0.5, float("nan")], dtype=torch.bfloat16), ref)
