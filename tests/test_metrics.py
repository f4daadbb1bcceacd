"""The parity metrics themselves (CPU)."""
import numpy as np
import pytest
import torch

from tests.helpers import assert_bf16_rounding, check, rel_err_bf16, rel_err_f32


def test_bf16_metric_is_max_error_over_rms():
    o = np.array([3.0, -4.0, 0.0, 0.0])          # rms 2.5
    g = o + np.array([0.0, 0.05, 0.0, -0.01])
    assert rel_err_bf16(g, o) == pytest.approx(0.05 / 2.5)


def test_bare_bar_sees_the_bf16_storage_rounding():
    # an exactly computed output of rms about 1 rounded to bf16 misses the bare 2e-2 * rms
    # bar once |o| >= 8 (the bf16 spacing there is 2^-4): the bar then measures the output
    # format, which is why the tests compare the float32 outputs and check the bf16 ones
    # by rounding
    o = np.array([8.03] + [0.3] * 63)
    g = torch.from_numpy(o).to(torch.bfloat16).to(torch.float64).numpy()
    assert rel_err_bf16(g, o) > 2e-2
    assert rel_err_bf16(o + 1e-3, o) < 2e-2


def test_f32_metric_floors_small_outputs_at_rms():
    o = np.array([1.0, -1.0, 1e-9])
    g = o + np.array([0.0, 0.0, 1e-6])
    assert rel_err_f32(g, o) < 2e-6


def test_check_applies_the_bare_bar():
    o = np.linspace(-2, 2, 100)
    check(o + 1e-3, o, "bf16", "within")
    with pytest.raises(AssertionError):
        check(o + 0.05, o, "bf16", "beyond")
    with pytest.raises(AssertionError):
        check(o * (1 + 2e-4), o, "f32", "beyond f32")


def test_bf16_rounding_check_is_bit_exact():
    rng = np.random.default_rng(3)
    f = torch.from_numpy(rng.standard_normal(5000).astype(np.float32) * 3)
    assert_bf16_rounding(f.to(torch.bfloat16), f, "rne")
    # a value on the other side of a rounding boundary (one ulp away) fails
    b = f.to(torch.bfloat16)
    b.view(torch.int16)[17] += 1
    with pytest.raises(AssertionError):
        assert_bf16_rounding(b, f, "one ulp off")
    # truncation instead of rounding fails
    trunc = (f.view(torch.int32) & ~0xFFFF).view(torch.float32).to(torch.bfloat16)
    with pytest.raises(AssertionError):
        assert_bf16_rounding(trunc, f, "truncated")
