"""The parity metric itself (CPU): half-ulp of bf16 and the stored-bf16 allowance."""
import numpy as np
import torch

from tests.helpers import half_ulp_bf16, rel_err_bf16, rel_err_f32


def test_half_ulp_bf16_matches_torch_rounding():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-8, 8, 20000))
    r = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    # round-to-nearest never moves a value by more than half an ulp (torch rounds through
    # float32, which can add 2^-24 relative), and the bound is tight
    assert np.all(np.abs(r - x) <= half_ulp_bf16(x) * (1 + 2.0 ** -14))
    assert np.max(np.abs(r - x) / half_ulp_bf16(x)) > 0.99
    assert half_ulp_bf16(np.array([1.0]))[0] == 2.0 ** -8
    assert half_ulp_bf16(np.array([-5.0]))[0] == 2.0 ** -6
    assert half_ulp_bf16(np.array([8.0]))[0] == 2.0 ** -5


def test_exact_result_rounded_to_bf16_passes_only_with_the_storage_allowance():
    rng = np.random.default_rng(1)
    o = rng.standard_normal(100000) * 1.5
    g = torch.from_numpy(o).to(torch.bfloat16).to(torch.float64).numpy()
    assert rel_err_bf16(g, o, stored_bf16=True) == 0.0
    assert rel_err_bf16(g, o) > 1e-2          # the bare bound sees the storage rounding
    # a real computation error on top is still measured
    g2 = g.copy()
    g2[123] += 0.05
    assert rel_err_bf16(g2, o, stored_bf16=True) > 0.02


def test_f32_metric_floors_small_outputs_at_rms():
    o = np.array([1.0, -1.0, 1e-9])
    g = o + np.array([0.0, 0.0, 1e-6])
    assert rel_err_f32(g, o) < 2e-6


def test_two_bf16_roundings_may_differ_by_one_ulp():
    # two computations within 1e-3 rms of each other, each rounded to bf16, can land
    # one ulp apart near a rounding boundary; comparing them allows half an ulp each
    rng = np.random.default_rng(2)
    x = rng.standard_normal(100000) * 3.0
    a = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    b = torch.from_numpy(x + 1e-3 * rng.standard_normal(x.size)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.max(np.abs(a - b) / (2 * half_ulp_bf16(np.maximum(np.abs(a), np.abs(b))))) >= 0.999   # some flip
    assert rel_err_bf16(a, b, stored_bf16=True) > 1e-2        # one allowance is not enough
    assert rel_err_bf16(a, b, both_stored=True) < 2e-3        # two are, and the 1e-3 difference remains
