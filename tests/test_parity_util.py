"""The parity bars themselves, on the CPU: the element bound for bf16
outputs (max-abs 1e-2; faithful rounding where |oracle| >= 4, where the bf16
grid is coarser than 1e-2) and the relative-L2 bound."""
import numpy as np
import pytest
import torch

from parity_util import assert_attention_close, bf16_ulp, violations


def _bf16(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)


def test_bf16_ulp_is_the_grid_spacing():
    for x in (1.0, 3.9, 4.0, 4.58, 7.99, 8.0, 100.0, -5.0):
        b = _bf16(x).float()
        nxt = torch.nextafter(b.to(torch.bfloat16), torch.tensor(1e30, dtype=torch.bfloat16))
        assert float(nxt.float() - b) == pytest.approx(bf16_ulp(np.array([float(b)]))[0])


def test_both_bf16_neighbours_of_a_large_value_pass_and_the_next_fails():
    ref = np.array([4.57943])  # between the bf16 values 4.5625 and 4.59375
    lo, hi, far = 4.5625, 4.59375, 4.53125
    for v in (lo, hi):
        assert not violations(np.abs(np.array([v]) - ref), ref, torch.bfloat16)[0].any()
    assert violations(np.abs(np.array([far]) - ref), ref, torch.bfloat16)[0].all()
    assert_attention_close(_bf16([lo]), ref, torch.bfloat16)
    with pytest.raises(AssertionError):
        assert_attention_close(_bf16([far]), ref, torch.bfloat16)


def test_small_values_keep_the_flat_bound():
    ref = np.array([1.0, -2.5, 0.01])
    ok = ref + np.array([0.0099, -0.0099, 0.0099])
    bad = ref + np.array([0.0, 0.0101, 0.0])
    assert not violations(np.abs(ok - ref), ref, torch.bfloat16)[0].any()
    assert violations(np.abs(bad - ref), ref, torch.bfloat16)[0].tolist() == [False, True, False]


def test_fp32_bounds_and_relative_l2():
    ref = np.linspace(-1, 1, 1000)
    assert_attention_close(torch.tensor(ref, dtype=torch.float32), ref, torch.float32)
    with pytest.raises(AssertionError):
        assert_attention_close(torch.tensor(ref + 2e-5, dtype=torch.float32), ref, torch.float32)
    # every element within 1e-2 but the relative L2 above 5e-3
    with pytest.raises(AssertionError):
        assert_attention_close(_bf16(ref * 0 + 0.5 + 0.009), ref * 0 + 0.5, torch.bfloat16)
