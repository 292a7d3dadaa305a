"""The comparison used by the GPU parity tests, checked on the CPU."""
import numpy as np
import pytest
import torch

from parity_util import compare, round_to_bf16


def test_round_to_bf16_matches_torch_on_fp32_values():
    x = torch.randn(100000, dtype=torch.float32) * 10
    ours = round_to_bf16(x.double().numpy())
    theirs = x.to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(ours, theirs)


def test_round_to_bf16_ties_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to 1 (even mantissa)
    assert round_to_bf16(np.array([1 + 2 ** -8]))[0] == 1.0
    assert round_to_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6


def test_compare_accepts_best_rounding_and_rejects_planted_error():
    rng = np.random.default_rng(0)
    o_ref = rng.normal(size=(2, 3, 5, 8)) * 3
    lse_ref = rng.normal(size=(2, 3, 5))
    o_best = torch.from_numpy(round_to_bf16(o_ref)).to(torch.bfloat16)
    stats = compare(o_best, torch.from_numpy(lse_ref).float(), o_ref, lse_ref)
    assert stats["max_excess_dO_from_4"] <= 1e-12 and stats["max_abs_dO_below_4"] <= 2 ** -7
    bad = o_ref.copy()
    bad[1, 2, 3, 4] += 0.05
    with pytest.raises(AssertionError):
        compare(torch.from_numpy(bad).to(torch.bfloat16), torch.from_numpy(lse_ref).float(), o_ref, lse_ref)
    with pytest.raises(AssertionError):
        compare(o_best, torch.from_numpy(lse_ref + 2e-3).float(), o_ref, lse_ref)


def test_compare_requires_zero_rows_and_minus_inf_where_no_keys():
    o_ref = np.zeros((1, 1, 2, 4)); o_ref[0, 0, 1] = 1.0
    lse_ref = np.array([[[-np.inf, 0.5]]])
    good = torch.from_numpy(o_ref).to(torch.bfloat16)
    compare(good, torch.tensor([[[-float("inf"), 0.5]]]), o_ref, lse_ref)
    with pytest.raises(AssertionError):
        compare(good, torch.tensor([[[0.0, 0.5]]]), o_ref, lse_ref)


def test_plain_bound_below_4_and_floor_allowance_from_4():
    lse_ref = np.zeros((1, 1, 1))
    lse = torch.zeros((1, 1, 1))
    # |O_ref| < 4: the next bf16 value up is 0.0101 away -> over the plain 1e-2 bound (the rounding
    # floor there is 0.0055, so an allowance over the floor would have let it through)
    o_ref = np.array([[[[3.0 + 0.0055]]]])
    with pytest.raises(AssertionError):
        compare(torch.tensor([[[[3.015625]]]]).to(torch.bfloat16), lse, o_ref, lse_ref)
    stats = compare(torch.tensor([[[[3.0]]]]).to(torch.bfloat16), lse, o_ref, lse_ref)
    assert abs(stats["max_abs_dO_by_bin"]["[2,4)"][1] - 0.0055) < 1e-12
    # |O_ref| >= 4: no bf16 value is within 1e-2 of 5.012 (floor 0.012), so one spacing up (0.0193 away)
    # passes as 0.0073 over the floor; two spacings up (0.0505 away) do not
    o_ref = np.array([[[[5.0 + 0.012]]]])
    stats = compare(torch.tensor([[[[5.03125]]]]).to(torch.bfloat16), lse, o_ref, lse_ref)
    assert abs(stats["max_excess_dO_from_4"] - (0.01925 - 0.012)) < 1e-12
    with pytest.raises(AssertionError):
        compare(torch.tensor([[[[5.0625]]]]).to(torch.bfloat16), lse, o_ref, lse_ref)


def test_statistics_are_binned_by_reference_magnitude():
    o_ref = np.array([0.5, 1.5, 3.0, 6.0, 10.0]).reshape(1, 1, 5, 1)
    o = torch.from_numpy(round_to_bf16(o_ref)).to(torch.bfloat16)
    stats = compare(o, torch.zeros(1, 1, 5), o_ref, np.zeros((1, 1, 5)))
    assert sorted(stats["max_abs_dO_by_bin"]) == sorted(["[0,1)", "[1,2)", "[2,4)", "[4,8)", "[8,inf)"])
    assert all(n == 1 and dmax == 0.0 for n, dmax in stats["max_abs_dO_by_bin"].values())
