"""The GPU parity checks themselves (CPU only): the forward check enforces the
stated tolerance against the unrounded fp64 oracle, widened only by half a
bf16 ulp where that exceeds 1e-2, and the gradient check the relative
Frobenius bound."""
import numpy as np
import pytest
import torch

from parity import bf16_half_ulp, check_fwd, check_grads


def _bf16(x):
    return torch.from_numpy(x).to(torch.bfloat16).double().numpy()


def test_half_ulp_values():
    # bf16 keeps 8 significant bits: spacing 2^-7 on [1, 2), 2^-5 on [4, 8)
    assert bf16_half_ulp(np.array([1.0]))[0] == 2.0 ** -8
    assert bf16_half_ulp(np.array([1.99]))[0] == 2.0 ** -8
    assert bf16_half_ulp(np.array([-5.0]))[0] == 2.0 ** -6
    assert bf16_half_ulp(np.array([0.3]))[0] == 2.0 ** -10


def test_correctly_rounded_output_passes_even_above_four():
    rng = np.random.default_rng(0)
    o_ref = rng.normal(size=(64, 16)) * 0.3
    o_ref[::7, 3] = rng.uniform(4.0, 7.9, size=o_ref[::7, 3].shape)  # |O| >= 4: half an ulp exceeds 1e-2
    lse = rng.normal(size=64)
    stats = check_fwd(torch.from_numpy(_bf16(o_ref)), torch.from_numpy(lse.astype(np.float32)), o_ref, lse)
    assert stats["o_max"] > 1e-2  # the widening was needed and applied


def test_rejects_an_error_just_above_the_bound():
    o_ref = np.full((4, 8), 0.5)
    o = o_ref.copy()
    o[2, 3] += 0.011  # above 1e-2, and half an ulp at 0.5 is only 2^-10
    lse = np.zeros(4)
    with pytest.raises(AssertionError):
        check_fwd(torch.from_numpy(o), torch.from_numpy(lse), o_ref, lse)


def test_rejects_a_full_ulp_off_at_large_magnitude():
    o_ref = np.full((2, 4), 5.0 + 2.0 ** -6)  # halfway between two bf16 values (spacing 2^-5)
    o = np.full_like(o_ref, 5.0 + 2.0 ** -5 + 2.0 ** -5)  # one step beyond the nearer neighbour
    lse = np.zeros(2)
    with pytest.raises(AssertionError):
        check_fwd(torch.from_numpy(o), torch.from_numpy(lse), o_ref, lse)


def test_rejects_a_mean_error_above_1e3():
    o_ref = np.zeros((32, 32))
    o = o_ref + 2e-3  # every element within 1e-2, mean 2e-3
    lse = np.zeros(32)
    with pytest.raises(AssertionError):
        check_fwd(torch.from_numpy(o), torch.from_numpy(lse), o_ref, lse)


def test_lse_and_empty_rows():
    o_ref = np.zeros((3, 4))
    lse_ref = np.array([0.5, -np.inf, 1.0])
    check_fwd(torch.from_numpy(o_ref), torch.from_numpy(lse_ref.copy()), o_ref, lse_ref)
    with pytest.raises(AssertionError):  # a dead row must stay -inf
        check_fwd(torch.from_numpy(o_ref), torch.from_numpy(np.array([0.5, 0.0, 1.0])), o_ref, lse_ref)
    with pytest.raises(AssertionError):  # LSE off by 2e-3
        check_fwd(torch.from_numpy(o_ref), torch.from_numpy(np.array([0.502, -np.inf, 1.0])), o_ref, lse_ref)


def test_gradient_bound():
    rng = np.random.default_rng(1)
    ref = {n: rng.normal(size=(16, 8)) for n in ("dq", "dk", "dv")}
    ok = {n: torch.from_numpy(x * (1 + 5e-3)) for n, x in ref.items()}
    check_grads(ok, ref)
    bad = dict(ok)
    bad["dk"] = torch.from_numpy(ref["dk"] * (1 + 2e-2))
    with pytest.raises(AssertionError):
        check_grads(bad, ref)
