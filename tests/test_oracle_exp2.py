"""Pins for the oracle's exp2 emulation (Cody-Waite split + degree-3 polynomial). CPU only."""

import numpy as np
import pytest
import torch

from oracle import exp2_exact, exp2_poly, fit_exp2_poly_remez


@pytest.fixture(scope="module")
def fit():
    return fit_exp2_poly_remez()


def test_fit_equioscillates(fit):
    # Equioscillation theorem: with 3 free coefficients the unique minimax error
    # alternates in sign with equal magnitude on 4 points, and is nowhere larger.
    c, ref = fit["c"], fit["ref"]
    assert c[0] == 1.0
    p = ((c[3] * ref + c[2]) * ref + c[1]) * ref + c[0]
    e = p / np.exp2(ref) - 1.0
    assert np.all(np.sign(e[:-1]) != np.sign(e[1:]))
    np.testing.assert_allclose(np.abs(e), fit["level"], rtol=1e-9)
    assert fit["max_rel_err"] <= fit["level"] * (1 + 1e-9)
    # A degree-3 fit of 2^f on [0,1) sits near 1e-4 (wittx: ~600x the hardware unit's error).
    assert 5e-5 < fit["max_rel_err"] < 1.5e-4


def test_integers_are_exact(fit):
    n = np.arange(-126, 9, dtype=np.float64)
    np.testing.assert_array_equal(exp2_poly(n, fit["c"]), np.exp2(n))


def test_relative_error_bound_over_softmax_range(fit):
    x = np.concatenate([np.linspace(-126, 8, 2_000_003), np.random.default_rng(0).uniform(-30, 8, 1_000_000)])
    rel = np.abs(exp2_poly(x, fit["c"]) / exp2_exact(x) - 1.0)
    assert rel.max() <= fit["max_rel_err"] * (1 + 1e-9)


def test_bf16_agreement_with_exact(fit):
    # wittx, section 用软件"伪造"硬件指令: in bf16 the cubic and the exact exponential
    # agree on 99% of inputs (a whole-percent figure: anything that rounds to 99%).
    x = np.random.default_rng(1).uniform(-16, 8, 2_000_000)
    ex = torch.from_numpy(exp2_exact(x)).to(torch.bfloat16)
    po = torch.from_numpy(exp2_poly(x, fit["c"])).to(torch.bfloat16)
    agree = (ex == po).double().mean().item()
    assert round(agree * 100) == 99, agree


def test_clamp_below_minus_127(fit):
    y = exp2_poly(np.array([-200.0, -127.0, -1e30]), fit["c"])
    assert np.all(y >= 0) and np.all(y < 2.0 ** -126)
