"""Pins for the oracle's backward pass: central finite differences of the
forward definition, invariants, closed forms and a hand-worked example. CPU only."""

import json
import os

import numpy as np
import pytest

from oracle import attention_bwd, attention_bwd_varlen, attention_fwd, visible_limit

RNG = np.random.default_rng(7)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def loss(q, k, v, do, scale, causal):
    o, _ = attention_fwd(q, k, v, scale, causal)
    return float((o * do).sum())


def fd_grad(f, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        g[idx] = (f(xp) - f(xm)) / (2 * h)
    return g


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk,dqk,dv", [(4, 4, 3, 3), (6, 3, 4, 2), (3, 7, 5, 4), (9, 9, 8, 8), (16, 5, 6, 3)])
def test_gradients_match_finite_differences(nq, nk, dqk, dv, causal):
    q, k, v, do = rand(nq, dqk), rand(nk, dqk), rand(nk, dv), rand(nq, dv)
    s = 0.45
    g = attention_bwd(q, k, v, do, s, causal)
    fq = fd_grad(lambda x: loss(x, k, v, do, s, causal), q)
    fk = fd_grad(lambda x: loss(q, x, v, do, s, causal), k)
    fv = fd_grad(lambda x: loss(q, k, x, do, s, causal), v)
    for name, a, b in (("dq", g["dq"], fq), ("dk", g["dk"], fk), ("dv", g["dv"], fv)):
        den = max(np.linalg.norm(b), 1e-12)
        assert np.linalg.norm(a - b) / den < 1e-6, name


@pytest.mark.parametrize("causal", [False, True])
def test_row_term_two_ways(causal):
    # D_i = sum_j P_ij dP_ij must equal dO_i . O_i
    q, k, v, do = rand(20, 6), rand(17, 6), rand(17, 5), rand(20, 5)
    g = attention_bwd(q, k, v, do, 0.3, causal)
    o, _ = attention_fwd(q, k, v, 0.3, causal)
    np.testing.assert_allclose(g["D"], (o * do).sum(axis=1), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_dk_sums_to_zero(causal):
    # sum_j dS_ij = 0 for each row, so sum_j dK_j = scale * sum_i (sum_j dS_ij) q_i = 0
    q, k, v, do = rand(23, 7), rand(23, 7), rand(23, 4), rand(23, 4)
    g = attention_bwd(q, k, v, do, 0.8, causal)
    assert np.abs(g["dk"].sum(axis=0)).max() < 1e-12 * max(1.0, np.abs(g["dk"]).max())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk", [(6, 6), (8, 5)])
def test_zero_q_closed_form_dv(nq, nk, causal):
    # Q = 0: P_ij = 1/n_i over the n_i visible keys, so dV_j = sum_{i sees j} dO_i / n_i
    v, do = rand(nk, 3), rand(nq, 3)
    g = attention_bwd(np.zeros((nq, 4)), rand(nk, 4), v, do, 1.0, causal)
    lim = visible_limit(np.arange(nq), nq, nk, causal)
    want = np.zeros((nk, 3))
    for i in range(nq):
        if lim[i] > 0:
            want[: lim[i]] += do[i] / lim[i]
    np.testing.assert_allclose(g["dv"], want, rtol=1e-13, atol=1e-14)


def test_rows_without_keys_have_zero_gradients():
    q, k, v, do = rand(6, 4), rand(3, 4), rand(3, 2), rand(6, 2)
    g = attention_bwd(q, k, v, do, 1.0, True)
    assert np.all(g["dq"][:3] == 0)
    g2 = attention_bwd(q[3:], k, v, do[3:], 1.0, True)  # same visible pairs without the dead rows
    np.testing.assert_allclose(g["dk"], g2["dk"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(g["dv"], g2["dv"], rtol=1e-14, atol=1e-15)


def test_hand_worked_example(repo_root):
    gd = json.load(open(os.path.join(repo_root, "tests", "golden", "hand_worked_2x2.json")))
    inp = gd["inputs"]
    for causal, key in [(False, "noncausal"), (True, "causal")]:
        g = attention_bwd(inp["q"], inp["k"], inp["v"], inp["do"], inp["softmax_scale"], causal)
        for n in ("dq", "dk", "dv"):
            np.testing.assert_allclose(g[n], gd[key][n], rtol=1e-15, atol=1e-16)


def test_row_block_does_not_change_result():
    q, k, v, do = rand(37, 5), rand(41, 5), rand(41, 3), rand(37, 3)
    a = attention_bwd(q, k, v, do, 0.5, True)
    b = attention_bwd(q, k, v, do, 0.5, True, row_block=5)
    for n in ("dq", "dk", "dv"):
        np.testing.assert_allclose(a[n], b[n], rtol=1e-13, atol=1e-14)


def test_varlen_backward_matches_per_sequence():
    lens = [4, 7]
    cu = np.cumsum([0] + lens)
    q, k, v, do = rand(11, 2, 3), rand(11, 2, 3), rand(11, 2, 2), rand(11, 2, 2)
    dq, dk, dv = attention_bwd_varlen(q, k, v, do, cu, cu, 0.5, True)
    for s in range(2):
        a, b = cu[s], cu[s + 1]
        for h in range(2):
            g = attention_bwd(q[a:b, h], k[a:b, h], v[a:b, h], do[a:b, h], 0.5, True)
            np.testing.assert_array_equal(dq[a:b, h], g["dq"])
            np.testing.assert_array_equal(dk[a:b, h], g["dk"])
            np.testing.assert_array_equal(dv[a:b, h], g["dv"])
