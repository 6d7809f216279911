"""Pins for the oracle's forward pass: closed forms, invariants, a hand-worked
example, and agreement of the conditional-rescale algorithm with the
definition. CPU only."""

import json
import math
import os

import numpy as np
import pytest

from oracle import attention_fwd, attention_fwd_online, attention_fwd_varlen, visible_limit

RNG = np.random.default_rng(20260311)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


SHAPES = [  # (nq, nk, d_qk, d_v)
    (5, 5, 4, 4),
    (7, 3, 8, 5),
    (3, 9, 6, 2),
    (130, 130, 16, 16),
    (257, 300, 12, 7),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_constant_v_gives_constant_o(shape, causal):
    nq, nk, dqk, dv = shape
    c = rand(dv)
    o, lse = attention_fwd(rand(nq, dqk), rand(nk, dqk), np.tile(c, (nk, 1)), 0.3, causal)
    live = visible_limit(np.arange(nq), nq, nk, causal) > 0
    np.testing.assert_allclose(o[live], np.tile(c, (live.sum(), 1)), rtol=1e-13, atol=1e-13)
    assert np.all(o[~live] == 0) and np.all(np.isneginf(lse[~live]))


@pytest.mark.parametrize("nq", [1, 4])
def test_single_key(nq):
    q, k, v = rand(nq, 6), rand(1, 6), rand(1, 3)
    o, lse = attention_fwd(q, k, v, 0.7, False)
    np.testing.assert_allclose(o, np.tile(v[0], (nq, 1)), rtol=1e-14)
    np.testing.assert_allclose(lse, 0.7 * (q @ k[0]), rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk", [(6, 6), (4, 9), (9, 4)])
def test_zero_q_gives_prefix_mean(nq, nk, causal):
    v = rand(nk, 3)
    o, lse = attention_fwd(np.zeros((nq, 5)), rand(nk, 5), v, 0.5, causal)
    for i in range(nq):
        n = int(visible_limit(i, nq, nk, causal))
        if n == 0:
            assert np.all(o[i] == 0) and np.isneginf(lse[i])
            continue
        np.testing.assert_allclose(o[i], v[:n].mean(axis=0), rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse[i], math.log(n), rtol=1e-14)


def test_one_hot_dominant_logit_selects_its_value_row():
    # k_j = e_j; q_i = 80 e_{pi(i)}: logit 80 for key pi(i), 0 elsewhere -> weight 1 - 7e^-80.
    d = 8
    k = np.eye(d)
    perm = np.array([3, 0, 7, 1, 6, 2, 5, 4])
    q = 80.0 * np.eye(d)[perm]
    v = rand(d, 4)
    o, lse = attention_fwd(q, k, v, 1.0, False)
    np.testing.assert_allclose(o, v[perm], rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(lse, 80.0, rtol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal):
    # V = identity turns O into the probability matrix P itself.
    nq, nk = 9, 6
    o, _ = attention_fwd(rand(nq, 4), rand(nk, 4), np.eye(nk), 0.9, causal)
    lim = visible_limit(np.arange(nq), nq, nk, causal)
    for i in range(nq):
        if lim[i] == 0:
            continue
        assert np.all(o[i] >= 0)
        assert np.all(o[i, lim[i]:] == 0)
        assert abs(o[i].sum() - 1.0) < 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_key_shift_invariance(causal):
    # k_j -> k_j + c changes every logit of row i by scale * q_i . c: O unchanged, LSE shifts.
    nq, nk, d = 11, 13, 6
    q, k, v, c = rand(nq, d), rand(nk, d), rand(nk, 3), rand(d) * 5
    o1, l1 = attention_fwd(q, k, v, 0.4, causal)
    o2, l2 = attention_fwd(q, k + c, v, 0.4, causal)
    live = np.isfinite(l1)
    np.testing.assert_allclose(o2, o1, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(l2[live], l1[live] + 0.4 * (q[live] @ c), rtol=1e-12, atol=1e-12)


def test_causal_rows_without_keys_and_single_query():
    q, k, v = rand(6, 4), rand(3, 4), rand(3, 2)
    o, lse = attention_fwd(q, k, v, 1.0, True)  # bottom-right: rows 0..2 see nothing
    assert np.all(o[:3] == 0) and np.all(np.isneginf(lse[:3]))
    assert np.all(np.isfinite(lse[3:]))
    # a single query row sees every key under the bottom-right causal mask
    o1, l1 = attention_fwd(q[:1], k, v, 1.0, True)
    o0, l0 = attention_fwd(q[:1], k, v, 1.0, False)
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(l1, l0)


def test_empty_inputs():
    o, lse = attention_fwd(np.zeros((0, 4)), rand(3, 4), rand(3, 2), 1.0, False)
    assert o.shape == (0, 2) and lse.shape == (0,)
    o, lse = attention_fwd(rand(3, 4), np.zeros((0, 4)), np.zeros((0, 2)), 1.0, False)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_hand_worked_example(repo_root):
    g = json.load(open(os.path.join(repo_root, "tests", "golden", "hand_worked_2x2.json")))
    inp = g["inputs"]
    for causal, key in [(False, "noncausal"), (True, "causal")]:
        o, lse = attention_fwd(inp["q"], inp["k"], inp["v"], inp["softmax_scale"], causal)
        np.testing.assert_allclose(o, g[key]["o"], rtol=1e-15, atol=1e-16)
        np.testing.assert_allclose(lse, g[key]["lse"], rtol=1e-15, atol=1e-16)


def test_row_block_does_not_change_result():
    q, k, v = rand(37, 5), rand(41, 5), rand(41, 3)
    a = attention_fwd(q, k, v, 0.5, True)
    b = attention_fwd(q, k, v, 0.5, True, row_block=4)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-13, atol=1e-14)  # BLAS may block sums differently
    np.testing.assert_allclose(a[1], b[1], rtol=1e-13, atol=1e-14)


# --- conditional-rescale online algorithm vs the definition -----------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("tile_n,threshold", [(128, 8.0), (4, 8.0), (3, 0.0), (5, 1e9)])
def test_online_equals_definition(shape, causal, tile_n, threshold):
    nq, nk, dqk, dv = shape
    q, k, v = rand(nq, dqk), rand(nk, dqk, scale=2.0), rand(nk, dv)
    o_ref, l_ref = attention_fwd(q, k, v, 0.6, causal)
    o, l, _ = attention_fwd_online(q, k, v, 0.6, causal, tile_n=tile_n, threshold=threshold)
    live = np.isfinite(l_ref)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l[live], l_ref[live], rtol=1e-12, atol=1e-13)
    assert np.all(np.isneginf(l[~live]))


def test_online_keeps_probabilities_bounded_and_counts_rescales():
    # Keys whose logits grow along the sequence force the running max up.
    nq, nk, d = 16, 64, 4
    q = np.abs(rand(nq, d)) + 0.5
    k = np.outer(np.arange(nk) * 0.05, np.ones(d))  # logit grows ~3 (log2) per tile of 8
    v = rand(nk, 2)
    _, _, st8 = attention_fwd_online(q, k, v, 1.0, False, tile_n=8, threshold=8.0)
    _, _, st0 = attention_fwd_online(q, k, v, 1.0, False, tile_n=8, threshold=0.0)
    assert st0["rescales"] == st0["opportunities"]  # strictly growing max: rescale at every tile
    assert 0 < st8["rescales"] < st0["rescales"]     # the threshold skips some of them
    _, _, stn = attention_fwd_online(rand(nq, d), rand(nk, d), v, 0.5, False, tile_n=8, threshold=8.0)
    assert stn["rescales"] == 0  # N(0,1) logits never rise 8 (log2) above the first tile's max


def test_outlier_keys_force_rescales():
    import torch
    import workloads
    w = workloads.dense_d128(1024, causal=False, outlier=True).with_(batch=1, heads=1)
    t = workloads.make_dense(w, with_do=False)
    q, k, v = (t[n][0, :, 0].double().numpy() for n in ("q", "k", "v"))
    o, l, st = attention_fwd_online(q, k, v, w.scale, False)
    o_ref, l_ref = attention_fwd(q, k, v, w.scale, False)
    assert st["rescales"] > 0
    np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-12)
    del torch


def test_varlen_is_blockwise_and_independent():
    lens = [5, 1, 9]
    cu = np.cumsum([0] + lens)
    H = 2
    q, k, v = rand(cu[-1], H, 4), rand(cu[-1], H, 4), rand(cu[-1], H, 3)
    o, lse = attention_fwd_varlen(q, k, v, cu, cu, 0.5, True)
    for s in range(3):
        for h in range(H):
            a, b = cu[s], cu[s + 1]
            oo, ll = attention_fwd(q[a:b, h], k[a:b, h], v[a:b, h], 0.5, True)
            np.testing.assert_array_equal(o[a:b, h], oo)
            np.testing.assert_array_equal(lse[h, a:b], ll)
    # perturbing the last sequence leaves the others untouched
    k2 = k.copy()
    k2[cu[2]:] += 3.0 * rand(cu[-1] - cu[2], H, 4)
    o2, _ = attention_fwd_varlen(q, k2, v, cu, cu, 0.5, True)
    np.testing.assert_array_equal(o2[: cu[2]], o[: cu[2]])
    assert not np.allclose(o2[cu[2]:], o[cu[2]:])
