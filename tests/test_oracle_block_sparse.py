"""Pins for the oracle's block-sparse mask (block lists → key visibility) and its
use in the forward definition. The references here are independent computations:
slicing the listed keys out and attending over them alone, and a brute-force
per-row softmax in plain Python."""
import math

import numpy as np
import pytest

from oracle import attention_fwd, block_sparse_visible, visible_limit


def rand(*shape, seed=0):
    return np.random.default_rng(seed + sum(shape)).standard_normal(shape)


def test_all_blocks_listed_is_the_dense_result():
    nq, nk = 300, 400
    q, k, v = rand(nq, 8), rand(nk, 8, seed=1), rand(nk, 4, seed=2)
    nkb = math.ceil(nk / 128)
    cnt = np.full(math.ceil(nq / 256), nkb)
    idx = np.tile(np.arange(nkb), (cnt.shape[0], 1))
    vis = block_sparse_visible(nq, nk, cnt, idx)
    assert vis.all()
    for causal in (False, True):
        o1, l1 = attention_fwd(q, k, v, 0.4, causal, visible=vis)
        o0, l0 = attention_fwd(q, k, v, 0.4, causal)
        assert np.array_equal(o1, o0) and np.array_equal(l1, l0)


@pytest.mark.parametrize("blocks", [[1], [0, 3], [3, 1], [2]])
def test_listed_blocks_equal_attention_over_the_sliced_keys(blocks):
    nq, nk = 200, 470  # 4 key blocks, the last one ragged (86 keys)
    q, k, v = rand(nq, 6), rand(nk, 6, seed=3), rand(nk, 5, seed=4)
    vis = block_sparse_visible(nq, nk, [len(blocks)], [blocks])
    keys = np.concatenate([np.arange(b * 128, min(nk, (b + 1) * 128)) for b in sorted(blocks)])
    o, lse = attention_fwd(q, k, v, 0.7, False, visible=vis)
    o_ref, l_ref = attention_fwd(q, k[keys], v[keys], 0.7, False)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, l_ref, rtol=1e-12, atol=1e-12)


def test_each_query_block_uses_its_own_list():
    nq, nk = 512, 384
    q, k, v = rand(nq, 4), rand(nk, 4, seed=5), rand(nk, 3, seed=6)
    vis = block_sparse_visible(nq, nk, [1, 2], [[2, 0], [0, 1]])
    o, _ = attention_fwd(q, k, v, 1.0, False, visible=vis)
    o_a, _ = attention_fwd(q[:256], k[256:], v[256:], 1.0, False)
    o_b, _ = attention_fwd(q[256:], k[:256], v[:256], 1.0, False)
    np.testing.assert_allclose(o[:256], o_a, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(o[256:], o_b, rtol=1e-12, atol=1e-12)


def test_empty_list_and_out_of_range_entries_see_nothing():
    nq, nk = 10, 200
    q, k, v = rand(nq, 4), rand(nk, 4, seed=7), rand(nk, 2, seed=8)
    for cnt, idx in (([0], [[1, 0]]), ([2], [[-1, 2]]), ([1], [[5]])):
        vis = block_sparse_visible(nq, nk, cnt, idx)
        assert not vis.any()
        o, lse = attention_fwd(q, k, v, 1.0, False, visible=vis)
        assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_causal_and_block_mask_combine_brute_force():
    nq, nk = 300, 300
    q, k, v = rand(nq, 3), rand(nk, 3, seed=9), rand(nk, 2, seed=10)
    cnt, idx = [2, 1], [[0, 2], [1, 0]]
    vis = block_sparse_visible(nq, nk, cnt, idx)
    o, lse = attention_fwd(q, k, v, 0.5, True, visible=vis)
    lim = visible_limit(np.arange(nq), nq, nk, True)
    for i in (0, 5, 127, 128, 255, 256, 280, 299):
        blocks = idx[i // 256][:cnt[i // 256]]
        js = [j for j in range(nk) if j < lim[i] and (j // 128) in blocks]
        if not js:
            assert np.all(o[i] == 0) and np.isneginf(lse[i])
            continue
        a = [0.5 * sum(q[i, d] * k[j, d] for d in range(3)) for j in js]
        m = max(a)
        w = [math.exp(x - m) for x in a]
        s = sum(w)
        ref = [sum(w[t] * v[js[t], c] for t in range(len(js))) / s for c in range(2)]
        assert abs(lse[i] - (m + math.log(s))) < 1e-12
        np.testing.assert_allclose(o[i], ref, rtol=1e-12, atol=1e-12)


def test_backward_all_blocks_listed_is_the_dense_result():
    from oracle import attention_bwd
    nq, nk = 300, 260
    q, k, v, do = rand(nq, 5), rand(nk, 5, seed=11), rand(nk, 3, seed=12), rand(nq, 3, seed=13)
    nkb = math.ceil(nk / 128)
    cnt = np.full(math.ceil(nq / 256), nkb)
    vis = block_sparse_visible(nq, nk, cnt, np.tile(np.arange(nkb), (cnt.shape[0], 1)))
    for causal in (False, True):
        g1 = attention_bwd(q, k, v, do, 0.6, causal, visible=vis)
        g0 = attention_bwd(q, k, v, do, 0.6, causal)
        for n in ("dq", "dk", "dv"):
            assert np.array_equal(g1[n], g0[n])


@pytest.mark.parametrize("blocks", [[1], [0, 2], [2, 0]])
def test_backward_equals_gradients_over_the_sliced_keys(blocks):
    # one query block listing some key blocks: dQ, and dK/dV on the listed keys, are the
    # gradients of attention over those keys alone; every other key gets zero gradient
    from oracle import attention_bwd
    nq, nk = 180, 300
    q, k, v, do = rand(nq, 4), rand(nk, 4, seed=14), rand(nk, 3, seed=15), rand(nq, 3, seed=16)
    vis = block_sparse_visible(nq, nk, [len(blocks)], [blocks])
    keys = np.concatenate([np.arange(b * 128, min(nk, (b + 1) * 128)) for b in sorted(blocks)])
    g = attention_bwd(q, k, v, do, 0.8, False, visible=vis)
    r = attention_bwd(q, k[keys], v[keys], do, 0.8, False)
    np.testing.assert_allclose(g["dq"], r["dq"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(g["dk"][keys], r["dk"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(g["dv"][keys], r["dv"], rtol=1e-11, atol=1e-12)
    rest = np.setdiff1d(np.arange(nk), keys)
    assert np.all(g["dk"][rest] == 0) and np.all(g["dv"][rest] == 0)
