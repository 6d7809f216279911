"""Pins for the oracle's score modifications (logit soft-capping, ALiBi distance
bias), forward and backward: limits that reduce to plain attention, an exact
identity that turns causal ALiBi into plain attention on augmented inputs, a
closed form at large slopes, bounds and orderings read off P, and central
finite differences of the forward definition. CPU only."""
import numpy as np
import pytest

from oracle import attention_bwd, attention_bwd_varlen, attention_fwd, attention_fwd_varlen, head_score_mod

RNG = np.random.default_rng(21)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


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


def close(a, b, tol):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300) < tol


@pytest.mark.parametrize("causal", [False, True])
def test_softcap_large_cap_is_plain_attention(causal):
    q, k, v, do = rand(7, 5), rand(9, 5), rand(9, 4), rand(7, 4)
    o, l = attention_fwd(q, k, v, 0.4, causal)
    oc, lc = attention_fwd(q, k, v, 0.4, causal, score_mod=("softcap", 1e7))
    assert np.allclose(oc, o, atol=1e-11) and np.allclose(lc, l, atol=1e-11)
    g = attention_bwd(q, k, v, do, 0.4, causal)
    gc = attention_bwd(q, k, v, do, 0.4, causal, score_mod=("softcap", 1e7))
    for n in ("dq", "dk", "dv"):
        assert np.allclose(gc[n], g[n], atol=1e-10), n


def test_softcap_bounds_and_order_of_p():
    """With V = I the output rows are the rows of P. Capped logits lie in
    (-c, c), so any two weights of a row differ by less than a factor e^(2c);
    tanh is increasing, so P keeps the order of the raw logits."""
    nq, nk, c = 6, 11, 0.7
    q, k = rand(nq, 4), rand(nk, 4)  # |logit| / c stays below ~15: tanh not yet rounded to +-1
    p, _ = attention_fwd(q, k, np.eye(nk), 1.0, False, score_mod=("softcap", c))
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-14)
    assert np.all(p.max(axis=1) / p.min(axis=1) < np.exp(2 * c))
    raw = q @ k.T
    for i in range(nq):
        assert np.array_equal(np.argsort(p[i], kind="stable"), np.argsort(raw[i], kind="stable"))


@pytest.mark.parametrize("causal", [False, True])
def test_alibi_zero_slope_is_plain_attention(causal):
    q, k, v, do = rand(5, 3), rand(8, 3), rand(8, 6), rand(5, 6)
    o, l = attention_fwd(q, k, v, 0.5, causal)
    oa, la = attention_fwd(q, k, v, 0.5, causal, score_mod=("alibi", 0.0))
    assert np.array_equal(oa, o) and np.array_equal(la, l)
    g, ga = attention_bwd(q, k, v, do, 0.5, causal), attention_bwd(q, k, v, do, 0.5, causal,
                                                                   score_mod=("alibi", 0.0))
    for n in ("dq", "dk", "dv"):
        assert np.array_equal(ga[n], g[n]), n


@pytest.mark.parametrize("nq,nk", [(6, 6), (4, 9)])
def test_causal_alibi_is_plain_attention_on_augmented_inputs(nq, nk):
    """Under the causal mask every visible key j has j <= i + nk - nq, so the
    penalty -m * |j - (i + nk - nq)| equals m * j minus a per-row constant,
    which the softmax cancels, but not the log-sum-exp (it moves by -m(i + nk - nq)). The
    m * j term is the logit of one extra dimension: q' = [q, 1],
    k' = [k, m j / scale]."""
    scale, m = 0.35, 0.8
    q, k, v, do = rand(nq, 4), rand(nk, 4), rand(nk, 3), rand(nq, 3)
    qa = np.concatenate([q, np.ones((nq, 1))], axis=1)
    ka = np.concatenate([k, (m / scale) * np.arange(nk)[:, None]], axis=1)
    o, lse = attention_fwd(q, k, v, scale, True, score_mod=("alibi", m))
    o2, lse2 = attention_fwd(qa, ka, v, scale, True)
    live = np.isfinite(lse2)
    assert np.allclose(o, o2, atol=1e-13)
    shift = m * (np.arange(nq) + nk - nq)
    assert np.allclose(lse[live], lse2[live] - shift[live], atol=1e-12)
    g = attention_bwd(q, k, v, do, scale, True, score_mod=("alibi", m))
    g2 = attention_bwd(qa, ka, v, do, scale, True)
    assert np.allclose(g["dq"], g2["dq"][:, :4], atol=1e-12)
    assert np.allclose(g["dk"], g2["dk"][:, :4], atol=1e-12)
    assert np.allclose(g["dv"], g2["dv"], atol=1e-12)


def test_alibi_large_slope_attends_to_the_aligned_key():
    """A slope far above the logits leaves only the key at distance 0:
    O_i = v_(i + nk - nq), LSE_i = the logit of that key."""
    nq, nk, scale = 5, 8, 0.3
    q, k, v = rand(nq, 4), rand(nk, 4), rand(nk, 2)
    o, lse = attention_fwd(q, k, v, scale, False, score_mod=("alibi", 200.0))
    j = np.arange(nq) + nk - nq
    assert np.allclose(o, v[j], atol=1e-12)
    assert np.allclose(lse, scale * np.einsum("id,id->i", q, k[j]), atol=1e-12)


@pytest.mark.parametrize("mod", [("softcap", 1.3), ("softcap", 0.4), ("alibi", 0.6)])
@pytest.mark.parametrize("causal", [False, True])
def test_score_mod_gradients_match_finite_differences(mod, causal):
    nq, nk, dqk, dv = 5, 7, 4, 3
    q, k, v, do = rand(nq, dqk), rand(nk, dqk), rand(nk, dv), rand(nq, dv)
    s = 0.6

    def loss(qq, kk, vv):
        o, _ = attention_fwd(qq, kk, vv, s, causal, score_mod=mod)
        return float((o * do).sum())

    g = attention_bwd(q, k, v, do, s, causal, score_mod=mod)
    for name, got, x, f in (("dq", g["dq"], q, lambda x: loss(x, k, v)), ("dk", g["dk"], k, lambda x: loss(q, x, v)),
                            ("dv", g["dv"], v, lambda x: loss(q, k, x))):
        assert close(got, fd_grad(f, x), 1e-6), name


def test_varlen_applies_per_head_slopes_within_each_sequence():
    """Positions restart at every sequence, and head h takes slope m[h]."""
    H, slopes = 3, np.array([0.25, 0.5, 1.0])
    cu = np.array([0, 4, 4, 11])
    q, k, v, do = rand(11, H, 4), rand(11, H, 4), rand(11, H, 2), rand(11, H, 2)
    o, lse = attention_fwd_varlen(q, k, v, cu, cu, 0.5, True, score_mod=("alibi", slopes))
    dq, dk, dv = attention_bwd_varlen(q, k, v, do, cu, cu, 0.5, True, score_mod=("alibi", slopes))
    for h in range(H):
        assert head_score_mod(("alibi", slopes), h) == ("alibi", float(slopes[h]))
        for a, b in ((0, 4), (4, 11)):
            oo, ll = attention_fwd(q[a:b, h], k[a:b, h], v[a:b, h], 0.5, True, score_mod=("alibi", slopes[h]))
            assert np.array_equal(o[a:b, h], oo) and np.array_equal(lse[h, a:b], ll)
            g = attention_bwd(q[a:b, h], k[a:b, h], v[a:b, h], do[a:b, h], 0.5, True,
                              score_mod=("alibi", slopes[h]))
            assert np.array_equal(dq[a:b, h], g["dq"]) and np.array_equal(dk[a:b, h], g["dk"])
    assert head_score_mod(("softcap", 2.0), 1) == ("softcap", 2.0)
