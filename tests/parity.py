"""Comparison helpers shared by the GPU parity tests (no attention arithmetic)."""
import numpy as np
import torch

# Tolerances for the forward pass: O max |err| <= 1e-2, mean |err| <= 1e-3; LSE |err| <= 1e-3.
O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3
# Backward: relative Frobenius error of dQ, dK, dV <= 1e-2.
GRAD_REL = 1e-2


def to64(t):
    return t.detach().to("cpu").double().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def bf16_half_ulp(x):
    """Half the spacing of bf16 values at |x| (8 significant bits): the largest
    error a correctly rounded bf16 output can carry."""
    m, e = np.frexp(np.abs(x))
    return np.ldexp(1.0, e - 9)


def check_fwd(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """Compares the GPU forward with the fp64 oracle, element by element.

    O (bf16): |O - O_ref| <= max(O_MAX, half a bf16 ulp of O_ref) per element,
    against the unrounded fp64 reference. The half-ulp term is the only
    widening: a bf16 output cannot come closer than that to the exact value,
    and it exceeds O_MAX only where |O_ref| >= 4. The mean of |O - O_ref|
    must stay <= O_MEAN. LSE (fp32): |LSE - LSE_ref| <= LSE_MAX; rows with no
    visible key must be -inf on both sides."""
    o, l = to64(o_gpu), to64(lse_gpu)
    assert o.shape == o_ref.shape and l.shape == lse_ref.shape, (o.shape, o_ref.shape, l.shape, lse_ref.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    err = np.abs(o - o_ref)
    allowed = np.maximum(O_MAX, bf16_half_ulp(o_ref))
    dead = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(l), dead), f"{what}: -inf LSE rows differ"
    lerr = np.abs(l[~dead] - lse_ref[~dead]) if (~dead).any() else np.zeros(1)
    stats = {"o_max": float(err.max(initial=0)), "o_mean": float(err.mean()) if err.size else 0.0,
             "o_excess": float((err - allowed).max(initial=-1.0)), "lse_max": float(lerr.max(initial=0))}
    assert np.all(err <= allowed), (what, "O element beyond max(1e-2, half ulp) of the fp64 oracle", stats)
    assert stats["o_mean"] <= O_MEAN, (what, "mean |O - O_ref| above 1e-3", stats)
    assert stats["lse_max"] <= LSE_MAX, (what, "LSE error above 1e-3", stats)
    return stats


def rel_fro(a, b):
    a, b = to64(a), to64(b)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a))


def check_grads(got, ref, what=""):
    out = {}
    for n in ("dq", "dk", "dv"):
        g = to64(got[n])
        assert np.all(np.isfinite(g)), f"{what}: non-finite {n}"
        out[n] = rel_fro(g, ref[n])
        assert out[n] <= GRAD_REL, (what, n, out)
    return out
