"""Comparison helpers shared by the GPU parity tests (no attention arithmetic)."""
import numpy as np
import torch

# Tolerances for the forward pass: O max |err| <= 1e-2, mean |err| <= 1e-3; LSE |err| <= 1e-3.
O_MAX, O_MEAN, LSE_MAX = 1e-2, 1e-3, 1e-3
# Backward: relative Frobenius error of dQ, dK, dV <= 1e-2.
GRAD_REL = 1e-2


def to64(t):
    return t.detach().to("cpu").double().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def bf16_round(x):
    """fp64 -> nearest bf16 -> fp64 (the best answer representable in the output format)."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def bf16_ulp(x):
    """Spacing of bf16 values at |x| (8 significant bits)."""
    m, e = np.frexp(np.abs(x))
    return np.ldexp(1.0, e - 8)


def check_fwd(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """O is bf16, so it is compared with the oracle's fp64 O correctly rounded
    to bf16: per element |O - bf16(O_ref)| <= max(O_MAX, one bf16 ulp of the
    reference) (the stated tolerance, widened only where one rounding step of
    the output format exceeds it, i.e. |O| >= 2), and the mean of that error
    <= O_MEAN. LSE (fp32) is compared with the fp64 oracle directly."""
    o, l = to64(o_gpu), to64(lse_gpu)
    assert o.shape == o_ref.shape and l.shape == lse_ref.shape, (o.shape, o_ref.shape, l.shape, lse_ref.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    ref_b = bf16_round(o_ref)
    err = np.abs(o - ref_b)
    allowed = np.maximum(O_MAX, bf16_ulp(ref_b))
    dead = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(l), dead), f"{what}: -inf LSE rows differ"
    lerr = np.abs(l[~dead] - lse_ref[~dead]) if (~dead).any() else np.zeros(1)
    stats = {"o_max": float(err.max(initial=0)), "o_mean": float(err.mean()) if err.size else 0.0,
             "o_excess": float((err - allowed).max(initial=-1.0)), "lse_max": float(lerr.max(initial=0)),
             "o_max_vs_fp64": float(np.abs(o - o_ref).max(initial=0))}
    assert np.all(err <= allowed) and stats["o_mean"] <= O_MEAN and stats["lse_max"] <= LSE_MAX, (what, stats)
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
