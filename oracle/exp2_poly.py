"""exp2 emulated with a Cody-Waite range split and a degree-3 polynomial.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The method (wittx "FlashAttention-4", section 用软件"伪造"硬件指令; jsqmd
"GPU 算力翻倍…FlashAttention-4", section 四.1) computes 2^x without the
special-function unit:
  1. split x = n + f with n = floor(x) an integer and f in [0, 1);
  2. 2^n is formed by writing n into the IEEE-754 exponent field;
  3. 2^f is approximated by a cubic, evaluated with Horner's rule on FMAs;
  4. 2^x = 2^n * p(f).
The pages print the cubic's form (a + b f + c f^2 + d f^3) but not its
coefficients. Reading taken here: the coefficients minimise the maximum
*relative* error of p(f) against 2^f on [0, 1], subject to p(0) = 1 (so 2^x is
exact at every integer x, in particular p = 1 for the row maximum). They are
found by the Remez exchange algorithm in fp64. This fit's error (8.6e-5) is
about 600x the ~1.4e-7 of the hardware ex2 and leaves bf16(p) == bf16(2^x)
on 99% of inputs, the two figures wittx gives in the same section.

Inputs below -127 are clamped to -127 (results there are below 2^-126 and
contribute nothing next to the row maximum's p = 1 in a softmax row).
"""

from __future__ import annotations

import numpy as np


def exp2_exact(x):
    """2^x in fp64 (library routine)."""
    return np.exp2(np.asarray(x, dtype=np.float64))


def _rel_err(c, x):
    p = ((c[3] * x + c[2]) * x + c[1]) * x + c[0]
    return p / np.exp2(x) - 1.0


def _extrema(c, grid):
    """Interior local extrema of the relative error (parabolic refinement) plus the endpoint f = 1."""
    e = _rel_err(c, grid)
    de = np.diff(e)
    idx = np.where(np.sign(de[:-1]) != np.sign(de[1:]))[0] + 1
    h = grid[1] - grid[0]
    pts = []
    for i in idx:
        y0, y1, y2 = e[i - 1], e[i], e[i + 1]
        den = y0 - 2 * y1 + y2
        xs = grid[i] + (0.5 * h * (y0 - y2) / den if den != 0 else 0.0)
        pts.append(min(max(xs, grid[i - 1]), grid[i + 1]))
    pts.append(1.0)
    return np.array(sorted(pts))


def fit_exp2_poly_remez(iters: int = 60, grid_points: int = 400001):
    """Minimax relative-error cubic for 2^f on [0, 1] with c0 = p(0) = 1.

    Three free coefficients (c1, c2, c3), so the optimum error equioscillates
    on four points of (0, 1]; the Remez exchange alternates between solving the
    levelled equations  p(x_i) - 2^x_i = (-1)^i E 2^x_i  on a reference set and
    moving the reference to the error's extrema. Returns a dict: ``c``
    (c0..c3), ``max_rel_err`` (max |p/2^f - 1| on a dense grid), ``level``
    (the levelled |E|) and ``ref`` (the final reference points).
    """
    ref = np.array([0.1, 0.4, 0.75, 1.0])
    grid = np.linspace(0.0, 1.0, grid_points)
    sgn = np.array([1.0, -1.0, 1.0, -1.0])
    c, E = None, None
    for _ in range(iters):
        A = np.stack([ref, ref ** 2, ref ** 3, -sgn * np.exp2(ref)], axis=1)
        rhs = np.exp2(ref) - 1.0
        c1, c2, c3, E = np.linalg.solve(A, rhs)
        c = np.array([1.0, c1, c2, c3])
        ext = _extrema(c, grid)
        if len(ext) != 4:
            break
        done = np.max(np.abs(ext - ref)) < 1e-13
        ref = ext
        if done:
            break
    err = np.abs(_rel_err(c, grid)).max()
    return {"c": c, "max_rel_err": float(err), "level": float(abs(E)), "ref": ref}


def exp2_poly(x, c):
    """2^x by the split-and-cubic method with coefficients c = (c0, c1, c2, c3)."""
    x = np.maximum(np.asarray(x, dtype=np.float64), -127.0)
    n = np.floor(x)                                  # integer part
    f = x - n                                        # fraction in [0, 1)
    p = ((c[3] * f + c[2]) * f + c[1]) * f + c[0]    # Horner on the cubic
    return np.ldexp(p, n.astype(np.int64))           # exponent-field scaling by 2^n
