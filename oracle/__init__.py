"""CPU oracle for exact scaled-dot-product attention (forward and backward).

TEST INFRASTRUCTURE ONLY. This package is the slow, obviously-correct fp64
reference that the CUDA path is checked against. Only the test-suite, the
package smoke check and the benchmark's CPU-baseline / reference arm may import
it. The product path (the C-ABI library and its Python binding) never imports,
calls or links anything here, and this package imports nothing from the
product path.

Contents
--------
attention.py  the plain definition of attention (dense softmax-then-matmul),
              forward and backward, dense and variable-length; and the
              conditional-rescale online-softmax algorithm restated in fp64;
              the key visibility of a block-sparse mask, element by element;
              the score modifications (logit soft-capping, ALiBi distance bias).
exp2_poly.py  the Cody-Waite split + degree-3 polynomial exp2 emulation, with
              its own minimax (Remez exchange) coefficient fit.
fp8.py        FP8 E4M3 codes to values, from the format's definition.

Every function is pinned by tests in ``tests/test_oracle_*.py`` against closed
forms, invariants, finite differences and hand-worked examples.
"""

from .attention import (  # noqa: F401
    attention_fwd,
    attention_bwd,
    attention_fwd_online,
    attention_fwd_varlen,
    attention_bwd_varlen,
    block_sparse_visible,
    head_score_mod,
    score_mod_apply,
    visible_limit,
)
from .exp2_poly import fit_exp2_poly_remez, exp2_poly, exp2_exact  # noqa: F401
from .fp8 import e4m3_decode  # noqa: F401
