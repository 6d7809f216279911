"""Seeded synthetic attention workloads shared by the tests, the benchmark and
the smoke check.

This module only draws inputs and names shapes. It holds none of the
attention arithmetic: no softmax, no matmul, no reference values. Both the
CUDA path and the CPU oracle consume what it produces.

Recipe: Q, K, V (and dO) are i.i.d. N(0, 1) drawn in fp32 from one
``torch.Generator`` seeded per workload, in the order Q, K, V, dO, each tensor
[B, N, H, d] (or packed [total, H, d] for variable length), then rounded to
bf16 (round-to-nearest-even). The outlier variant scales a seeded 1% of key
rows of every (batch, head) by 8 in fp32 before that rounding, so that row
maxima jump late in the key sequence and force rescales.

Shapes follow the ones the FlashAttention-4 pages discuss: head dims 64 and
128, the (192, 128) MLA shape (wittx "FlashAttention-4", section on the
DeepSeek performance figure), sequence lengths up to 32K (same page, section on
Mamba), causal and non-causal, and a variable-length packed batch (newton wiki
"FlashAttention-4", 核心技術: tile scheduler for causal and variable-length
balance).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

# 32 lengths drawn once with torch.randint(256, 32769, (32,),
# generator=torch.Generator().manual_seed(7)) on torch 2.11 (CPU) and frozen
# here so that every machine and torch version sees the same batch.
VARLEN_LENGTHS: List[int] = [
    10831, 16245, 9126, 7774, 28170, 8204, 24646, 25169, 13748, 16073, 10159, 11246, 690, 26519, 31297, 2499,
    25942, 24915, 15797, 23953, 9414, 22112, 30402, 28368, 10778, 22333, 6469, 1856, 1354, 3865, 10166, 18843,
]


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    seqlen_q: int
    seqlen_k: int
    d_qk: int
    d_v: int
    causal: bool
    seed: int = 0
    softmax_scale: Optional[float] = None
    outlier_frac: float = 0.0
    varlen_lengths: Optional[tuple] = None

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale is not None else 1.0 / math.sqrt(self.d_qk)

    @property
    def is_varlen(self) -> bool:
        return self.varlen_lengths is not None

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


def single_head_d64() -> Workload:
    """B=1, H=1, N=128, d=64, non-causal, scale 1/8."""
    return Workload("single_head_d64", 1, 1, 128, 128, 64, 64, False, seed=0)


def dense_d128(seqlen: int, causal: bool, outlier: bool = False) -> Workload:
    """H=16, d=128, B = 32768 / N (so every point holds the same number of tokens)."""
    assert 32768 % seqlen == 0
    return Workload(f"dense_d128_N{seqlen}{'_causal' if causal else ''}{'_outlier' if outlier else ''}",
                    32768 // seqlen, 16, seqlen, seqlen, 128, 128, causal, seed=0,
                    outlier_frac=0.01 if outlier else 0.0)


DENSE_SWEEP = (1024, 4096, 8192, 16384, 32768)


def mla_192_128() -> Workload:
    """B=2, H=32, N=8192, causal, d_qk=192, d_v=128, scale 1/sqrt(192)."""
    return Workload("mla_192_128_N8192_causal", 2, 32, 8192, 8192, 192, 128, True, seed=0)


def bwd_d128_N16384() -> Workload:
    """B=2, H=16, N=16384, causal, d=128 (training shape for the backward pass)."""
    return Workload("bwd_d128_N16384_causal", 2, 16, 16384, 16384, 128, 128, True, seed=0)


def varlen_32seq() -> Workload:
    """32 packed sequences (lengths frozen above, 498,963 tokens), H=32, d=128, causal."""
    return Workload("varlen_32seq_H32_d128_causal", 1, 32, max(VARLEN_LENGTHS), max(VARLEN_LENGTHS), 128, 128,
                    True, seed=0, varlen_lengths=tuple(VARLEN_LENGTHS))


def make_dense(w: Workload, device="cpu", with_do: bool = True, outlier_seed: int = 1):
    """Returns dict(q, k, v[, do]) of bf16 tensors shaped [B, N, H, d]."""
    g = torch.Generator(device=device).manual_seed(w.seed)
    B, H = w.batch, w.heads
    f32 = dict(generator=g, device=device, dtype=torch.float32)
    q = torch.randn((B, w.seqlen_q, H, w.d_qk), **f32)
    k = torch.randn((B, w.seqlen_k, H, w.d_qk), **f32)
    v = torch.randn((B, w.seqlen_k, H, w.d_v), **f32)
    do = torch.randn((B, w.seqlen_q, H, w.d_v), **f32) if with_do else None
    if w.outlier_frac > 0:
        n_out = math.ceil(w.outlier_frac * w.seqlen_k)
        go = torch.Generator(device="cpu").manual_seed(outlier_seed)
        for b in range(B):
            for h in range(H):
                rows = torch.randperm(w.seqlen_k, generator=go)[:n_out].to(device)
                k[b, rows, h, :] *= 8.0
    out = {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16)}
    if with_do:
        out["do"] = do.to(torch.bfloat16)
    return out


def cu_seqlens_of(lengths) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def make_varlen(w: Workload, device="cpu", with_do: bool = True):
    """Returns dict(q, k, v[, do], cu_seqlens) with packed [total, H, d] bf16 tensors
    (queries and keys share the same lengths)."""
    assert w.is_varlen
    total = sum(w.varlen_lengths)
    g = torch.Generator(device=device).manual_seed(w.seed)
    H = w.heads
    f32 = dict(generator=g, device=device, dtype=torch.float32)
    q = torch.randn((total, H, w.d_qk), **f32).to(torch.bfloat16)
    k = torch.randn((total, H, w.d_qk), **f32).to(torch.bfloat16)
    v = torch.randn((total, H, w.d_v), **f32).to(torch.bfloat16)
    out = {"q": q, "k": k, "v": v, "cu_seqlens": cu_seqlens_of(w.varlen_lengths).to(device)}
    if with_do:
        out["do"] = torch.randn((total, H, w.d_v), **f32).to(torch.bfloat16)
    return out


def make_varlen_qk(q_lengths, k_lengths, heads: int, d_qk: int, d_v: int, seed: int, device="cpu"):
    """Packed varlen inputs whose query and key lengths differ per sequence:
    dict(q [total_q, H, d_qk], k, v [total_k, H, d], do [total_q, H, d_v],
    cu_q, cu_k), i.i.d. N(0,1) rounded to bf16 from one seeded generator."""
    assert len(q_lengths) == len(k_lengths)
    tq, tk = sum(q_lengths), sum(k_lengths)
    g = torch.Generator(device=device).manual_seed(seed)
    f32 = dict(generator=g, device=device, dtype=torch.float32)
    q = torch.randn((tq, heads, d_qk), **f32).to(torch.bfloat16)
    k = torch.randn((tk, heads, d_qk), **f32).to(torch.bfloat16)
    v = torch.randn((tk, heads, d_v), **f32).to(torch.bfloat16)
    do = torch.randn((tq, heads, d_v), **f32).to(torch.bfloat16)
    return {"q": q, "k": k, "v": v, "do": do, "cu_q": cu_seqlens_of(q_lengths).to(device),
            "cu_k": cu_seqlens_of(k_lengths).to(device)}


def sample_pairs(batch: int, heads: int, n: int, seed: int = 1234):
    """A seeded subset of (batch, head) units for spot-checking large workloads."""
    g = torch.Generator().manual_seed(seed)
    idx = torch.randperm(batch * heads, generator=g)[: min(n, batch * heads)].tolist()
    return [(i // heads, i % heads) for i in idx]


# ---------------------------------------------------------------------------
# Work counting (a measurement convention, not part of the computation)
# ---------------------------------------------------------------------------
def causal_pairs(nq: int, nk: int) -> float:
    """Visible (query, key) pairs under the bottom-right causal mask: row i sees
    clip(i + nk - nq + 1, 0, nk) keys. When nq == nk the usual half-square
    convention nq * nk / 2 is used instead of the exact nq (nq + 1) / 2."""
    if nq == nk:
        return nq * nk / 2.0
    lo, hi = nk - nq + 1, nk  # the first and last row's unclipped counts

    def tri(x):  # 1 + 2 + ... + x
        return x * (x + 1) // 2 if x > 0 else 0

    a, b = max(lo, 1), min(hi, nk)
    ramp = tri(b) - tri(a - 1) if a <= b else 0  # rows with 1 .. nk visible keys
    full = max(0, hi - max(lo, nk + 1) + 1) * nk  # rows past the last key see all nk
    return float(ramp + full)


def attn_flops(nq: int, nk: int, d_qk: int, d_v: int, causal: bool, direction: str = "fwd") -> float:
    """Algorithmic FLOPs of one (batch, head): forward = 2 Nq Nk (d_qk + d_v)
    (QK^T and PV); backward = 2 Nq Nk (3 d_qk + 2 d_v) (QK^T, dO V^T, P^T dO,
    dS^T Q, dS K). Causal counts half of the square."""
    pairs = causal_pairs(nq, nk) if causal else float(nq) * nk
    per = (d_qk + d_v) if direction == "fwd" else (3 * d_qk + 2 * d_v)
    return 2.0 * pairs * per


def workload_flops(w: Workload, direction: str = "fwd") -> float:
    if w.is_varlen:
        return w.heads * sum(attn_flops(n, n, w.d_qk, w.d_v, w.causal, direction) for n in w.varlen_lengths)
    return w.batch * w.heads * attn_flops(w.seqlen_q, w.seqlen_k, w.d_qk, w.d_v, w.causal, direction)
