"""Causal launches that dispatch their blocks in groups of heads (heaviest
blocks of a group first): every block of every (batch, head) is computed once.

Outputs are pre-filled with NaN, so a block that no CTA wrote stays NaN; the
forward is compared with the oracle on two rows of every 128-row tile of
(batch, head) pairs drawn from every dispatch group (each row against the
oracle on that row alone, which under the causal mask sees keys 0 .. row);
the backward on whole (batch, head) pairs from both of its groups."""
import numpy as np
import pytest
import torch

import workloads
from oracle import attention_bwd, attention_fwd
from parity import check_fwd, check_grads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ea():
    import exact_attention_bf16_gb300 as ea
    return ea


def test_grouped_causal_forward_writes_every_block(ea):
    # B8 H16 N4096 d128: 128 (batch, head) pairs of 2 MB of K and V each, 16 blocks of
    # 256 rows per pair: the launch walks 8 groups of 16 pairs, heaviest blocks first.
    w = workloads.Workload("grouped_fwd", 8, 16, 4096, 4096, 128, 128, True, seed=41)
    t = workloads.make_dense(w, device="cuda", with_do=False)
    o = torch.full_like(t["q"], float("nan"))
    lse = torch.full((w.batch, w.heads, w.seqlen_q), float("nan"), device="cuda")
    ea.attn_fwd(t["q"], t["k"], t["v"], causal=True, softmax_scale=w.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    ea.attn_get_device_status()
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all()), "a block was not written"
    q, k, v = (t[n].cpu() for n in ("q", "k", "v"))
    o_h, l_h = o.cpu(), lse.cpu()
    pairs = [(bh // w.heads, bh % w.heads) for bh in (0, 15, 16, 47, 64, 95, 112, 127)]
    rows = [r for m in range(w.seqlen_q // 128) for r in (128 * m, 128 * m + 127)]
    for b, h in pairs:
        o_ref = np.empty((len(rows), w.d_v))
        l_ref = np.empty(len(rows))
        for n, r in enumerate(rows):
            oo, ll = attention_fwd(q[b, r:r + 1, h], k[b, :r + 1, h], v[b, :r + 1, h], w.scale, False)
            o_ref[n], l_ref[n] = oo[0], ll[0]
        check_fwd(o_h[b, rows, h], l_h[b, h, rows], o_ref, l_ref, f"grouped forward b{b} h{h}")


def test_grouped_causal_backward_writes_every_block(ea):
    # B4 H16 N2048 d128: 64 pairs of 1 MB each, 16 key blocks (dK/dV) and query
    # blocks (dQ) of 128 rows per pair: two dispatch groups of 32 pairs.
    w = workloads.Workload("grouped_bwd", 4, 16, 2048, 2048, 128, 128, True, seed=43)
    t = workloads.make_dense(w, device="cuda")
    o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=True, softmax_scale=w.scale)
    dq, dk, dv = (torch.full_like(t[n], float("nan")) for n in ("q", "k", "v"))
    ea.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=True, softmax_scale=w.scale, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    ea.attn_get_device_status()
    for n, g in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert bool(torch.isfinite(g).all()), f"{n}: a block was not written"
    q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
    for bh in (0, 31, 32, 63):
        b, h = bh // w.heads, bh % w.heads
        ref = attention_bwd(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], w.scale, True, row_block=1024)
        check_grads({"dq": dq[b, :, h], "dk": dk[b, :, h], "dv": dv[b, :, h]}, ref, f"grouped backward b{b} h{h}")
