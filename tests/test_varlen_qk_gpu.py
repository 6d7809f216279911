"""Variable-length batches whose query and key lengths differ per sequence
(the ABI takes separate cu_seqlens for queries and keys), with the causal mask
aligned bottom-right (key j visible to query i iff j <= i + Nk - Nq), and
without it. The cases include sequences with no keys (O = 0, LSE = -inf, zero
gradients) and with no queries (zero dK, dV). The forward and the backward are
compared with the oracle per (sequence, head), and two backward runs must be
bitwise equal."""
import numpy as np
import pytest
import torch

import workloads
from oracle import attention_bwd, attention_fwd
from parity import check_fwd, check_grads

pytestmark = pytest.mark.gpu

QL = [5, 130, 0, 257, 64, 300, 1]
KL = [7, 100, 3, 300, 0, 129, 1]


@pytest.mark.parametrize("dims", [(64, 64), (128, 128), (192, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_distinct_q_and_k_lengths(dims, causal):
    import exact_attention_bf16_gb300 as ea
    dqk, dv_ = dims
    H = 2
    t = workloads.make_varlen_qk(QL, KL, H, dqk, dv_, seed=17, device="cuda")
    scale = 1.0 / np.sqrt(dqk)
    Lq, Lk = max(QL), max(KL)
    o, lse = ea.attn_fwd_varlen(t["q"], t["k"], t["v"], t["cu_q"], t["cu_k"], Lq, Lk, causal=causal,
                                softmax_scale=scale)
    g1 = ea.attn_bwd_varlen(t["q"], t["k"], t["v"], o, lse, t["do"], t["cu_q"], t["cu_k"], Lq, Lk, causal=causal,
                            softmax_scale=scale)
    g2 = ea.attn_bwd_varlen(t["q"], t["k"], t["v"], o, lse, t["do"], t["cu_q"], t["cu_k"], Lq, Lk, causal=causal,
                            softmax_scale=scale, deterministic=True)
    torch.cuda.synchronize()
    ea.attn_get_device_status()
    for a, b in zip(g1, g2):
        assert torch.equal(a, b), "backward is not bitwise reproducible"
    dq, dk, dv = g1
    q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
    cq, ck = t["cu_q"].cpu().numpy(), t["cu_k"].cpu().numpy()
    for s in range(len(QL)):
        a, b = int(cq[s]), int(cq[s + 1])
        c, d = int(ck[s]), int(ck[s + 1])
        for h in range(H):
            if b > a and d > c:
                oo, ll = attention_fwd(q[a:b, h], k[c:d, h], v[c:d, h], scale, causal)
                check_fwd(o[a:b, h], lse[h, a:b], oo, ll, f"seq{s} h{h}")
                ref = attention_bwd(q[a:b, h], k[c:d, h], v[c:d, h], do[a:b, h], scale, causal)
                check_grads({"dq": dq[a:b, h], "dk": dk[c:d, h], "dv": dv[c:d, h]}, ref, f"seq{s} h{h}")
            elif b > a:  # queries without keys
                assert torch.all(o[a:b, h] == 0) and torch.all(torch.isneginf(lse[h, a:b]))
                assert torch.all(dq[a:b, h] == 0)
            elif d > c:  # keys without queries
                assert torch.all(dk[c:d, h] == 0) and torch.all(dv[c:d, h] == 0)
