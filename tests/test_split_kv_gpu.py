"""Dense forwards whose (query block, head, batch) grid would leave most SMs
idle and whose keys are long run with the keys split across CTAs: each CTA
computes O and the LSE over one range of key blocks, and a second kernel merges
the ranges (LSE = ln sum_r exp(LSE_r), O = sum_r exp(LSE_r - LSE) O_r).

The outputs are compared with the oracle on every element, for d = 64 and 128,
with and without the causal mask (bottom-right, so with Nq < Nk every row sees
most keys, and with Nq = Nk the early rows see no key of the later ranges), on
ragged lengths; the backward runs on the split forward's O and LSE; and two
calls must give the same bits."""
import numpy as np
import pytest
import torch

import workloads
from oracle import attention_bwd, attention_fwd
from parity import check_fwd, check_grads

pytestmark = pytest.mark.gpu


def _forward_vs_oracle(ea, w, what):
    t = workloads.make_dense(w, device="cuda")
    o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=w.causal, softmax_scale=w.scale)
    o2, lse2 = ea.attn_fwd(t["q"], t["k"], t["v"], causal=w.causal, softmax_scale=w.scale)
    torch.cuda.synchronize()
    ea.attn_get_device_status()
    assert torch.equal(o, o2) and torch.equal(lse, lse2), f"{what}: two calls differ"
    q, k, v = (t[n].cpu() for n in ("q", "k", "v"))
    for b in range(w.batch):
        for h in range(w.heads):
            o_ref, l_ref = attention_fwd(q[b, :, h], k[b, :, h], v[b, :, h], w.scale, w.causal)
            check_fwd(o[b, :, h], lse[b, h], o_ref, l_ref, f"{what} b{b} h{h}")
    return t, o, lse


@pytest.mark.parametrize("dims", [(64, 64), (128, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_short_queries_long_keys(dims, causal):
    import exact_attention_bf16_gb300 as ea
    dqk, dv_ = dims
    # one 256-row block per (batch, head): 4 CTAs before the split; 4,000 keys = 32 key blocks
    w = workloads.Workload("split", 2, 2, 200, 4000, dqk, dv_, causal, seed=61)
    _forward_vs_oracle(ea, w, f"split d{dqk} causal={causal}")


def test_ranges_without_visible_keys():
    """Causal, Nq = Nk: the first rows see only the first key range; the other
    ranges give them LSE = -inf and no weight in the merge."""
    import exact_attention_bf16_gb300 as ea
    w = workloads.Workload("split_sq", 1, 1, 3000, 3000, 128, 128, True, seed=62)
    _forward_vs_oracle(ea, w, "split causal square")


def test_backward_on_a_split_forward():
    import exact_attention_bf16_gb300 as ea
    w = workloads.Workload("split_bwd", 1, 2, 300, 2500, 128, 128, True, seed=63)
    t, o, lse = _forward_vs_oracle(ea, w, "split for backward")
    dq, dk, dv = ea.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=True, softmax_scale=w.scale)
    torch.cuda.synchronize()
    ea.attn_get_device_status()
    q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
    for h in range(w.heads):
        ref = attention_bwd(q[0, :, h], k[0, :, h], v[0, :, h], do[0, :, h], w.scale, True)
        check_grads({"dq": dq[0, :, h], "dk": dk[0, :, h], "dv": dv[0, :, h]}, ref, f"split backward h{h}")
