"""The two-SM forward (attn_fwd_params.cta_pair, d = 128): every (batch, head)
of small shapes with ragged tails against the fp64 oracle, both masks, dense
and varlen, V beyond fp16's range (bf16 fallback), a sampled check at the
benchmark's shape, and bitwise reproducibility."""
import numpy as np
import pytest
import torch

import workloads
from oracle import attention_fwd
from parity import check_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ea():
    import exact_attention_bf16_gb300 as ea
    return ea


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk", [(300, 300), (200, 520), (777, 1000), (1100, 700), (513, 513)])
def test_dense_pair_forward(ea, causal, nq, nk):
    w = workloads.Workload("pf", 2, 2, nq, nk, 128, 128, causal, seed=nq + 2 * nk + causal)
    t = workloads.make_dense(w, device="cuda", with_do=False)
    o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=causal, softmax_scale=w.scale, cta_pair=True)
    o2, lse2 = ea.attn_fwd(t["q"], t["k"], t["v"], causal=causal, softmax_scale=w.scale, cta_pair=True)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == 0
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    q, k, v = (t[n].cpu() for n in ("q", "k", "v"))
    for b in range(w.batch):
        for h in range(w.heads):
            oo, ll = attention_fwd(q[b, :, h], k[b, :, h], v[b, :, h], w.scale, causal)
            check_fwd(o[b, :, h], lse[b, h], oo, ll, f"b{b} h{h}")


def test_varlen_pair_forward(ea):
    ql = [5, 300, 0, 257, 1000, 1, 600]
    kl = [7, 260, 3, 257, 900, 1, 0]
    H = 2
    t = workloads.make_varlen_qk(ql, kl, H, 128, 128, seed=31, device="cuda")
    o, lse = ea.attn_fwd_varlen(t["q"], t["k"], t["v"], t["cu_q"], t["cu_k"], max(ql), max(kl), causal=True,
                                cta_pair=True)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == 0
    q, k, v = (x.cpu() for x in (t["q"], t["k"], t["v"]))
    o_ref = np.zeros((sum(ql), H, 128))
    lse_ref = np.full((H, sum(ql)), -np.inf)
    cq, ck = t["cu_q"].cpu().numpy(), t["cu_k"].cpu().numpy()
    for s in range(len(ql)):
        a, b, c, d = int(cq[s]), int(cq[s + 1]), int(ck[s]), int(ck[s + 1])
        for h in range(H):
            if b > a and d > c:
                o_ref[a:b, h], lse_ref[h, a:b] = attention_fwd(q[a:b, h], k[c:d, h], v[c:d, h], 128 ** -0.5, True)
    check_fwd(o, lse, o_ref, lse_ref, "varlen pair")


def test_pair_forward_with_v_beyond_fp16(ea):
    w = workloads.Workload("pfv", 1, 2, 400, 400, 128, 128, False, seed=4)
    t = workloads.make_dense(w, device="cuda", with_do=False)
    v = t["v"].clone()
    v[0, 7, 1, :] = 1.0e5  # outside fp16's range: P and V stay bf16 for the whole call
    o, lse = ea.attn_fwd(t["q"], t["k"], v, cta_pair=True)
    o1, lse1 = ea.attn_fwd(t["q"], t["k"], v)
    torch.cuda.synchronize()
    assert torch.all(torch.isfinite(o.float()))
    rel = float((o.double() - o1.double()).norm() / o1.double().norm())
    assert rel < 1e-2, rel


@pytest.mark.parametrize("causal", [False, True])
def test_pair_forward_at_the_benchmark_shape_sampled(ea, causal):
    w = workloads.dense_d128(8192, causal)
    t = workloads.make_dense(w, device="cuda", with_do=False)
    o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=causal, softmax_scale=w.scale, cta_pair=True)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == 0
    for b, h in workloads.sample_pairs(w.batch, w.heads, 2, seed=8 + causal):
        q, k, v = (t[n][b, :, h].cpu() for n in ("q", "k", "v"))
        oo, ll = attention_fwd(q, k, v, w.scale, causal, row_block=2048)
        check_fwd(o[b, :, h], lse[b, h], oo, ll, f"b{b} h{h}")


def test_pair_forward_rejections(ea):
    x = torch.zeros((1, 128, 2, 64), device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ea.AttnError):  # d = 128 only
        ea.attn_fwd(x, x, x, cta_pair=True)
    y = torch.zeros((1, 128, 2, 128), device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ea.AttnError):
        ea.attn_fwd(y, y, y, cta_pair=True, exp2_emu_period=8)
    with pytest.raises(ea.AttnError):
        ea.attn_fwd(y, y, y, cta_pair=True, softcap=2.0)
