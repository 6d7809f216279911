"""Single-pass backward (d = 64): dK, dV and dQ partials from one key-stationary
kernel, the partials reduced across CTAs in an fp32 buffer, against the fp64
oracle on every (batch, head) / (sequence, head). The deterministic mode orders
the reduction by key tile through semaphores: repeated runs must be bitwise
identical. The non-deterministic mode's order is the hardware's: its results
must match the oracle, not each other bit for bit."""
import numpy as np
import pytest
import torch

import workloads
from oracle import attention_bwd
from parity import check_grads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ea():
    import exact_attention_bf16_gb300 as ea
    return ea


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("nq,nk", [(300, 300), (200, 520), (777, 333)])
def test_dense_single_pass(ea, causal, deterministic, nq, nk):
    w = workloads.Workload("sp", 2, 3, nq, nk, 64, 64, causal, seed=nq * 3 + nk + causal)
    t = workloads.make_dense(w, device="cuda")
    o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=causal, softmax_scale=w.scale)
    dq, dk, dv = ea.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=causal, softmax_scale=w.scale,
                             deterministic=deterministic, single_pass=True)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == 0
    q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    for b in range(w.batch):
        for h in range(w.heads):
            ref = attention_bwd(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], w.scale, causal)
            check_grads({"dq": dq[b, :, h], "dk": dk[b, :, h], "dv": dv[b, :, h]}, ref, f"b{b} h{h}")


@pytest.mark.parametrize("causal", [False, True])
def test_deterministic_mode_is_bitwise_reproducible(ea, causal):
    """Many key tiles add into every query tile (N = 4096: 32 key tiles), so an
    unordered reduction would differ between runs; the ordered one may not."""
    w = workloads.Workload("det", 2, 4, 4096, 4096, 64, 64, causal, seed=5)
    t = workloads.make_dense(w, device="cuda")
    o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=causal)
    args = (t["q"], t["k"], t["v"], o, lse, t["do"])
    first = ea.attn_bwd(*args, causal=causal, deterministic=True, single_pass=True)
    for _ in range(9):
        again = ea.attn_bwd(*args, causal=causal, deterministic=True, single_pass=True)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == 0
    # the dK / dV of a key tile do not depend on the reduction order; dQ does only in rounding
    loose = ea.attn_bwd(*args, causal=causal, deterministic=False, single_pass=True)
    two_kernel = ea.attn_bwd(*args, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(first[1], loose[1]) and torch.equal(first[2], loose[2])
    for a, b in zip(first, two_kernel):
        a64, b64 = a.double(), b.double()
        assert float((a64 - b64).norm() / b64.norm()) < 1e-2


@pytest.mark.parametrize("deterministic", [False, True])
def test_varlen_single_pass(ea, deterministic):
    ql = [5, 300, 0, 257, 700, 1, 130]
    kl = [7, 260, 3, 257, 640, 1, 0]
    H = 3
    t = workloads.make_varlen_qk(ql, kl, H, 64, 64, seed=19, device="cuda")
    args = (t["q"], t["k"], t["v"])
    o, lse = ea.attn_fwd_varlen(*args, t["cu_q"], t["cu_k"], max(ql), max(kl), causal=True)
    dq, dk, dv = ea.attn_bwd_varlen(*args, o, lse, t["do"], t["cu_q"], t["cu_k"], max(ql), max(kl), causal=True,
                                    deterministic=deterministic, single_pass=True)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == 0
    q, k, v, do = (x.cpu() for x in (t["q"], t["k"], t["v"], t["do"]))
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    cq, ck = t["cu_q"].cpu().numpy(), t["cu_k"].cpu().numpy()
    for s in range(len(ql)):
        a, b, c, d = int(cq[s]), int(cq[s + 1]), int(ck[s]), int(ck[s + 1])
        for h in range(H):
            if b > a and d > c:
                ref = attention_bwd(q[a:b, h], k[c:d, h], v[c:d, h], do[a:b, h], 0.125, True)
                check_grads({"dq": dq[a:b, h], "dk": dk[c:d, h], "dv": dv[c:d, h]}, ref, f"seq{s} h{h}")
            elif b > a:
                assert torch.all(dq[a:b, h] == 0)
            elif d > c:
                assert torch.all(dk[c:d, h] == 0) and torch.all(dv[c:d, h] == 0)


def test_single_pass_rejections(ea):
    x = torch.zeros((1, 128, 2, 128), device="cuda", dtype=torch.bfloat16)
    o, lse = ea.attn_fwd(x, x, x)
    with pytest.raises(ea.AttnError):  # d = 64 only
        ea.attn_bwd(x, x, x, o, lse, x, single_pass=True)
    y = torch.zeros((1, 128, 2, 64), device="cuda", dtype=torch.bfloat16)
    o, lse = ea.attn_fwd(y, y, y, softcap=2.0)
    with pytest.raises(ea.AttnError):  # no score modification
        ea.attn_bwd(y, y, y, o, lse, y, single_pass=True, softcap=2.0)
