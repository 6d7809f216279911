"""The two-SM dK/dV kernel (cta_pair=True: a cluster of two CTAs sharing one
tcgen05 MMA, accumulator split along the keys, B operand split along N)
against the fp64 oracle, through the same entry points as the default kernel:
ragged and unequal lengths, both masks, packed varlen, a sampled training
shape, and bitwise reproducibility."""
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


def _run(ea, t, w, cta_pair=True, deterministic=False):
    o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=w.causal, softmax_scale=w.scale)
    g = ea.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=w.causal, softmax_scale=w.scale,
                    deterministic=deterministic, cta_pair=cta_pair)
    torch.cuda.synchronize()
    ea.attn_get_device_status()
    return g


def _check(t, w, grads, pairs):
    q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
    dq, dk, dv = grads
    for b, h in pairs:
        ref = attention_bwd(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], w.scale, w.causal, row_block=2048)
        check_grads({"dq": dq[b, :, h], "dk": dk[b, :, h], "dv": dv[b, :, h]}, ref, f"pair {w.name} b{b} h{h}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk", [(1, 1), (17, 17), (128, 128), (200, 200), (256, 256), (257, 257), (384, 384),
                                   (513, 513), (100, 300), (300, 100), (384, 640), (1000, 1000)])
def test_pair_small_shapes(ea, causal, nq, nk):
    w = workloads.Workload("pair", 2, 3, nq, nk, 128, 128, causal, seed=nq * 5 + nk)
    t = workloads.make_dense(w, device="cuda")
    _check(t, w, _run(ea, t, w), [(b, h) for b in range(2) for h in range(3)])


def test_pair_varlen(ea):
    lens = [1, 130, 0, 257, 64, 300, 700]
    w = workloads.Workload("pvl", 1, 2, max(lens), max(lens), 128, 128, True, seed=12, varlen_lengths=tuple(lens))
    t = workloads.make_varlen(w, device="cuda")
    cu, L = t["cu_seqlens"], max(lens)
    o, lse = ea.attn_fwd_varlen(t["q"], t["k"], t["v"], cu, cu, L, L, causal=True, softmax_scale=w.scale)
    dq, dk, dv = ea.attn_bwd_varlen(t["q"], t["k"], t["v"], o, lse, t["do"], cu, cu, L, L, causal=True,
                                    softmax_scale=w.scale, cta_pair=True)
    torch.cuda.synchronize()
    ea.attn_get_device_status()
    cu_h = cu.cpu().numpy()
    q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
    for s in range(len(lens)):
        a, b = int(cu_h[s]), int(cu_h[s + 1])
        if b == a:
            continue
        for h in range(2):
            ref = attention_bwd(q[a:b, h], k[a:b, h], v[a:b, h], do[a:b, h], w.scale, True)
            check_grads({"dq": dq[a:b, h], "dk": dk[a:b, h], "dv": dv[a:b, h]}, ref, f"pair vl seq{s} h{h}")


def test_pair_training_shape_sampled_and_reproducible(ea):
    w = workloads.bwd_d128_N16384()
    t = workloads.make_dense(w, device="cuda")
    first = [x.clone() for x in _run(ea, t, w, deterministic=True)]
    for _ in range(3):
        again = _run(ea, t, w, deterministic=True)
        for a, b in zip(first, again):
            assert torch.equal(a, b), "the two-SM backward is not bitwise reproducible"
    _check(t, w, first, workloads.sample_pairs(w.batch, w.heads, 2, seed=16385))
