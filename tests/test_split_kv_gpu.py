"""Dense forwards whose (query block, head, batch) grid would leave most SMs
idle and whose keys are long run with the keys split across CTAs: each CTA
computes O and the LSE over one range of key blocks, and a second kernel merges
the ranges (LSE = ln sum_r exp(LSE_r), O = sum_r exp(LSE_r - LSE) O_r).

The outputs are compared with the oracle on every element, for d = 64 and 128,
with and without the causal mask (bottom-right, so with Nq < Nk every row sees
most keys, and with Nq = Nk the early rows see no key of the later ranges), on
ragged lengths; the backward runs on the split forward's O and LSE; and two
calls must give the same bits.

The dense backward splits the keys of its dQ kernel by the same rule over its
128-row query tiles: each CTA stores the fp32 dQ of one key range and a merge
kernel adds the ranges in order. Its gradients are compared with the oracle,
with the same call run unsplit (a workspace that holds only the D vector: dK
and dV must be the same bits, dQ the same within rounding), and with a repeat
call (the same bits), including ranges that see no key and the full-size
short-query, long-key shape."""
import ctypes

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


def _bwd_through_abi(ea, t, o, lse, w, ws_bytes=None):
    """attn_bwd through the C ABI with a workspace of ws_bytes (default: the size
    attn_bwd_workspace_size gives). Returns ((dq, dk, dv), that size)."""
    from exact_attention_bf16_gb300 import _abi as abi
    lib = abi.load()
    grads = [torch.full_like(t[n], float("nan")) for n in ("q", "k", "v")]
    p = abi.AttnBwdParams()
    ea._fill_fwd(p.fwd, t["q"], t["k"], t["v"], o, lse, ea._strides4, w.scale, w.causal)
    p.fwd.batch, p.fwd.seqlen_q, p.fwd.seqlen_k = w.batch, w.seqlen_q, w.seqlen_k
    ea._fill_bwd(p, t["do"], *grads, ea._strides4, False)
    full = lib.attn_bwd_workspace_size(ctypes.byref(p))
    nbytes = full if ws_bytes is None else ws_bytes
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.attn_bwd(ctypes.byref(p), ctypes.c_void_p(ws.data_ptr()), nbytes, stream) == abi.ATTN_OK
    torch.cuda.synchronize()
    ea.attn_get_device_status()
    return grads, full


def _split_dq_case(w, heads_vs_oracle):
    import exact_attention_bf16_gb300 as ea
    from parity import rel_fro, to64
    t = workloads.make_dense(w, device="cuda")
    o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=w.causal, softmax_scale=w.scale)
    torch.cuda.synchronize()
    split, full = _bwd_through_abi(ea, t, o, lse, w)
    d_only = (4 * w.batch * w.heads * w.seqlen_q + 255) // 256 * 256
    assert full > d_only, "this shape should split the dQ kernel's keys"
    again, _ = _bwd_through_abi(ea, t, o, lse, w)
    whole, _ = _bwd_through_abi(ea, t, o, lse, w, d_only)
    what = f"split dQ {w.name} d{w.d_qk} causal={w.causal}"
    for n, a, b in zip(("dq", "dk", "dv"), split, again):
        assert torch.equal(a, b), f"{what}: {n} differs between two calls"
    assert torch.equal(split[1], whole[1]) and torch.equal(split[2], whole[2]), f"{what}: dK/dV changed"
    r = rel_fro(to64(split[0]), to64(whole[0]))
    assert r <= 1e-3, f"{what}: split dQ vs unsplit rel {r:.2e}"
    q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
    for b, h in heads_vs_oracle:
        ref = attention_bwd(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], w.scale, w.causal)
        check_grads({"dq": split[0][b, :, h], "dk": split[1][b, :, h], "dv": split[2][b, :, h]}, ref,
                    f"{what} b{b} h{h}")


@pytest.mark.parametrize("dims", [(64, 64), (128, 128), (192, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_split_dq(dims, causal):
    # 6 query tiles of 128 (ragged), 20 key blocks (ragged): 2 ranges of 10
    w = workloads.Workload("sq", 1, 2, 300, 2500, dims[0], dims[1], causal, seed=64)
    _split_dq_case(w, [(0, 0), (0, 1)])


def test_backward_split_dq_ranges_without_visible_keys():
    """Causal, Nq = Nk = 2048: 16 query tiles, 2 ranges of 8 key blocks; the first
    eight tiles see no key of the second range, whose partial is zero."""
    w = workloads.Workload("sq_square", 1, 1, 2048, 2048, 128, 128, True, seed=65)
    _split_dq_case(w, [(0, 0)])


@pytest.mark.parametrize("causal", [False, True])
def test_backward_split_dq_full_size(causal):
    """B1 H16 Nq 512, Nk 32768, d 128 (the benchmark's short-query shape): 64
    query tiles, 2 ranges of 128 key blocks; two heads against the oracle."""
    w = workloads.Workload("sq_full", 1, 16, 512, 32768, 128, 128, causal, seed=66)
    _split_dq_case(w, [(0, 0), (0, 15)])
