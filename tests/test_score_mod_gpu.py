"""Score modifications (logit soft-capping, ALiBi distance bias) and block lists
per (batch, head), forward and backward, through the C ABI against the fp64
oracle, element by element on every (batch, head) of small shapes that span
several tiles with ragged tails. The backward is also checked for bitwise
reproducibility, and lists per (batch, head) that repeat one shared set must
give the shared-list result bit for bit."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attention_bwd, attention_fwd, block_sparse_visible
from parity import check_fwd, check_grads

pytestmark = pytest.mark.gpu

DIMS = [(64, 64), (128, 128), (192, 128)]


@pytest.fixture(scope="module")
def ea():
    import exact_attention_bf16_gb300 as ea
    return ea


def alibi_slopes(heads):
    """The usual geometric ALiBi slopes 2^(-8 (h + 1) / H)."""
    return np.array([2.0 ** (-8.0 * (h + 1) / heads) for h in range(heads)], dtype=np.float32)


def mods(heads):
    return {"softcap_1.5": dict(softcap=1.5), "softcap_30": dict(softcap=30.0),
            "alibi": dict(alibi_slopes=alibi_slopes(heads))}


def oracle_mod(kw, h):
    if "softcap" in kw:
        return ("softcap", kw["softcap"])
    return ("alibi", float(kw["alibi_slopes"][h]))


def to_gpu(kw):
    return {k: (torch.from_numpy(v).cuda() if isinstance(v, np.ndarray) else v) for k, v in kw.items()}


@pytest.mark.parametrize("dims", DIMS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mod", ["softcap_1.5", "softcap_30", "alibi"])
@pytest.mark.parametrize("nq,nk", [(300, 300), (200, 520)])
def test_dense_forward_and_backward(ea, dims, causal, mod, nq, nk):
    dqk, dv = dims
    w = workloads.Workload("sm", 2, 3, nq, nk, dqk, dv, causal, seed=nq + nk + dqk)
    t = workloads.make_dense(w, device="cuda")
    kw = mods(w.heads)[mod]
    g = to_gpu(kw)
    o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=causal, softmax_scale=w.scale, **g)
    g1 = ea.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=causal, softmax_scale=w.scale, **g)
    g2 = ea.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=causal, softmax_scale=w.scale,
                     deterministic=True, **g)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == 0
    for a, b in zip(g1, g2):
        assert torch.equal(a, b), "backward is not bitwise reproducible"
    q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
    dq, dk, dvv = (x.cpu() for x in g1)
    for b in range(w.batch):
        for h in range(w.heads):
            sm = oracle_mod(kw, h)
            oo, ll = attention_fwd(q[b, :, h], k[b, :, h], v[b, :, h], w.scale, causal, score_mod=sm)
            check_fwd(o[b, :, h], lse[b, h], oo, ll, f"{mod} b{b} h{h}")
            ref = attention_bwd(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], w.scale, causal, score_mod=sm)
            check_grads({"dq": dq[b, :, h], "dk": dk[b, :, h], "dv": dvv[b, :, h]}, ref, f"{mod} b{b} h{h}")


@pytest.mark.parametrize("mod", ["softcap_1.5", "alibi"])
def test_varlen_positions_restart_per_sequence(ea, mod):
    ql = [5, 300, 0, 257, 700, 1]
    kl = [7, 260, 3, 257, 640, 1]
    H = 4
    t = workloads.make_varlen_qk(ql, kl, H, 128, 128, seed=41, device="cuda")
    kw = mods(H)[mod]
    g = to_gpu(kw)
    scale = 128 ** -0.5
    args = (t["q"], t["k"], t["v"])
    o, lse = ea.attn_fwd_varlen(*args, t["cu_q"], t["cu_k"], max(ql), max(kl), causal=True, **g)
    dq, dk, dv = ea.attn_bwd_varlen(*args, o, lse, t["do"], t["cu_q"], t["cu_k"], max(ql), max(kl), causal=True, **g)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == 0
    q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
    cq, ck = t["cu_q"].cpu().numpy(), t["cu_k"].cpu().numpy()
    for s in range(len(ql)):
        a, b, c, d = int(cq[s]), int(cq[s + 1]), int(ck[s]), int(ck[s + 1])
        if b == a or d == c:
            continue
        for h in range(H):
            sm = oracle_mod(kw, h)
            oo, ll = attention_fwd(q[a:b, h], k[c:d, h], v[c:d, h], scale, True, score_mod=sm)
            check_fwd(o[a:b, h], lse[h, a:b], oo, ll, f"seq{s} h{h}")
            ref = attention_bwd(q[a:b, h], k[c:d, h], v[c:d, h], do[a:b, h], scale, True, score_mod=sm)
            check_grads({"dq": dq[a:b, h], "dk": dk[c:d, h], "dv": dv[c:d, h]}, ref, f"seq{s} h{h}")


def per_head_lists(B, H, nq, nk, seed, density=0.5):
    """Random lists, a different set per (batch, head), some query blocks empty."""
    rng = np.random.default_rng(seed)
    nqb, nkb = math.ceil(nq / 256), math.ceil(nk / 128)
    rows = [[[sorted(rng.choice(nkb, size=rng.integers(0, nkb + 1), replace=False).tolist()) if rng.random() < 0.9
              else [] for _ in range(nqb)] for _ in range(H)] for _ in range(B)]
    max_kv = max(1, max(len(r) for bb in rows for hh in bb for r in hh))
    cnt = np.zeros((B, H, nqb), dtype=np.int32)
    idx = np.zeros((B, H, nqb, max_kv), dtype=np.int32)
    for b in range(B):
        for h in range(H):
            for qb, r in enumerate(rows[b][h]):
                r = list(r)
                rng.shuffle(r)  # any order
                cnt[b, h, qb] = len(r)
                idx[b, h, qb, :len(r)] = r
    return cnt, idx


@pytest.mark.parametrize("dims", DIMS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mod", [None, "softcap_30", "alibi"])
def test_block_lists_per_batch_and_head(ea, dims, causal, mod):
    dqk, dv = dims
    B, H, nq, nk = 2, 3, 600, 700
    w = workloads.Workload("bh", B, H, nq, nk, dqk, dv, causal, seed=dqk + causal)
    t = workloads.make_dense(w, device="cuda")
    cnt, idx = per_head_lists(B, H, nq, nk, seed=dqk * 3 + causal)
    kc, ki = torch.from_numpy(cnt).cuda(), torch.from_numpy(idx).cuda()
    kw = mods(H)[mod] if mod else {}
    g = to_gpu(kw)
    o, lse = ea.attn_fwd_block_sparse(t["q"], t["k"], t["v"], kc, ki, causal=causal, softmax_scale=w.scale, **g)
    dq, dk, dvv = ea.attn_bwd_block_sparse(t["q"], t["k"], t["v"], o, lse, t["do"], kc, ki, causal=causal,
                                           softmax_scale=w.scale, **g)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == 0
    q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
    dq, dk, dvv = dq.cpu(), dk.cpu(), dvv.cpu()
    for b in range(B):
        for h in range(H):
            vis = block_sparse_visible(nq, nk, cnt[b, h], idx[b, h])
            sm = oracle_mod(kw, h) if mod else None
            oo, ll = attention_fwd(q[b, :, h], k[b, :, h], v[b, :, h], w.scale, causal, visible=vis, score_mod=sm)
            check_fwd(o[b, :, h], lse[b, h], oo, ll, f"b{b} h{h}")
            ref = attention_bwd(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], w.scale, causal, visible=vis,
                                score_mod=sm)
            check_grads({"dq": dq[b, :, h], "dk": dk[b, :, h], "dv": dvv[b, :, h]}, ref, f"b{b} h{h}")


def test_per_head_lists_repeating_one_set_match_shared_lists_bitwise(ea):
    B, H, nq, nk = 2, 4, 1000, 900
    w = workloads.Workload("rep", B, H, nq, nk, 128, 128, True, seed=12)
    t = workloads.make_dense(w, device="cuda")
    cnt, idx = per_head_lists(1, 1, nq, nk, seed=5)
    shared_c, shared_i = torch.from_numpy(cnt[0, 0]).cuda(), torch.from_numpy(idx[0, 0]).cuda()
    rep_c = shared_c.expand(B, H, -1).contiguous()
    rep_i = shared_i.expand(B, H, -1, -1).contiguous()
    args = (t["q"], t["k"], t["v"])
    o1, l1 = ea.attn_fwd_block_sparse(*args, shared_c, shared_i, causal=True)
    o2, l2 = ea.attn_fwd_block_sparse(*args, rep_c, rep_i, causal=True)
    g1 = ea.attn_bwd_block_sparse(*args, o1, l1, t["do"], shared_c, shared_i, causal=True)
    g2 = ea.attn_bwd_block_sparse(*args, o1, l1, t["do"], rep_c, rep_i, causal=True)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_autograd_wrapper_with_softcap(ea):
    g = torch.Generator(device="cuda").manual_seed(8)
    q, k, v = (torch.randn((2, 260, 4, 64), generator=g, device="cuda").to(torch.bfloat16).requires_grad_(True)
               for _ in range(3))
    do = torch.randn((2, 260, 4, 64), generator=g, device="cuda").to(torch.bfloat16)
    o = ea.attention(q, k, v, causal=True, softcap=2.0)
    o.backward(do)
    qc, kc, vc, doc = (x.detach().cpu() for x in (q, k, v, do))
    for b in range(2):
        for h in range(4):
            oo, ll = attention_fwd(qc[b, :, h], kc[b, :, h], vc[b, :, h], 0.125, True, score_mod=("softcap", 2.0))
            assert np.abs(o[b, :, h].detach().cpu().double().numpy() - oo).max() < 1e-2
            ref = attention_bwd(qc[b, :, h], kc[b, :, h], vc[b, :, h], doc[b, :, h], 0.125, True,
                                score_mod=("softcap", 2.0))
            check_grads({"dq": q.grad[b, :, h], "dk": k.grad[b, :, h], "dv": v.grad[b, :, h]}, ref, f"b{b} h{h}")


def test_score_mod_rejections_on_the_gpu(ea):
    q = torch.zeros((1, 128, 2, 64), device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ea.attn_fwd(q, q, q, softcap=2.0, alibi_slopes=torch.zeros(2, device="cuda"))
    with pytest.raises(ValueError):
        ea.attn_fwd(q, q, q, alibi_slopes=torch.zeros(3, device="cuda"))  # one slope per head
    with pytest.raises(ea.AttnError):
        ea.attn_fwd(q, q, q, softcap=2.0, exp2_emu_period=8)  # emulated exp2 is not built with a modification
    q128 = torch.zeros((1, 128, 2, 128), device="cuda", dtype=torch.bfloat16)
    o, lse = ea.attn_fwd(q128, q128, q128, softcap=2.0)
    with pytest.raises(ea.AttnError):
        ea.attn_bwd(q128, q128, q128, o, lse, q128, softcap=2.0, cta_pair=True)
