"""Block-sparse forward (attn_fwd_block_sparse) against the fp64 oracle with the
same block lists turned into key visibility element by element, and against the
dense forward when every block is listed."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attention_fwd, block_sparse_visible
from parity import check_fwd

pytestmark = pytest.mark.gpu

DIMS = [(64, 64), (128, 128), (192, 128)]


@pytest.fixture(scope="module")
def ea():
    import exact_attention_bf16_gb300 as ea
    return ea


def random_lists(nq, nk, density, seed, extra=None):
    rng = np.random.default_rng(seed)
    nqb, nkb = math.ceil(nq / 256), math.ceil(nk / 128)
    cnt = np.zeros(nqb, dtype=np.int32)
    rows = []
    for b in range(nqb):
        blocks = [kb for kb in range(nkb) if rng.random() < density]
        rng.shuffle(blocks)  # any order
        cnt[b] = len(blocks)
        rows.append(blocks)
    if extra:
        for b, blocks in extra.items():
            rows[b] = blocks
            cnt[b] = len(blocks)
    max_kv = max(1, max(len(r) for r in rows))
    idx = np.zeros((nqb, max_kv), dtype=np.int32)
    for b, r in enumerate(rows):
        idx[b, :len(r)] = r
    return cnt, idx


def run_sparse(ea, w, cnt, idx, pairs=None):
    t = workloads.make_dense(w, device="cuda", with_do=False)
    kc = torch.from_numpy(cnt).cuda()
    ki = torch.from_numpy(idx).cuda()
    o, lse = ea.attn_fwd_block_sparse(t["q"], t["k"], t["v"], kc, ki, causal=w.causal, softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == 0
    vis = block_sparse_visible(w.seqlen_q, w.seqlen_k, cnt, idx)
    q, k, v = (t[n].cpu() for n in ("q", "k", "v"))
    pairs = pairs or [(b, h) for b in range(w.batch) for h in range(w.heads)]
    for b, h in pairs:
        o_ref, l_ref = attention_fwd(q[b, :, h], k[b, :, h], v[b, :, h], w.scale, w.causal, row_block=1024,
                                     visible=vis)
        check_fwd(o[b, :, h], lse[b, h], o_ref, l_ref, f"{w.name} b{b} h{h}")
    return t, o, lse


@pytest.mark.parametrize("dims", DIMS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk,density", [(300, 700, 0.5), (513, 513, 0.3), (1000, 260, 0.7), (200, 1500, 0.2)])
def test_random_block_lists(ea, dims, causal, nq, nk, density):
    dqk, dv = dims
    w = workloads.Workload("bs", 2, 3, nq, nk, dqk, dv, causal, seed=nq + nk + dqk)
    # query block 0 lists nothing: its rows must come out O = 0, LSE = -inf
    cnt, idx = random_lists(nq, nk, density, seed=nq * 7 + nk, extra={0: []})
    run_sparse(ea, w, cnt, idx)


@pytest.mark.parametrize("causal", [False, True])
def test_every_block_listed_matches_the_dense_forward_bitwise(ea, causal):
    # the listed blocks in ascending order are exactly the dense kernel's key walk
    nq = nk = 1000
    w = workloads.Workload("all", 2, 4, nq, nk, 128, 128, causal, seed=3)
    nqb, nkb = math.ceil(nq / 256), math.ceil(nk / 128)
    cnt = np.full(nqb, nkb, dtype=np.int32)
    if causal:  # the dense causal walk stops at the query block's last visible key block
        cnt = np.array([math.ceil(min(nk, 256 * (b + 1)) / 128) for b in range(nqb)], dtype=np.int32)
    idx = np.tile(np.arange(nkb, dtype=np.int32), (nqb, 1))
    t, o, lse = run_sparse(ea, w, cnt, idx, pairs=[(0, 0), (1, 3)])
    o_d, l_d = ea.attn_fwd(t["q"], t["k"], t["v"], causal=causal, softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o, o_d) and torch.equal(lse, l_d)


def test_out_of_range_indices_and_counts_are_ignored(ea):
    nq, nk = 512, 384
    w = workloads.Workload("oor", 1, 2, nq, nk, 64, 64, False, seed=9)
    # block 0: [1, -5, 99] with count 3 → only key block 1 is real; block 1: count 7 > max_kv (clamped to 3)
    cnt = np.array([3, 7], dtype=np.int32)
    idx = np.array([[1, -5, 99], [2, 0, 2**30]], dtype=np.int32)
    run_sparse(ea, w, cnt, idx)


def test_sliding_window_sampled(ea):
    # a local-attention pattern at a larger size: query block b sees key blocks 2b-3 .. 2b+1
    nq = nk = 8192
    w = workloads.Workload("window", 2, 8, nq, nk, 128, 128, True, seed=21)
    nqb, nkb = nq // 256, nk // 128
    rows = [[kb for kb in range(2 * b - 3, 2 * b + 2) if 0 <= kb < nkb] for b in range(nqb)]
    cnt = np.array([len(r) for r in rows], dtype=np.int32)
    idx = np.zeros((nqb, 5), dtype=np.int32)
    for b, r in enumerate(rows):
        idx[b, :len(r)] = r
    run_sparse(ea, w, cnt, idx, pairs=[(0, 0), (1, 5)])


def run_sparse_bwd(ea, w, cnt, idx, pairs=None):
    from oracle import attention_bwd
    from parity import check_grads
    t = workloads.make_dense(w, device="cuda", with_do=True)
    kc = torch.from_numpy(cnt).cuda()
    ki = torch.from_numpy(idx).cuda()
    o, lse = ea.attn_fwd_block_sparse(t["q"], t["k"], t["v"], kc, ki, causal=w.causal, softmax_scale=w.scale)
    dq, dk, dv = ea.attn_bwd_block_sparse(t["q"], t["k"], t["v"], o, lse, t["do"], kc, ki, causal=w.causal,
                                          softmax_scale=w.scale)
    dq2, dk2, dv2 = ea.attn_bwd_block_sparse(t["q"], t["k"], t["v"], o, lse, t["do"], kc, ki, causal=w.causal,
                                             softmax_scale=w.scale, deterministic=True)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == 0
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)  # reproducible
    vis = block_sparse_visible(w.seqlen_q, w.seqlen_k, cnt, idx)
    q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
    pairs = pairs or [(b, h) for b in range(w.batch) for h in range(w.heads)]
    for b, h in pairs:
        ref = attention_bwd(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], w.scale, w.causal, row_block=1024,
                            visible=vis)
        check_grads({"dq": dq[b, :, h], "dk": dk[b, :, h], "dv": dv[b, :, h]}, ref, f"{w.name} b{b} h{h}")
    return t, o, lse, (dq, dk, dv)


@pytest.mark.parametrize("dims", DIMS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk,density", [(300, 700, 0.5), (1000, 260, 0.6), (513, 1100, 0.3)])
def test_backward_random_block_lists(ea, dims, causal, nq, nk, density):
    dqk, dv = dims
    w = workloads.Workload("bsb", 2, 2, nq, nk, dqk, dv, causal, seed=nq + 3 * nk + dqk)
    cnt, idx = random_lists(nq, nk, density, seed=nq * 5 + nk, extra={0: []})
    run_sparse_bwd(ea, w, cnt, idx)


@pytest.mark.parametrize("dims", DIMS)
@pytest.mark.parametrize("causal", [False, True])
def test_backward_every_block_listed_matches_the_dense_backward_bitwise(ea, dims, causal):
    # extra listed blocks the dense walk skips are fully masked and add exact zeros
    dqk, dv = dims
    nq = nk = 1000
    w = workloads.Workload("ball", 2, 2, nq, nk, dqk, dv, causal, seed=4)
    nqb, nkb = math.ceil(nq / 256), math.ceil(nk / 128)
    cnt = np.full(nqb, nkb, dtype=np.int32)
    if causal:
        cnt = np.array([math.ceil(min(nk, 256 * (b + 1)) / 128) for b in range(nqb)], dtype=np.int32)
    idx = np.tile(np.arange(nkb, dtype=np.int32), (nqb, 1))
    t, o, lse, (dq, dk, dv_) = run_sparse_bwd(ea, w, cnt, idx, pairs=[(1, 1)])
    o_d, l_d = ea.attn_fwd(t["q"], t["k"], t["v"], causal=causal, softmax_scale=w.scale)
    g = ea.attn_bwd(t["q"], t["k"], t["v"], o_d, l_d, t["do"], causal=causal, softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(dq, g[0]) and torch.equal(dk, g[1]) and torch.equal(dv_, g[2])


def test_autograd_block_mask(ea):
    # the autograd wrapper routes a block mask to the block-sparse forward and backward
    nq = nk = 600
    w = workloads.Workload("ag", 1, 2, nq, nk, 128, 128, True, seed=8)
    cnt, idx = random_lists(nq, nk, 0.5, seed=77)
    t = workloads.make_dense(w, device="cuda", with_do=True)
    q, k, v = (t[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    kc, ki = torch.from_numpy(cnt).cuda(), torch.from_numpy(idx).cuda()
    o = ea.attention(q, k, v, causal=True, block_mask=(kc, ki))
    o.backward(t["do"])
    o2, l2 = ea.attn_fwd_block_sparse(t["q"], t["k"], t["v"], kc, ki, causal=True)
    g = ea.attn_bwd_block_sparse(t["q"], t["k"], t["v"], o2, l2, t["do"], kc, ki, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o.detach(), o2)
    assert torch.equal(q.grad, g[0]) and torch.equal(k.grad, g[1]) and torch.equal(v.grad, g[2])
