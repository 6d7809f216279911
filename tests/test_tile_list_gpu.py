"""Packed variable-length launches run from a tile list: one CTA per real block
of a sequence, the sequences with the most blocks first. These cases stress the
list builder (more sequences than it has threads, runs of empty sequences,
query and key lengths that differ) and check that every sequence gets bitwise
the result of a dense call on that sequence alone (one batch entry, CTAs from
the block index), besides the oracle on a seeded sample of sequences. A
max_seqlen above the list's limit (2047 blocks of rows) makes the call launch
from the block index instead; that path gets the same comparison."""
import numpy as np
import pytest
import torch

import workloads
from oracle import attention_bwd, attention_fwd
from parity import check_fwd, check_grads

pytestmark = pytest.mark.gpu

FWD_LIST_MAX = 2047 * 256  # longest sequence, in rows, the forward builds a list for
BWD_LIST_MAX = 2047 * 128  # the same for the backward (128-row blocks)


def same_as_dense(ea, t, o, lse, grads, causal, scale, seqs=None):
    """Each sequence's varlen result equals, bit for bit, a dense call on it alone."""
    cq, ck = t["cu_q"].cpu().tolist(), t["cu_k"].cpu().tolist()
    for s in seqs if seqs is not None else range(len(cq) - 1):
        a, b, c, d = cq[s], cq[s + 1], ck[s], ck[s + 1]
        if b == a and d == c:
            continue
        q, k, v, do = (x.unsqueeze(0) for x in (t["q"][a:b], t["k"][c:d], t["v"][c:d], t["do"][a:b]))
        od, ld = ea.attn_fwd(q, k, v, causal=causal, softmax_scale=scale)
        assert torch.equal(od[0], o[a:b]) and torch.equal(ld[0], lse[:, a:b]), f"seq{s}: forward differs"
        if b > a and d > c:
            gd = ea.attn_bwd(q, k, v, od, ld, do, causal=causal, softmax_scale=scale, deterministic=True)
            for n, x, y in zip(("dq", "dk", "dv"), gd, (grads[0][a:b], grads[1][c:d], grads[2][c:d])):
                assert torch.equal(x[0], y), f"seq{s}: {n} differs"


def lengths(n, seed):
    """A length mix with many empty sequences, most short, a few long."""
    rng = np.random.default_rng(seed)
    kind = rng.choice(3, size=n, p=[0.3, 0.6, 0.1])
    short = rng.integers(1, 200, size=n)
    long = rng.integers(200, 700, size=n)
    return [int(x) for x in np.where(kind == 0, 0, np.where(kind == 1, short, long))]


@pytest.mark.parametrize("dims", [(64, 64), (128, 128), (192, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_many_sequences(dims, causal):
    import exact_attention_bf16_gb300 as ea
    dqk, dv_ = dims
    S, H = 1300, 2
    ql = lengths(S, 40 + dqk)
    kl = [q if s % 2 == 0 else k for s, (q, k) in enumerate(zip(ql, lengths(S, 90 + dqk)))]
    t = workloads.make_varlen_qk(ql, kl, H, dqk, dv_, seed=dqk + causal, device="cuda")
    scale = 1.0 / np.sqrt(dqk)
    Lq, Lk = max(ql), max(kl)
    args = (t["q"], t["k"], t["v"])
    o, lse = ea.attn_fwd_varlen(*args, t["cu_q"], t["cu_k"], Lq, Lk, causal=causal, softmax_scale=scale)
    g = ea.attn_bwd_varlen(*args, o, lse, t["do"], t["cu_q"], t["cu_k"], Lq, Lk, causal=causal,
                           softmax_scale=scale, deterministic=True)
    g3 = ea.attn_bwd_varlen(*args, o, lse, t["do"], t["cu_q"], t["cu_k"], Lq, Lk, causal=causal,
                            softmax_scale=scale)
    torch.cuda.synchronize()
    ea.attn_get_device_status()
    for n, a, b in zip(("dq", "dk", "dv"), g, g3):
        assert torch.equal(a, b), f"backward {n}: not reproducible"
    same_as_dense(ea, t, o, lse, g, causal, scale)
    dq, dk, dv = g3
    q, k, v, do = (t[n].cpu() for n in ("q", "k", "v", "do"))
    cq, ck = t["cu_q"].cpu().numpy(), t["cu_k"].cpu().numpy()
    o_c, lse_c, dq_c, dk_c, dv_c = (x.cpu() for x in (o, lse, dq, dk, dv))
    for s in range(S):  # sequences with no queries or no keys: exact zeros and -inf
        a, b, c, d = int(cq[s]), int(cq[s + 1]), int(ck[s]), int(ck[s + 1])
        if b > a and d == c:
            assert torch.all(o_c[a:b] == 0) and torch.all(torch.isneginf(lse_c[:, a:b])), f"seq{s}"
            assert torch.all(dq_c[a:b] == 0), f"seq{s}"
        if d > c and b == a:
            assert torch.all(dk_c[c:d] == 0) and torch.all(dv_c[c:d] == 0), f"seq{s}"
    rng = np.random.default_rng(7)
    live = [s for s in range(S) if ql[s] and kl[s]]
    pick = sorted(set(rng.choice(live, size=24, replace=False).tolist()) | {int(np.argmax(ql)), live[-1]})
    for s in pick:
        a, b, c, d = int(cq[s]), int(cq[s + 1]), int(ck[s]), int(ck[s + 1])
        h = s % H
        oo, ll = attention_fwd(q[a:b, h], k[c:d, h], v[c:d, h], scale, causal)
        check_fwd(o_c[a:b, h], lse_c[h, a:b], oo, ll, f"seq{s} h{h}")
        ref = attention_bwd(q[a:b, h], k[c:d, h], v[c:d, h], do[a:b, h], scale, causal)
        check_grads({"dq": dq_c[a:b, h], "dk": dk_c[c:d, h], "dv": dv_c[c:d, h]}, ref, f"seq{s} h{h}")


def test_single_sequence_and_all_empty_but_one():
    """One real sequence among many empty ones, placed last: the list holds
    its blocks only and every other CTA of the bounded grid exits."""
    import exact_attention_bf16_gb300 as ea
    ql = [0] * 1100 + [777]
    t = workloads.make_varlen_qk(ql, ql, 3, 128, 128, seed=5, device="cuda")
    o, lse = ea.attn_fwd_varlen(t["q"], t["k"], t["v"], t["cu_q"], t["cu_k"], 777, 777, causal=True)
    dq, dk, dv = ea.attn_bwd_varlen(t["q"], t["k"], t["v"], o, lse, t["do"], t["cu_q"], t["cu_k"], 777, 777,
                                    causal=True)
    torch.cuda.synchronize()
    ea.attn_get_device_status()
    q, k, v, do = (x.cpu() for x in (t["q"], t["k"], t["v"], t["do"]))
    for h in range(3):
        oo, ll = attention_fwd(q[:, h], k[:, h], v[:, h], 128 ** -0.5, True)
        check_fwd(o[:, h], lse[h], oo, ll, f"h{h}")
        ref = attention_bwd(q[:, h], k[:, h], v[:, h], do[:, h], 128 ** -0.5, True)
        check_grads({"dq": dq[:, h], "dk": dk[:, h], "dv": dv[:, h]}, ref, f"h{h}")


def test_block_index_path_beyond_the_list_limit():
    """A sequence longer than the list's limit: the calls launch from the block
    index (a grid slice of max_seqlen rows per sequence) and still give each
    sequence bitwise the dense result."""
    import exact_attention_bf16_gb300 as ea
    ql = [300, FWD_LIST_MAX + 68, 0, 129]
    t = workloads.make_varlen_qk(ql, ql, 1, 64, 64, seed=23, device="cuda")
    L = max(ql)
    assert L > FWD_LIST_MAX and L > BWD_LIST_MAX
    o, lse = ea.attn_fwd_varlen(t["q"], t["k"], t["v"], t["cu_q"], t["cu_k"], L, L, causal=True)
    g = ea.attn_bwd_varlen(t["q"], t["k"], t["v"], o, lse, t["do"], t["cu_q"], t["cu_k"], L, L, causal=True,
                           deterministic=True)
    torch.cuda.synchronize()
    ea.attn_get_device_status()
    same_as_dense(ea, t, o, lse, g, True, 64 ** -0.5)
    q, k, v, do = (x.cpu() for x in (t["q"][:300], t["k"][:300], t["v"][:300], t["do"][:300]))
    oo, ll = attention_fwd(q[:, 0], k[:, 0], v[:, 0], 64 ** -0.5, True)
    check_fwd(o[:300, 0], lse[0, :300], oo, ll, "seq0")
