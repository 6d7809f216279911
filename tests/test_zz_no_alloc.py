"""attn_bwd_noalloc, the backward entry point for callers that cannot allocate
device memory (for example an engine that plans all memory at start-up and
forbids later cudaMalloc, or a plugin that is only handed tensors): it must
give the same gradients as attn_bwd with a caller-provided workspace, on two
calls in a row (the second reuses the library's fixed scratch array left over
from the first), and must refuse problems larger than that array.

This file is named so that pytest collects it last."""
import ctypes

import pytest
import torch

import workloads
from parity import check_grads, to64

pytestmark = pytest.mark.gpu


def _params(ea, abi, t, w, o, lse, dq, dk, dv):
    p = abi.AttnBwdParams()
    ea._fill_fwd(p.fwd, t["q"], t["k"], t["v"], o, lse, ea._strides4, w.scale, w.causal)
    p.fwd.batch, p.fwd.seqlen_q, p.fwd.seqlen_k = w.batch, w.seqlen_q, w.seqlen_k
    ea._fill_bwd(p, t["do"], dq, dk, dv, ea._strides4, False)
    return p


@pytest.mark.parametrize("dims,causal", [((128, 128), True), ((64, 64), False), ((192, 128), True)])
def test_noalloc_matches_workspace_entry_point(dims, causal):
    import exact_attention_bf16_gb300 as ea
    from exact_attention_bf16_gb300 import _abi as abi
    lib = abi.load()
    dqk, dv_ = dims
    w = workloads.Workload("noalloc", 2, 4, 1000, 1000, dqk, dv_, causal, seed=21)
    t = workloads.make_dense(w, device="cuda")
    o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=causal, softmax_scale=w.scale)
    ref = ea.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=causal, softmax_scale=w.scale)
    torch.cuda.synchronize()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        dq, dk, dv = (torch.full_like(t[n], float("nan")) for n in ("q", "k", "v"))
        p = _params(ea, abi, t, w, o, lse, dq, dk, dv)
        assert lib.attn_bwd_noalloc(ctypes.byref(p), stream) == abi.ATTN_OK
        torch.cuda.synchronize()
        ea.attn_get_device_status()
        got = {"dq": dq, "dk": dk, "dv": dv}
        # same tolerance as the parity tests (relative Frobenius 1e-2), per (batch, head)
        for b in range(w.batch):
            for h in range(w.heads):
                check_grads({n: got[n][b, :, h] for n in got},
                            {n: to64(x[b, :, h]) for n, x in zip(("dq", "dk", "dv"), ref)},
                            f"noalloc call {call} b{b} h{h}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    import exact_attention_bf16_gb300 as ea
    from exact_attention_bf16_gb300 import _abi as abi
    lib = abi.load()
    rows = abi.BWD_NOALLOC_SCRATCH_BYTES // 4
    # one query row more than the fixed scratch holds; shapes only, nothing is launched
    w = workloads.Workload("big", 1, 1, rows + 1, 8, 64, 64, False)
    q = torch.empty((1, rows + 1, 1, 64), dtype=torch.bfloat16, device="cuda")
    kv = torch.empty((1, 8, 1, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, rows + 1), dtype=torch.float32, device="cuda")
    t = {"q": q, "k": kv, "v": kv, "do": o}
    p = _params(ea, abi, t, w, o, lse, torch.empty_like(q), torch.empty_like(kv), torch.empty_like(kv))
    assert lib.attn_bwd_workspace_size(ctypes.byref(p)) > abi.BWD_NOALLOC_SCRATCH_BYTES
    assert lib.attn_bwd_noalloc(ctypes.byref(p), None) == abi.ATTN_ERR_WORKSPACE
