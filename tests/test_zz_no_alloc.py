"""attn_bwd_noalloc, the backward entry point for callers that cannot allocate
device memory (for example an engine that plans all memory at start-up and
forbids later cudaMalloc, or a plugin that is only handed tensors): it must
give exactly the gradients of attn_bwd with a caller-provided workspace (the
same kernels run, and both are bitwise reproducible), on two calls in a row
(the second reuses the library's fixed scratch array left over from the
first), dense and packed variable-length, in both modes, and must refuse
problems larger than that array. The dense gradients are also compared with
the fp64 oracle on one (batch, head) pair.

This file is named so that pytest collects it last."""
import ctypes

import pytest
import torch

import workloads
from oracle import attention_bwd
from parity import check_grads

pytestmark = pytest.mark.gpu


def _params(ea, abi, t, w, o, lse, dq, dk, dv, deterministic=False):
    p = abi.AttnBwdParams()
    ea._fill_fwd(p.fwd, t["q"], t["k"], t["v"], o, lse, ea._strides4, w.scale, w.causal)
    p.fwd.batch, p.fwd.seqlen_q, p.fwd.seqlen_k = w.batch, w.seqlen_q, w.seqlen_k
    ea._fill_bwd(p, t["do"], dq, dk, dv, ea._strides4, deterministic)
    return p


def _two_calls(lib, abi, make_params, like, ref, what):
    import exact_attention_bf16_gb300 as ea
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        grads = [torch.full_like(x, float("nan")) for x in like]
        p = make_params(*grads)
        assert lib.attn_bwd_noalloc(ctypes.byref(p), stream) == abi.ATTN_OK
        torch.cuda.synchronize()
        ea.attn_get_device_status()
        for name, got, want in zip(("dq", "dk", "dv"), grads, ref):
            assert torch.equal(got, want), f"{what} call {call}: {name} differs from attn_bwd"


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("dims,causal", [((128, 128), True), ((64, 64), False), ((192, 128), True)])
def test_noalloc_matches_workspace_entry_point(dims, causal, deterministic):
    import exact_attention_bf16_gb300 as ea
    from exact_attention_bf16_gb300 import _abi as abi
    lib = abi.load()
    dqk, dv_ = dims
    w = workloads.Workload("noalloc", 2, 4, 1000, 1000, dqk, dv_, causal, seed=21)
    t = workloads.make_dense(w, device="cuda")
    o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=causal, softmax_scale=w.scale)
    ref = ea.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=causal, softmax_scale=w.scale,
                      deterministic=deterministic)
    torch.cuda.synchronize()
    _two_calls(lib, abi, lambda dq, dk, dv: _params(ea, abi, t, w, o, lse, dq, dk, dv, deterministic),
               (t["q"], t["k"], t["v"]), ref, f"dense {dims} causal={causal} det={deterministic}")
    b, h = 1, 2  # the no-allocation gradients equal ref bit for bit (above); ref against the oracle
    q, k, v, do = (t[n][b, :, h].cpu() for n in ("q", "k", "v", "do"))
    want = attention_bwd(q, k, v, do, w.scale, causal)
    check_grads({"dq": ref[0][b, :, h], "dk": ref[1][b, :, h], "dv": ref[2][b, :, h]}, want,
                f"no-allocation dense {dims} causal={causal} det={deterministic} b{b} h{h}")


def test_noalloc_varlen_matches_workspace_entry_point():
    """Packed sequences: the scratch size comes from heads x total_q."""
    import exact_attention_bf16_gb300 as ea
    from exact_attention_bf16_gb300 import _abi as abi
    lib = abi.load()
    lens = [300, 1, 0, 700, 129]
    w = workloads.Workload("noalloc_vl", 1, 3, max(lens), max(lens), 128, 128, True, seed=22,
                           varlen_lengths=tuple(lens))
    t = workloads.make_varlen(w, device="cuda")
    cu, L = t["cu_seqlens"], max(lens)
    o, lse = ea.attn_fwd_varlen(t["q"], t["k"], t["v"], cu, cu, L, L, causal=True, softmax_scale=w.scale)
    ref = ea.attn_bwd_varlen(t["q"], t["k"], t["v"], o, lse, t["do"], cu, cu, L, L, causal=True,
                             softmax_scale=w.scale)
    torch.cuda.synchronize()

    def make(dq, dk, dv):
        p = abi.AttnBwdParams()
        ea._fill_fwd(p.fwd, t["q"], t["k"], t["v"], o, lse, ea._strides3, w.scale, True)
        p.fwd.cu_seqlens_q = p.fwd.cu_seqlens_k = ctypes.c_void_p(cu.data_ptr())
        p.fwd.num_seqs = len(lens)
        p.fwd.max_seqlen_q = p.fwd.max_seqlen_k = L
        p.fwd.total_q = p.fwd.total_k = sum(lens)
        p.fwd.batch = 1
        ea._fill_bwd(p, t["do"], dq, dk, dv, ea._strides3, False)
        return p

    _two_calls(lib, abi, make, (t["q"], t["k"], t["v"]), ref, "varlen")


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
