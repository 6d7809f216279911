"""Failure detection of the bounded waits, exercised on the GPU without a
fault or a hang: attn_diag_wait_timeout runs the forward kernel with its
loader issuing no copies and every wait limited to a small number of polls,
so the MMA and softmax waits run out. The call must return, the device status
must report ATTN_ERR_TIMEOUT with the site of a wait that gave up, and the
next normal call must work and pass parity."""
import ctypes

import pytest
import torch

import workloads
from oracle import attention_fwd
from parity import check_fwd

pytestmark = pytest.mark.gpu

# sites (low 24 bits of the status word) of the waits that can give up first:
# the MMA thread's Q waits and the softmax warps' S waits (forward kernel)
SITES = {0x200, 0x201, 0x300, 0x301}
DEV_TIMEOUT_MBAR = 1


def test_wait_that_runs_out_is_reported_and_the_context_survives():
    import exact_attention_bf16_gb300 as ea
    from exact_attention_bf16_gb300 import _abi as abi
    lib = abi.load()
    w = workloads.Workload("timeout", 1, 2, 256, 256, 64, 64, False, seed=5)
    t = workloads.make_dense(w, device="cuda")
    assert ea.attn_get_device_status() == 0
    o = torch.empty_like(t["q"])
    lse = torch.empty((1, 2, 256), dtype=torch.float32, device="cuda")
    p = abi.AttnFwdParams()
    ea._fill_fwd(p, t["q"], t["k"], t["v"], o, lse, ea._strides4, w.scale, False)
    p.batch, p.seqlen_q, p.seqlen_k = 1, 256, 256
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for rep in range(2):
        assert lib.attn_diag_wait_timeout(ctypes.byref(p), 1024, stream) == abi.ATTN_OK
        detail = ctypes.c_uint32(0)
        st = lib.attn_get_device_status(stream, ctypes.byref(detail))
        assert st == abi.ATTN_ERR_TIMEOUT, (rep, st, hex(detail.value))
        assert detail.value >> 24 == DEV_TIMEOUT_MBAR, hex(detail.value)
        assert detail.value & 0xFFF in SITES and (detail.value >> 12) & 0xFFF == 0, hex(detail.value)  # at step 0
        # reading the status cleared it
        assert lib.attn_get_device_status(stream, ctypes.byref(detail)) == abi.ATTN_OK and detail.value == 0
    # the context is intact: a normal forward runs and matches the oracle
    o2, lse2 = ea.attn_fwd(t["q"], t["k"], t["v"], softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == 0
    q, k, v = (t[n].cpu() for n in ("q", "k", "v"))
    for h in range(2):
        o_ref, l_ref = attention_fwd(q[0, :, h], k[0, :, h], v[0, :, h], w.scale, False)
        check_fwd(o2[0, :, h], lse2[0, h], o_ref, l_ref, f"after timeout h{h}")


def test_entry_points_leave_the_current_device_unchanged():
    """Every entry point runs on its data's device and restores the calling
    thread's current device. With a second GPU the data sits on the other
    device; with one GPU the check still covers every call."""
    import exact_attention_bf16_gb300 as ea
    n = torch.cuda.device_count()
    data_dev = 1 if n > 1 else 0
    torch.cuda.set_device(0)
    w = workloads.Workload("dev", 1, 2, 300, 300, 64, 64, True, seed=8)
    t = workloads.make_dense(w, device=f"cuda:{data_dev}")
    before = torch.cuda.current_device()
    o, lse = ea.attn_fwd(t["q"], t["k"], t["v"], causal=True, stream=torch.cuda.current_stream(data_dev))
    assert torch.cuda.current_device() == before
    ea.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=True, stream=torch.cuda.current_stream(data_dev))
    assert torch.cuda.current_device() == before
    ea.attn_exp2_eval(torch.zeros(16, device=f"cuda:{data_dev}"), stream=torch.cuda.current_stream(data_dev))
    assert torch.cuda.current_device() == before
    cnt, idx = ea.block_lists_from_mask(torch.ones((2, 3), dtype=torch.bool, device=f"cuda:{data_dev}"))
    ea.attn_fwd_block_sparse(t["q"], t["k"], t["v"], cnt, idx, stream=torch.cuda.current_stream(data_dev))
    assert torch.cuda.current_device() == before
    torch.cuda.synchronize(data_dev)


def test_block_lists_on_another_device_are_rejected():
    import exact_attention_bf16_gb300 as ea
    w = workloads.Workload("dev", 1, 1, 300, 300, 64, 64, False, seed=8)
    t = workloads.make_dense(w, device="cuda")
    cnt, idx = ea.block_lists_from_mask(torch.ones((2, 3), dtype=torch.bool))  # host tensors
    with pytest.raises(ValueError):
        ea.attn_fwd_block_sparse(t["q"], t["k"], t["v"], cnt, idx)
    # the C entry point itself refuses lists that are not on q's device
    from exact_attention_bf16_gb300 import _abi as abi
    lib = abi.load()
    o = torch.empty_like(t["q"])
    lse = torch.empty((1, 1, 300), dtype=torch.float32, device="cuda")
    p = abi.AttnFwdParams()
    ea._fill_fwd(p, t["q"], t["k"], t["v"], o, lse, ea._strides4, w.scale, False)
    p.batch, p.seqlen_q, p.seqlen_k = 1, 300, 300
    ws = torch.empty(lib.attn_fwd_workspace_size(ctypes.byref(p)), dtype=torch.uint8, device="cuda")
    st = lib.attn_fwd_block_sparse(ctypes.byref(p), ctypes.c_void_p(cnt.data_ptr()),
                                   ctypes.c_void_p(idx.data_ptr()), int(idx.shape[1]), 0, ctypes.c_void_p(ws.data_ptr()),
                                   ws.numel(), None)
    assert st == abi.ATTN_ERR_INVALID_ARG
