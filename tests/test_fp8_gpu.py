"""Forward with FP8 E4M3 inputs through the C ABI against the fp64 oracle on the
decoded values times their descale factors, element by element, dense (both
masks, Nq = Nk and Nq != Nk, ragged tails) and packed variable length."""
import numpy as np
import pytest
import torch

import workloads
from oracle import attention_fwd, e4m3_decode
from parity import check_fwd

pytestmark = pytest.mark.gpu


def quantise(x: torch.Tensor):
    """E4M3 codes of x / descale with descale = max|x| / 448 (the whole range used), and the descale."""
    descale = float(x.abs().max()) / 448.0
    return (x / descale).to(torch.float8_e4m3fn), descale


def decoded(t: torch.Tensor, descale: float) -> np.ndarray:
    return e4m3_decode(t.cpu().view(torch.uint8).numpy()) * descale


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk", [(300, 300), (200, 520), (1100, 700)])
def test_dense_e4m3_forward(causal, nq, nk):
    import exact_attention_bf16_gb300 as ea
    g = torch.Generator(device="cuda").manual_seed(nq + nk + causal)
    B, H, d = 2, 3, 128
    q32, k32, v32 = (torch.randn((B, n, H, d), generator=g, device="cuda") for n in (nq, nk, nk))
    (q, qd), (k, kd), (v, vd) = quantise(q32), quantise(k32), quantise(1.5 * v32)
    o, lse = ea.attn_fwd(q, k, v, causal=causal, q_descale=qd, k_descale=kd, v_descale=vd)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == 0
    qq, kk, vv = decoded(q, qd), decoded(k, kd), decoded(v, vd)
    for b in range(B):
        for h in range(H):
            oo, ll = attention_fwd(qq[b, :, h], kk[b, :, h], vv[b, :, h], d ** -0.5, causal)
            check_fwd(o[b, :, h], lse[b, h], oo, ll, f"b{b} h{h}")


def test_varlen_e4m3_forward():
    import exact_attention_bf16_gb300 as ea
    ql = [5, 300, 0, 257, 1000, 1]
    kl = [7, 260, 3, 257, 900, 1]
    H, d = 4, 128
    g = torch.Generator(device="cuda").manual_seed(77)
    q32, k32, v32 = (torch.randn((sum(n), H, d), generator=g, device="cuda") for n in (ql, kl, kl))
    (q, qd), (k, kd), (v, vd) = quantise(q32), quantise(k32), quantise(v32)
    cq, ck = workloads.cu_seqlens_of(ql).cuda(), workloads.cu_seqlens_of(kl).cuda()
    o, lse = ea.attn_fwd_varlen(q, k, v, cq, ck, max(ql), max(kl), causal=True, q_descale=qd, k_descale=kd,
                                v_descale=vd)
    torch.cuda.synchronize()
    assert ea.attn_get_device_status() == 0
    qq, kk, vv = decoded(q, qd), decoded(k, kd), decoded(v, vd)
    # The whole packed output at once: the mean bound is over the output, and a
    # one-key sequence's row alone is just V's row rounded to bf16.
    o_ref = np.zeros((sum(ql), H, d))
    lse_ref = np.full((H, sum(ql)), -np.inf)
    cqh, ckh = cq.cpu().numpy(), ck.cpu().numpy()
    for s in range(len(ql)):
        a, b, c, e = int(cqh[s]), int(cqh[s + 1]), int(ckh[s]), int(ckh[s + 1])
        for h in range(H):
            if b > a and e > c:
                o_ref[a:b, h], lse_ref[h, a:b] = attention_fwd(qq[a:b, h], kk[c:e, h], vv[c:e, h], d ** -0.5, True)
    check_fwd(o, lse, o_ref, lse_ref, "varlen e4m3")


def test_e4m3_rejections_on_the_gpu():
    import exact_attention_bf16_gb300 as ea
    x64 = torch.zeros((1, 128, 2, 64), device="cuda").to(torch.float8_e4m3fn)
    with pytest.raises(ea.AttnError):  # E4M3 is built for d = 128 only
        ea.attn_fwd(x64, x64, x64)
    x = torch.zeros((1, 128, 2, 128), device="cuda").to(torch.float8_e4m3fn)
    with pytest.raises(ea.AttnError):  # no score modification with E4M3
        ea.attn_fwd(x, x, x, softcap=2.0)
    with pytest.raises(ea.AttnError):  # descales must be > 0
        ea.attn_fwd(x, x, x, q_descale=0.0)
    with pytest.raises(TypeError):  # mixed element types
        ea.attn_fwd(x, x.to(torch.bfloat16), x)
