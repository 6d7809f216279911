"""Exhaustive check of the kernel's exp2 emulation (Cody-Waite split plus the
minimax cubic; wittx "FlashAttention-4", section 用软件"伪造"硬件指令) over
every fp32 input the softmax can feed it, x in [-127, 8].

Each input is compared with an fp64 exp2. Where the result is a normal fp32
number (x >= -126), the relative error must stay within the cubic's minimax
bound plus fp32 evaluation rounding. Below that, the result lies under 2^-126
and only an absolute bound applies. A strided sample is also checked on the CPU
against the oracle's own restatement of the same method, with coefficients
fitted independently."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

POLY_BOUND = 8.6e-5 + 3e-7   # minimax relative error of the cubic + fp32 evaluation
CHUNK = 1 << 27


def _bit_ranges():
    # fp32 bit patterns: +0 .. 8.0 and -0 .. -127.0 (sign-magnitude order)
    pos_hi = int(np.array(8.0, dtype=np.float32).view(np.int32))
    neg_hi = int(np.array(127.0, dtype=np.float32).view(np.int32))
    return [(0, pos_hi, 1.0), (0, neg_hi, -1.0)]


def test_exp2_emulation_exhaustive():
    import exact_attention_bf16_gb300 as ea
    from oracle import exp2_poly, fit_exp2_poly_remez
    c = fit_exp2_poly_remez()["c"]
    worst_rel, worst_abs_sub, count = 0.0, 0.0, 0
    sample_x, sample_y = [], []
    rng = np.random.default_rng(0)
    for lo, hi, sign in _bit_ranges():
        for start in range(lo, hi + 1, CHUNK):
            stop = min(start + CHUNK, hi + 1)
            bits = torch.arange(start, stop, dtype=torch.int64, device="cuda").to(torch.int32)
            x = bits.view(torch.float32)
            if sign < 0:
                x = -x
            yp, _ = ea.attn_exp2_eval(x)
            ref = torch.exp2(x.double())
            normal = x >= -126.0
            rel = ((yp.double() / ref) - 1.0).abs()
            worst_rel = max(worst_rel, rel[normal].max().item() if normal.any() else 0.0)
            if (~normal).any():
                worst_abs_sub = max(worst_abs_sub, (yp.double() - ref)[~normal].abs().max().item())
            assert torch.isfinite(yp).all()
            count += x.numel()
            idx = torch.from_numpy(rng.integers(0, x.numel(), 2048)).cuda()
            sample_x.append(x[idx].cpu().numpy())
            sample_y.append(yp[idx].cpu().numpy())
            del bits, x, yp, ref, rel, normal
    assert count > 2_000_000_000  # every fp32 value in [-127, 8]
    assert worst_rel < POLY_BOUND, worst_rel
    assert worst_abs_sub <= 2.0 ** -126
    # same method as the oracle's independent fit, on a random sample of the inputs
    xs = np.concatenate(sample_x).astype(np.float64)
    ys = np.concatenate(sample_y).astype(np.float64)
    keep = xs >= -126.0
    ref = exp2_poly(xs[keep], c)
    assert np.abs(ys[keep] / ref - 1.0).max() < 1e-6
