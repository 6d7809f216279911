"""The split-key plan of the dense forward, seen through attn_fwd_workspace_size
(CPU only, nothing is launched). A dense bf16 forward with d_qk = d_v = 64 or
128, no score modification, no exp2 emulation and no CTA pairs splits its keys
when its (256-row block, head, batch) grid has at most 74 CTAs and its keys
span at least 16 blocks of 128: into s = min(148 // ctas, blocks // 8, 32)
ranges of ceil(blocks / s) blocks (then as many ranges as that needs), so that
the split grid stays within one wave. The
workspace then holds an fp32 O row and an fp32 LSE per range and query row
after the range flag and the fp16 copy of V, each part rounded up to 256 bytes."""
import ctypes
import math

import pytest

import __graft_entry__


@pytest.fixture(scope="module")
def lib_abi():
    __graft_entry__.build()
    from exact_attention_bf16_gb300 import _abi as abi
    return abi.load(), abi


def r256(n):
    return (n + 255) // 256 * 256


def expected_splits(B, H, nq, nk):
    ctas = B * H * math.ceil(nq / 256)
    blocks = math.ceil(nk / 128)
    if ctas * 2 > 148 or blocks < 16:
        return 1
    s = min(148 // ctas, blocks // 8, 32)
    if s < 2:
        return 1
    per = math.ceil(blocks / s)
    return math.ceil(blocks / per)


def workspace(lib, abi, B, H, nq, nk, d, **kw):
    p = abi.AttnFwdParams()
    p.batch, p.heads, p.seqlen_q, p.seqlen_k, p.d_qk, p.d_v = B, H, nq, nk, d, d
    fields = {f[0] for f in abi.AttnFwdParams._fields_}
    for k, v in kw.items():
        assert k in fields, k  # ctypes would take an unknown name silently
        setattr(p, k, v)
    return lib.attn_fwd_workspace_size(ctypes.byref(p))


@pytest.mark.parametrize("B,H,nq,nk,d", [
    (1, 16, 512, 32768, 128),   # 32 CTAs, 256 key blocks: 4 ranges of 64 (128 CTAs)
    (1, 16, 512, 32768, 64),
    (2, 8, 256, 16384, 128),    # 16 CTAs: 9 ranges
    (1, 1, 128, 4096, 128),     # 1 CTA, 32 blocks: 4 ranges of 8
    (2, 2, 200, 4000, 128),     # the GPU test's shape: 4 ranges
    (1, 1, 3000, 3000, 128),    # 12 CTAs, 24 blocks: 3 ranges
    (1, 1, 128, 1024, 128),     # 8 key blocks: no split
    (4, 16, 8192, 8192, 128),   # 2,048 CTAs: no split
    (1, 37, 256, 65536, 128),   # 37 CTAs (at most 74): 4 ranges (148 CTAs)
    (1, 75, 256, 65536, 128),   # 75 CTAs: no split
])
def test_dense_split_plan(lib_abi, B, H, nq, nk, d):
    lib, abi = lib_abi
    s = expected_splits(B, H, nq, nk)
    v16 = r256(B * nk * H * d * 2)
    parts = 0 if s == 1 else r256(s * B * H * nq * d * 4) + r256(s * B * H * nq * 4)
    assert workspace(lib, abi, B, H, nq, nk, d) == 256 + v16 + parts


@pytest.mark.parametrize("kw", [
    {"exp2_emu_period": 8},
    {"score_mod": 1, "softcap": 30.0},
    {"cta_pair": 1},
])
def test_no_split_for_other_variants(lib_abi, kw):
    lib, abi = lib_abi
    B, H, nq, nk, d = 1, 16, 512, 32768, 128
    assert workspace(lib, abi, B, H, nq, nk, d, **kw) == 256 + r256(B * nk * H * d * 2)


def test_no_split_at_d192(lib_abi):
    lib, abi = lib_abi
    p = abi.AttnFwdParams()
    p.batch, p.heads, p.seqlen_q, p.seqlen_k, p.d_qk, p.d_v = 1, 16, 512, 32768, 192, 128
    assert lib.attn_fwd_workspace_size(ctypes.byref(p)) == 256 + r256(32768 * 16 * 128 * 2)


# The dense two-kernel backward splits the dQ kernel's keys by the same rule over
# its (128-row query tile, head, batch) grid. Its workspace is the D vector
# (4 bytes per (batch, head, query row), rounded up to 256), then, when it
# splits, each range's fp32 dQ partial: s x batch x heads x seqlen_q x d_qk x 4
# bytes, rounded up to 256. d_v only decides which head sizes are supported.
def expected_dq_splits(B, H, nq, nk):
    ctas = B * H * math.ceil(nq / 128)
    blocks = math.ceil(nk / 128)
    if ctas * 2 > 148 or blocks < 16:
        return 1
    s = min(148 // ctas, blocks // 8, 32)
    if s < 2:
        return 1
    per = math.ceil(blocks / s)
    return math.ceil(blocks / per)


def bwd_workspace(lib, abi, B, H, nq, nk, dqk, dv, **kw):
    p = abi.AttnBwdParams()
    f = p.fwd
    f.batch, f.heads, f.seqlen_q, f.seqlen_k, f.d_qk, f.d_v = B, H, nq, nk, dqk, dv
    names = {x[0] for x in abi.AttnBwdParams._fields_}
    for k, v in kw.items():
        assert k in names, k
        setattr(p, k, v)
    return lib.attn_bwd_workspace_size(ctypes.byref(p))


@pytest.mark.parametrize("B,H,nq,nk,dqk,dv,splits", [
    (1, 16, 512, 32768, 128, 128, 2),   # 64 tiles, 256 key blocks: 2 ranges of 128 (128 CTAs)
    (1, 16, 512, 32768, 64, 64, 2),
    (1, 16, 512, 32768, 192, 128, 2),
    (2, 8, 256, 16384, 128, 128, 4),    # 32 tiles, 128 blocks: 4 ranges of 32
    (1, 2, 300, 2500, 128, 128, 2),     # 6 tiles, 20 blocks: 2 ranges of 10
    (1, 1, 4096, 4096, 128, 128, 4),    # 32 tiles, 32 blocks: 4 ranges of 8
    (1, 1, 128, 4096, 64, 64, 4),       # 1 tile, 32 blocks: 4 ranges of 8
    (1, 1, 128, 1920, 128, 128, 1),     # 15 key blocks: no split
    (1, 75, 128, 65536, 128, 128, 1),   # 75 tiles: no split
    (4, 16, 8192, 8192, 128, 128, 1),   # 4,096 tiles: no split
])
def test_dense_backward_dq_split_plan(lib_abi, B, H, nq, nk, dqk, dv, splits):
    lib, abi = lib_abi
    s = expected_dq_splits(B, H, nq, nk)
    assert s == splits
    parts = 0 if s == 1 else r256(s * B * H * nq * dqk * 4)
    assert bwd_workspace(lib, abi, B, H, nq, nk, dqk, dv) == r256(4 * B * H * nq) + parts


def test_backward_dq_split_not_in_single_pass(lib_abi):
    """The single-pass backward reduces dQ in its own fp32 buffer and never splits."""
    lib, abi = lib_abi
    B, H, nq, nk = 1, 16, 512, 32768
    assert bwd_workspace(lib, abi, B, H, nq, nk, 64, 64, single_pass=1) == r256(4 * B * H * nq) + r256(4 * B * H * nq * 64)
