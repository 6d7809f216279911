"""The C-ABI library loads, exports every entry point include/attn.h declares,
agrees with the binding on struct layout, and rejects bad arguments before
touching the GPU. CPU only (no kernel is launched)."""
import ctypes
import os
import re
import subprocess

import pytest

import __graft_entry__


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    from exact_attention_bf16_gb300 import _abi as abi
    return abi.load()


@pytest.fixture(scope="module")
def _abi(lib):
    from exact_attention_bf16_gb300 import _abi as abi
    return abi


def declared_functions():
    import os
    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("attn_fwd", "attn_fwd_varlen", "attn_bwd", "attn_bwd_varlen", "attn_fwd_workspace_size",
                 "attn_bwd_workspace_size", "attn_get_device_status", "attn_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(lib, _abi):
    out = subprocess.run(["nm", "-D", "--defined-only", _abi.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(attn_[a-z0-9_]+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)


def test_struct_layout_and_version(lib, _abi):
    assert lib.attn_abi_version() == _abi.ABI_VERSION
    assert lib.attn_fwd_params_size() == ctypes.sizeof(_abi.AttnFwdParams)
    assert lib.attn_bwd_params_size() == ctypes.sizeof(_abi.AttnBwdParams)


def test_status_strings(lib, _abi):
    for code, name in _abi.STATUS.items():
        assert lib.attn_status_string(code).decode() == name


def _valid_fwd(_abi):
    p = _abi.AttnFwdParams()
    fake = 0x10000  # 16-byte aligned non-null dummy; never dereferenced by the checks below
    p.q = p.k = p.v = p.o = p.lse = fake
    for t in "qkvo":
        setattr(p, f"{t}_batch_stride", 128 * 4 * 64)
        setattr(p, f"{t}_row_stride", 4 * 64)
        setattr(p, f"{t}_head_stride", 64)
    p.batch, p.heads, p.seqlen_q, p.seqlen_k, p.d_qk, p.d_v = 1, 4, 128, 128, 64, 64
    p.softmax_scale = 0.125
    return p


INVALID, UNSUPPORTED = 1, 2


@pytest.mark.parametrize("mutate,expect", [
    (lambda p: setattr(p, "d_qk", 96), UNSUPPORTED),
    (lambda p: (setattr(p, "d_qk", 128), setattr(p, "d_v", 64)), UNSUPPORTED),
    (lambda p: setattr(p, "d_qk", 0), INVALID),
    (lambda p: setattr(p, "softmax_scale", 0.0), INVALID),
    (lambda p: setattr(p, "softmax_scale", float("nan")), INVALID),
    (lambda p: setattr(p, "softmax_scale", -1.0), INVALID),
    (lambda p: setattr(p, "heads", 0), INVALID),
    (lambda p: setattr(p, "batch", 0), INVALID),
    (lambda p: setattr(p, "seqlen_q", -1), INVALID),
    (lambda p: setattr(p, "q", 0x10008), INVALID),       # misaligned
    (lambda p: setattr(p, "k", None), INVALID),           # null
    (lambda p: setattr(p, "v_row_stride", 4 * 64 + 4), INVALID),  # not a multiple of 8
    (lambda p: setattr(p, "lse", 0x10002), INVALID),
    (lambda p: setattr(p, "cu_seqlens_q", 0x10000), INVALID),  # dense call with offsets
    (lambda p: setattr(p, "exp2_emu_period", 3), INVALID),      # only 0, 4, 8 are built
    (lambda p: setattr(p, "exp2_emu_period", -8), INVALID),
])
def test_fwd_rejects_bad_arguments_without_a_gpu(lib, _abi, mutate, expect):
    p = _valid_fwd(_abi)
    mutate(p)
    assert lib.attn_fwd(ctypes.byref(p), None, 0, None) == expect


def test_varlen_requires_offsets(lib, _abi):
    p = _valid_fwd(_abi)
    p.num_seqs, p.total_q, p.total_k, p.max_seqlen_q, p.max_seqlen_k = 1, 128, 128, 128, 128
    assert lib.attn_fwd_varlen(ctypes.byref(p), None, 0, None) == _abi.ATTN_ERR_INVALID_ARG
    p.cu_seqlens_q = p.cu_seqlens_k = 0x10000
    p.max_seqlen_q = 129  # longer than the packed batch
    assert lib.attn_fwd_varlen(ctypes.byref(p), None, 0, None) == _abi.ATTN_ERR_INVALID_ARG


def test_null_params(lib, _abi):
    assert lib.attn_fwd(None, None, 0, None) == _abi.ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd(None, None, 0, None) == _abi.ATTN_ERR_INVALID_ARG
    assert lib.attn_exp2_eval(None, None, None, 4, None) == _abi.ATTN_ERR_INVALID_ARG


def test_product_path_does_not_import_the_oracle(_abi):
    pkg = os.path.dirname(_abi.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(root, f), encoding="utf-8").read()
                assert "oracle" not in src.replace("CPU oracle", ""), f


def _valid_sparse_args():
    return 0x20000, 0x30000, 3  # kv_count, kv_index (dummy aligned device addresses), max_kv


@pytest.mark.parametrize("mutate,expect", [
    (lambda p, a: (p, (a[0], a[1], -1)), INVALID),                   # negative max_kv
    (lambda p, a: (p, (None, a[1], a[2])), INVALID),                 # no counts
    (lambda p, a: (p, (a[0], None, a[2])), INVALID),                 # no index array with max_kv > 0
    (lambda p, a: (p, (a[0] + 2, a[1], a[2])), INVALID),             # misaligned counts
    (lambda p, a: (p, (a[0], a[1] + 1, a[2])), INVALID),             # misaligned indices
    (lambda p, a: (p, (a[0], a[1], 0x7fffffff)), INVALID),           # n_qblk * max_kv overflows int32
    (lambda p, a: (setattr(p, "exp2_emu_period", 4) or p, a), INVALID),  # exp2 emulation not built here
    (lambda p, a: (setattr(p, "cu_seqlens_q", 0x10000) or p, a), INVALID),  # dense layout only
    (lambda p, a: (setattr(p, "d_qk", 96) or p, a), UNSUPPORTED),
])
def test_block_sparse_rejects_bad_arguments_without_a_gpu(lib, _abi, mutate, expect):
    p = _valid_fwd(_abi)
    p.seqlen_q = 600  # three query blocks of 256 rows
    p, (cnt, idx, max_kv) = mutate(p, _valid_sparse_args())
    assert lib.attn_fwd_block_sparse(ctypes.byref(p), cnt, idx, max_kv, 0, None, 0, None) == expect


@pytest.mark.parametrize("mutate,expect", [
    (lambda p, a: (p, (a[0], a[1], -1)), INVALID),
    (lambda p, a: (p, (None, a[1], a[2])), INVALID),
    (lambda p, a: (p, (a[0], None, a[2])), INVALID),
    (lambda p, a: (p, (a[0] + 2, a[1], a[2])), INVALID),
    (lambda p, a: (setattr(p.fwd, "cu_seqlens_q", 0x10000) or p, a), INVALID),
    (lambda p, a: (setattr(p.fwd, "d_qk", 96) or p, a), UNSUPPORTED),
])
def test_block_sparse_backward_rejects_bad_arguments_without_a_gpu(lib, _abi, mutate, expect):
    p = _abi.AttnBwdParams()
    p.fwd = _valid_fwd(_abi)
    p.fwd.seqlen_q = 600
    p, (cnt, idx, max_kv) = mutate(p, _valid_sparse_args())
    assert lib.attn_bwd_block_sparse(ctypes.byref(p), cnt, idx, max_kv, 0, None, 0, None) == expect


def test_block_sparse_backward_workspace_size(lib, _abi):
    p = _abi.AttnBwdParams()
    p.fwd = _valid_fwd(_abi)
    p.fwd.seqlen_q, p.fwd.seqlen_k = 600, 1000  # 3 query blocks of 256, 8 key blocks of 128
    dense = lib.attn_bwd_workspace_size(ctypes.byref(p))
    r256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    sparse = lib.attn_bwd_block_sparse_workspace_size(ctypes.byref(p), 0)
    assert sparse == dense + r256(8 * 4) + r256(8 * 3 * 4)  # q_count[8] and q_index[8][3] after the D vector
    per_head = lib.attn_bwd_block_sparse_workspace_size(ctypes.byref(p), 1)  # B1 H4: four sets
    assert per_head == dense + r256(4 * 8 * 4) + r256(4 * 8 * 3 * 4)
    assert lib.attn_bwd_block_sparse_workspace_size(ctypes.byref(p), 2) == 0
    p.fwd.cu_seqlens_q = 0x10000
    assert lib.attn_bwd_block_sparse_workspace_size(ctypes.byref(p), 0) == 0  # dense layout only


@pytest.mark.parametrize("lists_per_head,max_kv,expect", [
    (2, 3, INVALID),                 # neither shared nor per (batch, head)
    (-1, 3, INVALID),
    (1, 0x7fffffff // 12 + 1, INVALID),  # B1 H4 x 3 query blocks x max_kv overflows int32
])
def test_block_lists_per_head_rejects_bad_arguments_without_a_gpu(lib, _abi, lists_per_head, max_kv, expect):
    p = _valid_fwd(_abi)
    p.seqlen_q = 600
    cnt, idx, _ = _valid_sparse_args()
    assert lib.attn_fwd_block_sparse(ctypes.byref(p), cnt, idx, max_kv, lists_per_head, None, 0, None) == expect
    b = _abi.AttnBwdParams()
    b.fwd = p
    b.dout = b.dq = b.dk = b.dv = 0x10000
    for t in ("do", "dq", "dk", "dv"):
        setattr(b, f"{t}_batch_stride", 128 * 4 * 64)
        setattr(b, f"{t}_row_stride", 4 * 64)
        setattr(b, f"{t}_head_stride", 64)
    assert lib.attn_bwd_block_sparse(ctypes.byref(b), cnt, idx, max_kv, lists_per_head, None, 0, None) == expect


@pytest.mark.parametrize("mutate,expect", [
    (lambda p: setattr(p, "score_mod", 3), INVALID),                              # unknown modification
    (lambda p: setattr(p, "score_mod", -1), INVALID),
    (lambda p: (setattr(p, "score_mod", 1), setattr(p, "softcap", 0.0)), INVALID),   # cap must be > 0
    (lambda p: (setattr(p, "score_mod", 1), setattr(p, "softcap", -2.0)), INVALID),
    (lambda p: (setattr(p, "score_mod", 1), setattr(p, "softcap", float("inf"))), INVALID),
    (lambda p: (setattr(p, "score_mod", 1), setattr(p, "softcap", float("nan"))), INVALID),
    (lambda p: (setattr(p, "score_mod", 1), setattr(p, "softcap", 3e38)), INVALID),   # cap / scale overflows
    (lambda p: setattr(p, "score_mod", 2), INVALID),                              # ALiBi without slopes
    (lambda p: (setattr(p, "score_mod", 2), setattr(p, "alibi_slopes", 0x10002)), INVALID),  # misaligned
    (lambda p: (setattr(p, "score_mod", 1), setattr(p, "softcap", 30.0),
                setattr(p, "exp2_emu_period", 8)), UNSUPPORTED),                  # no emulated exp2 with a mod
])
def test_score_mod_rejects_bad_arguments_without_a_gpu(lib, _abi, mutate, expect):
    p = _valid_fwd(_abi)
    mutate(p)
    assert lib.attn_fwd(ctypes.byref(p), None, 0, None) == expect


def test_score_mod_rejected_with_the_two_sm_backward(lib, _abi):
    p = _abi.AttnBwdParams()
    p.fwd = _valid_fwd(_abi)
    p.fwd.d_qk = p.fwd.d_v = 128
    p.fwd.score_mod, p.fwd.softcap = 1, 30.0
    p.dout = p.dq = p.dk = p.dv = 0x10000
    for t in ("do", "dq", "dk", "dv"):
        setattr(p, f"{t}_batch_stride", 128 * 4 * 128)
        setattr(p, f"{t}_row_stride", 4 * 128)
        setattr(p, f"{t}_head_stride", 128)
    p.cta_pair = 1
    assert lib.attn_bwd(ctypes.byref(p), None, 0, None) == UNSUPPORTED


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++17")])
def test_header_compiles_as_c_and_cpp(lang, std):
    import shutil
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    src = '#include "attn.h"\nint main(void) { return (int)sizeof(attn_fwd_params) == 0; }\n'
    r = subprocess.run([cc, "-x", lang, std, "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I", inc, "-"],
                       input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


@pytest.mark.parametrize("mutate,limit", [
    (lambda p: None, 0),                                     # no poll limit
    (lambda p: None, (1 << 20) + 1),                         # limit above 2^20
    (lambda p: (setattr(p, "d_qk", 128), setattr(p, "d_v", 128)), 1024),  # built for d = 64 only
    (lambda p: setattr(p, "exp2_emu_period", 8), 1024),
    (lambda p: setattr(p, "seqlen_k", 0), 1024),            # the kernel would not launch
    (lambda p: setattr(p, "cu_seqlens_q", 0x10000), 1024),  # dense layout only
])
def test_diag_wait_timeout_rejects_bad_arguments_without_a_gpu(lib, _abi, mutate, limit):
    p = _valid_fwd(_abi)
    mutate(p)
    assert lib.attn_diag_wait_timeout(ctypes.byref(p), limit, None) == _abi.ATTN_ERR_INVALID_ARG


def test_bwd_workspace_size_is_zero_for_negative_shapes(lib, _abi):
    p = _abi.AttnBwdParams()
    p.fwd = _valid_fwd(_abi)
    assert lib.attn_bwd_workspace_size(ctypes.byref(p)) >= 4 * 4 * 128
    for field, value in (("seqlen_q", -1), ("heads", -3), ("batch", -2)):
        p.fwd = _valid_fwd(_abi)
        setattr(p.fwd, field, value)
        assert lib.attn_bwd_workspace_size(ctypes.byref(p)) == 0, field


@pytest.mark.parametrize("field,value", [("seqlen_q", -1), ("heads", -3), ("heads", 0), ("batch", -2),
                                         ("seqlen_k", -5)])
def test_noalloc_rejects_negative_shapes_as_invalid(lib, _abi, field, value):
    """A negative size is a bad argument (ATTN_ERR_INVALID_ARG), not a problem
    too large for the fixed scratch (ATTN_ERR_WORKSPACE); checked before any
    device call."""
    p = _abi.AttnBwdParams()
    p.fwd = _valid_fwd(_abi)
    setattr(p.fwd, field, value)
    assert lib.attn_bwd_noalloc(ctypes.byref(p), None) == _abi.ATTN_ERR_INVALID_ARG


def test_cta_pair_backward_only_for_d128_without_lists(lib, _abi):
    """The two-SM dK/dV kernel exists for d_qk = d_v = 128 without block lists;
    asking for it elsewhere is ATTN_ERR_UNSUPPORTED before any device call."""
    p = _abi.AttnBwdParams()
    p.fwd = _valid_fwd(_abi)  # d = 64
    p.dout = p.dq = p.dk = p.dv = 0x10000
    for t in ("do", "dq", "dk", "dv"):
        setattr(p, f"{t}_batch_stride", 128 * 4 * 64)
        setattr(p, f"{t}_row_stride", 4 * 64)
        setattr(p, f"{t}_head_stride", 64)
    p.cta_pair = 1
    assert lib.attn_bwd(ctypes.byref(p), None, 0, None) == _abi.ATTN_ERR_UNSUPPORTED
    p.fwd.d_qk, p.fwd.d_v = 192, 128
    assert lib.attn_bwd(ctypes.byref(p), None, 0, None) == _abi.ATTN_ERR_UNSUPPORTED
    p.fwd.d_qk, p.fwd.d_v = 128, 128
    cnt, idx, max_kv = _valid_sparse_args()
    assert lib.attn_bwd_block_sparse(ctypes.byref(p), cnt, idx, max_kv, 0, None, 0, None) in (
        _abi.ATTN_ERR_UNSUPPORTED, _abi.ATTN_ERR_INVALID_ARG)


def test_fwd_workspace_size_holds_the_fp16_copy_of_v(lib, _abi):
    p = _valid_fwd(_abi)  # B1 H4 Nk128 d_v 64
    assert lib.attn_fwd_workspace_size(ctypes.byref(p)) == 256 + 128 * 4 * 64 * 2
    p.seqlen_k = 0
    assert lib.attn_fwd_workspace_size(ctypes.byref(p)) == 0
    p.seqlen_k, p.heads = 128, -1
    assert lib.attn_fwd_workspace_size(ctypes.byref(p)) == 0
    p = _valid_fwd(_abi)
    p.cu_seqlens_q = p.cu_seqlens_k = 0x10000
    p.num_seqs, p.total_q, p.total_k, p.max_seqlen_q, p.max_seqlen_k = 2, 300, 301, 200, 200
    # packed variable length adds the tile list: heads * (total_q // 256 + sequences)
    # entries of 32 bytes, then 8 bytes per sequence of scratch, each rounded to 256
    r256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    v16 = r256(301 * 4 * 64 * 2)
    assert lib.attn_fwd_workspace_size(ctypes.byref(p)) == 256 + v16 + r256(32 * 4 * (300 // 256 + 2)) + r256(8 * 2)
    p.max_seqlen_q = 2047 * 256 + 1  # a sequence may exceed the list's block limit: no list
    p.total_q = p.total_k = 2047 * 256 + 1
    assert lib.attn_fwd_workspace_size(ctypes.byref(p)) == 256 + r256(p.total_k * 4 * 64 * 2)


def test_bwd_workspace_size_holds_the_tile_lists(lib, _abi):
    """Packed variable length: D (4 bytes per query row and head), the dK/dV list
    (128 keys per block), the dQ list (128 queries per block), the scratch."""
    r256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    p = _abi.AttnBwdParams()
    p.fwd = _valid_fwd(_abi)
    f = p.fwd
    f.cu_seqlens_q = f.cu_seqlens_k = 0x10000
    f.num_seqs, f.total_q, f.total_k, f.max_seqlen_q, f.max_seqlen_k = 2, 300, 301, 200, 200
    d = r256(4 * 4 * 300)
    kv = r256(32 * 4 * (301 // 128 + 2))
    q = r256(32 * 4 * (300 // 128 + 2))
    assert lib.attn_bwd_workspace_size(ctypes.byref(p)) == d + kv + q + r256(8 * 2)
    p.cta_pair = 1  # the two-SM dK/dV kernel takes no list
    assert lib.attn_bwd_workspace_size(ctypes.byref(p)) == d + q + r256(8 * 2)
    p.cta_pair = 0
    f.cu_seqlens_q = f.cu_seqlens_k = 0  # dense: D only
    assert lib.attn_bwd_workspace_size(ctypes.byref(p)) == r256(4 * 4 * 128)


def _valid_fwd_e4m3(_abi):
    p = _valid_fwd(_abi)
    p.d_qk = p.d_v = 128
    for t in "qkvo":
        setattr(p, f"{t}_batch_stride", 128 * 4 * 128)
        setattr(p, f"{t}_row_stride", 4 * 128)
        setattr(p, f"{t}_head_stride", 128)
    p.input_dtype, p.q_descale, p.k_descale, p.v_descale = 1, 0.01, 0.02, 0.03
    return p


@pytest.mark.parametrize("mutate,expect", [
    (lambda p: setattr(p, "input_dtype", 2), INVALID),                   # unknown element type
    (lambda p: setattr(p, "q_descale", 0.0), INVALID),                   # descales finite and > 0
    (lambda p: setattr(p, "k_descale", -1.0), INVALID),
    (lambda p: setattr(p, "v_descale", float("nan")), INVALID),
    (lambda p: setattr(p, "v_descale", float("inf")), INVALID),
    (lambda p: setattr(p, "q_row_stride", 4 * 128 + 8), INVALID),        # byte strides: multiples of 16
    (lambda p: setattr(p, "k_head_stride", 136), INVALID),
    (lambda p: (setattr(p, "d_qk", 64), setattr(p, "d_v", 64)), UNSUPPORTED),  # d = 128 only
    (lambda p: setattr(p, "exp2_emu_period", 8), UNSUPPORTED),
    (lambda p: (setattr(p, "score_mod", 1), setattr(p, "softcap", 30.0)), UNSUPPORTED),
])
def test_e4m3_forward_rejects_bad_arguments_without_a_gpu(lib, _abi, mutate, expect):
    p = _valid_fwd_e4m3(_abi)
    mutate(p)
    assert lib.attn_fwd(ctypes.byref(p), None, 0, None) == expect


def test_e4m3_is_forward_only(lib, _abi):
    p = _valid_fwd_e4m3(_abi)
    p.seqlen_q = 600
    cnt, idx, max_kv = _valid_sparse_args()
    assert lib.attn_fwd_block_sparse(ctypes.byref(p), cnt, idx, max_kv, 0, None, 0, None) == UNSUPPORTED
    b = _abi.AttnBwdParams()
    b.fwd = _valid_fwd_e4m3(_abi)
    b.dout = b.dq = b.dk = b.dv = 0x10000
    for t in ("do", "dq", "dk", "dv"):
        setattr(b, f"{t}_batch_stride", 128 * 4 * 128)
        setattr(b, f"{t}_row_stride", 4 * 128)
        setattr(b, f"{t}_head_stride", 128)
    assert lib.attn_bwd(ctypes.byref(b), None, 0, None) == UNSUPPORTED
    b.fwd.input_dtype = 2
    assert lib.attn_bwd(ctypes.byref(b), None, 0, None) == INVALID


def test_single_pass_workspace_and_rejections_without_a_gpu(lib, _abi):
    r256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    p = _abi.AttnBwdParams()
    p.fwd = _valid_fwd(_abi)  # B1 H4 N128 d64
    p.dout = p.dq = p.dk = p.dv = 0x10000
    for t in ("do", "dq", "dk", "dv"):
        setattr(p, f"{t}_batch_stride", 128 * 4 * 64)
        setattr(p, f"{t}_row_stride", 4 * 64)
        setattr(p, f"{t}_head_stride", 64)
    base = lib.attn_bwd_workspace_size(ctypes.byref(p))
    p.single_pass = 1
    assert lib.attn_bwd_workspace_size(ctypes.byref(p)) == base + r256(4 * 128 * 64 * 4)  # the fp32 dQ
    p.deterministic = 1  # plus one semaphore per (batch, head, 64-row tile)
    assert lib.attn_bwd_workspace_size(ctypes.byref(p)) == base + r256(4 * 128 * 64 * 4) + r256(1 * 4 * 2 * 4)
    p.cta_pair = 1
    assert lib.attn_bwd(ctypes.byref(p), None, 0, None) == UNSUPPORTED
    p.cta_pair = 0
    p.fwd.score_mod, p.fwd.softcap = 1, 30.0
    assert lib.attn_bwd(ctypes.byref(p), None, 0, None) == UNSUPPORTED
    p.fwd.score_mod = 0
    p.fwd.d_qk = p.fwd.d_v = 128
    assert lib.attn_bwd(ctypes.byref(p), None, 0, None) == UNSUPPORTED


@pytest.mark.parametrize("mutate,expect", [
    (lambda p: (setattr(p, "d_qk", 64), setattr(p, "d_v", 64)), UNSUPPORTED),  # d = 128 only
    (lambda p: setattr(p, "exp2_emu_period", 4), UNSUPPORTED),
    (lambda p: (setattr(p, "score_mod", 2), setattr(p, "alibi_slopes", 0x10000)), UNSUPPORTED),
    (lambda p: (setattr(p, "input_dtype", 1), setattr(p, "q_descale", 1.0), setattr(p, "k_descale", 1.0),
                setattr(p, "v_descale", 1.0)), UNSUPPORTED),
])
def test_pair_forward_rejects_without_a_gpu(lib, _abi, mutate, expect):
    p = _valid_fwd(_abi)
    p.d_qk = p.d_v = 128
    for t in "qkvo":
        setattr(p, f"{t}_batch_stride", 128 * 4 * 128)
        setattr(p, f"{t}_row_stride", 4 * 128)
        setattr(p, f"{t}_head_stride", 128)
    p.cta_pair = 1
    mutate(p)
    assert lib.attn_fwd(ctypes.byref(p), None, 0, None) == expect


def test_pair_forward_takes_no_tile_list(lib, _abi):
    p = _valid_fwd(_abi)
    p.cu_seqlens_q = p.cu_seqlens_k = 0x10000
    p.num_seqs, p.total_q, p.total_k, p.max_seqlen_q, p.max_seqlen_k = 2, 300, 301, 200, 200
    with_list = lib.attn_fwd_workspace_size(ctypes.byref(p))
    p.cta_pair = 1
    assert lib.attn_fwd_workspace_size(ctypes.byref(p)) == 256 + (301 * 4 * 64 * 2 + 255) // 256 * 256 < with_list
