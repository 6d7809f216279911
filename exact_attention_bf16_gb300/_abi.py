"""ctypes view of include/attn.h: the shared library, its status codes and the
two parameter structs. Loading fails loudly if the library is missing; there is
no fallback implementation."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libattn_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(HERE), "include", "attn.h")

ABI_VERSION = 5
BWD_NOALLOC_SCRATCH_BYTES = 8 << 20  # ATTN_BWD_NOALLOC_SCRATCH_BYTES

STATUS = {
    0: "ATTN_OK",
    1: "ATTN_ERR_INVALID_ARG",
    2: "ATTN_ERR_UNSUPPORTED",
    3: "ATTN_ERR_CUDA",
    4: "ATTN_ERR_TIMEOUT",
    5: "ATTN_ERR_WORKSPACE",
}
ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT, ATTN_ERR_WORKSPACE = range(6)
SCORE_NONE, SCORE_SOFTCAP, SCORE_ALIBI = range(3)  # attn_score_mod_t
INPUT_BF16, INPUT_E4M3 = range(2)  # attn_input_dtype_t

c_i32, c_i64, c_f32, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p


class AttnFwdParams(ctypes.Structure):
    _fields_ = [
        ("q", c_vp), ("k", c_vp), ("v", c_vp), ("o", c_vp), ("lse", c_vp),
        ("q_batch_stride", c_i64), ("q_row_stride", c_i64), ("q_head_stride", c_i64),
        ("k_batch_stride", c_i64), ("k_row_stride", c_i64), ("k_head_stride", c_i64),
        ("v_batch_stride", c_i64), ("v_row_stride", c_i64), ("v_head_stride", c_i64),
        ("o_batch_stride", c_i64), ("o_row_stride", c_i64), ("o_head_stride", c_i64),
        ("batch", c_i32), ("heads", c_i32), ("seqlen_q", c_i32), ("seqlen_k", c_i32),
        ("d_qk", c_i32), ("d_v", c_i32),
        ("cu_seqlens_q", c_vp), ("cu_seqlens_k", c_vp),
        ("num_seqs", c_i32), ("max_seqlen_q", c_i32), ("max_seqlen_k", c_i32),
        ("total_q", c_i32), ("total_k", c_i32),
        ("softmax_scale", c_f32), ("causal", c_i32), ("exp2_emu_period", c_i32),
        ("rescale_stats", c_vp),
        ("score_mod", c_i32), ("softcap", ctypes.c_float), ("alibi_slopes", c_vp),
        ("input_dtype", c_i32), ("q_descale", ctypes.c_float), ("k_descale", ctypes.c_float),
        ("v_descale", ctypes.c_float), ("cta_pair", c_i32),
    ]


class AttnBwdParams(ctypes.Structure):
    _fields_ = [
        ("fwd", AttnFwdParams),
        ("dout", c_vp), ("dq", c_vp), ("dk", c_vp), ("dv", c_vp),
        ("do_batch_stride", c_i64), ("do_row_stride", c_i64), ("do_head_stride", c_i64),
        ("dq_batch_stride", c_i64), ("dq_row_stride", c_i64), ("dq_head_stride", c_i64),
        ("dk_batch_stride", c_i64), ("dk_row_stride", c_i64), ("dk_head_stride", c_i64),
        ("dv_batch_stride", c_i64), ("dv_row_stride", c_i64), ("dv_head_stride", c_i64),
        ("deterministic", c_i32), ("cta_pair", c_i32),
        ("phase_events", c_vp * 3),
        ("single_pass", c_i32),
    ]


_lib = None


def load(path: str = LIB_PATH):
    """Loads libattn_gb300.so and declares the C signatures (once)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python exact_attention_bf16_gb300/build.py` "
            "(nvcc, sm_103a). There is no non-CUDA fallback.")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    sig = {
        "attn_fwd_workspace_size": (ctypes.c_size_t, [P(AttnFwdParams)]),
        "attn_bwd_workspace_size": (ctypes.c_size_t, [P(AttnBwdParams)]),
        "attn_fwd": (ctypes.c_int, [P(AttnFwdParams), c_vp, ctypes.c_size_t, c_vp]),
        "attn_fwd_varlen": (ctypes.c_int, [P(AttnFwdParams), c_vp, ctypes.c_size_t, c_vp]),
        "attn_fwd_block_sparse": (ctypes.c_int, [P(AttnFwdParams), c_vp, c_vp, ctypes.c_int32, ctypes.c_int32, c_vp,
                                                 ctypes.c_size_t, c_vp]),
        "attn_bwd_block_sparse_workspace_size": (ctypes.c_size_t, [P(AttnBwdParams), ctypes.c_int32]),
        "attn_bwd_block_sparse": (ctypes.c_int, [P(AttnBwdParams), c_vp, c_vp, ctypes.c_int32, ctypes.c_int32, c_vp,
                                                 ctypes.c_size_t, c_vp]),
        "attn_bwd": (ctypes.c_int, [P(AttnBwdParams), c_vp, ctypes.c_size_t, c_vp]),
        "attn_bwd_varlen": (ctypes.c_int, [P(AttnBwdParams), c_vp, ctypes.c_size_t, c_vp]),
        "attn_bwd_noalloc": (ctypes.c_int, [P(AttnBwdParams), c_vp]),
        "attn_exp2_eval": (ctypes.c_int, [c_vp, c_vp, c_vp, c_i64, c_vp]),
        "attn_diag_wait_timeout": (ctypes.c_int, [P(AttnFwdParams), ctypes.c_uint32, c_vp]),
        "attn_get_device_status": (ctypes.c_int, [c_vp, P(ctypes.c_uint32)]),
        "attn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "attn_last_cuda_error": (ctypes.c_char_p, []),
        "attn_abi_version": (c_i32, []),
        "attn_fwd_params_size": (ctypes.c_size_t, []),
        "attn_bwd_params_size": (ctypes.c_size_t, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.attn_abi_version() != ABI_VERSION:
        raise ImportError(f"libattn_gb300.so ABI {lib.attn_abi_version()} != binding ABI {ABI_VERSION}")
    if lib.attn_fwd_params_size() != ctypes.sizeof(AttnFwdParams) or \
            lib.attn_bwd_params_size() != ctypes.sizeof(AttnBwdParams):
        raise ImportError("libattn_gb300.so parameter-struct layout differs from the binding")
    _lib = lib
    return lib


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = _lib
        detail = lib.attn_last_cuda_error().decode() if (lib is not None and status == ATTN_ERR_CUDA) else ""
        super().__init__(f"{where}: {STATUS.get(status, status)}" + (f" ({detail})" if detail else ""))
        self.status = status


def check(status: int, where: str):
    if status != ATTN_OK:
        raise AttnError(status, where)
