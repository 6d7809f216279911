"""Exact fused scaled-dot-product attention (bf16) for NVIDIA GB300 (sm_103a).

The compute lives in libattn_gb300.so (hand-written CUDA: TMA, tcgen05 MMAs
with Tensor Memory accumulators, warp-specialised pipelines); see
include/attn.h for the C ABI. This package is a thin binding with the same
entry-point names: it only marshals torch tensors (device memory, strides,
the current CUDA stream) into the C parameter structs. Nothing here computes
attention, and there is no CPU or library fallback: if the shared library is
missing, importing this package raises.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Tuple

import torch

from . import _abi
from ._abi import AttnBwdParams, AttnError, AttnFwdParams  # noqa: F401

_lib = _abi.load()

SUPPORTED_HEAD_DIMS = ((64, 64), (128, 128), (192, 128))

__all__ = [
    "attn_fwd", "attn_fwd_block_sparse", "attn_fwd_varlen", "attn_bwd", "attn_bwd_block_sparse",
    "block_lists_from_mask", "attn_bwd_varlen", "attn_exp2_eval",
    "attn_get_device_status", "attention", "AttnError", "SUPPORTED_HEAD_DIMS", "library_path",
]


def library_path() -> str:
    return _abi.LIB_PATH


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _check_bf16(name: str, t: torch.Tensor, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got shape {tuple(t.shape)}")
    if t.stride(-1) != 1:
        raise ValueError(f"{name}: head_dim must be contiguous")


def _check_inputs(q, k, v, ndim: int) -> bool:
    """q, k, v all bf16, or all FP8 E4M3 (torch.float8_e4m3fn, forward only); returns True for E4M3."""
    f8 = q.dtype == torch.float8_e4m3fn
    for n, t in (("q", q), ("k", k), ("v", v)):
        if f8:
            if not isinstance(t, torch.Tensor) or t.dtype != torch.float8_e4m3fn:
                raise TypeError(f"{n} must be float8_e4m3fn like q")
            if not t.is_cuda or t.dim() != ndim or t.stride(-1) != 1:
                raise ValueError(f"{n} must be a CUDA tensor of {ndim} dims with contiguous head_dim")
        else:
            _check_bf16(n, t, ndim)
    return f8


def _set_input_dtype(p: AttnFwdParams, f8: bool, q_descale, k_descale, v_descale):
    if f8:
        p.input_dtype = _abi.INPUT_E4M3
        p.q_descale, p.k_descale, p.v_descale = float(q_descale), float(k_descale), float(v_descale)


def _strides4(t: torch.Tensor):
    # [B, N, H, d] -> (batch, row, head) element strides
    return t.stride(0), t.stride(1), t.stride(2)


def _strides3(t: torch.Tensor):
    # packed [total, H, d] -> batch stride unused
    return 0, t.stride(0), t.stride(1)


def _fill_fwd(p: AttnFwdParams, q, k, v, o, lse, strides, scale, causal):
    p.q, p.k, p.v, p.o, p.lse = _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse)
    (p.q_batch_stride, p.q_row_stride, p.q_head_stride) = strides(q)
    (p.k_batch_stride, p.k_row_stride, p.k_head_stride) = strides(k)
    (p.v_batch_stride, p.v_row_stride, p.v_head_stride) = strides(v)
    (p.o_batch_stride, p.o_row_stride, p.o_head_stride) = strides(o)
    p.d_qk, p.d_v = q.shape[-1], v.shape[-1]
    p.heads = q.shape[-2]
    p.softmax_scale = scale
    p.causal = 1 if causal else 0


def _set_score_mod(p: AttnFwdParams, q: torch.Tensor, softcap, alibi_slopes):
    """Score modification: logits soft-capped at ``softcap`` (a' = c tanh(a / c)), or ALiBi with one
    slope per head (``alibi_slopes`` float32 [H] on q's GPU, each >= 0)."""
    if softcap is not None and alibi_slopes is not None:
        raise ValueError("choose one score modification: softcap or alibi_slopes")
    if softcap is not None:
        p.score_mod, p.softcap = _abi.SCORE_SOFTCAP, float(softcap)
    elif alibi_slopes is not None:
        t = alibi_slopes
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or t.shape != (q.shape[-2],):
            raise ValueError(f"alibi_slopes must be a contiguous float32 CUDA tensor of shape [{q.shape[-2]}]")
        if t.device != q.device:
            raise ValueError(f"alibi_slopes is on {t.device} but q is on {q.device}")
        p.score_mod, p.alibi_slopes = _abi.SCORE_ALIBI, _ptr(t)


def _workspace(size: int, device) -> Tuple[Optional[torch.Tensor], int]:
    if size == 0:
        return None, 0
    return torch.empty(size, dtype=torch.uint8, device=device), size


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, causal: bool = False,
             softmax_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
             lse: Optional[torch.Tensor] = None, rescale_stats: Optional[torch.Tensor] = None,
             exp2_emu_period: int = 0, softcap: Optional[float] = None,
             alibi_slopes: Optional[torch.Tensor] = None, q_descale: float = 1.0, k_descale: float = 1.0,
             v_descale: float = 1.0, cta_pair: bool = False, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Dense forward. q [B, Nq, H, d_qk], k [B, Nk, H, d_qk], v [B, Nk, H, d_v] (bf16, CUDA).
    Returns (O [B, Nq, H, d_v] bf16, LSE [B, H, Nq] fp32, natural log). ``exp2_emu_period`` (0, 4, 8)
    sends one column in that many of every row's exp2 to the FMA-pipe polynomial. ``softcap`` or
    ``alibi_slopes`` select a score modification (include/attn.h, attn_fwd_params.score_mod).
    q, k, v may instead all be torch.float8_e4m3fn (d = 128), standing for their values times
    ``q_descale``, ``k_descale``, ``v_descale``. ``cta_pair`` runs the two-SM forward (d = 128)."""
    f8 = _check_inputs(q, k, v, 4)
    B, Nq, H, dqk = q.shape
    Nk, dv = k.shape[1], v.shape[-1]
    if k.shape != (B, Nk, H, dqk) or v.shape[:3] != (B, Nk, H):
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    scale = float(softmax_scale) if softmax_scale is not None else 1.0 / math.sqrt(dqk)
    if out is None:
        out = torch.empty((B, Nq, H, dv), dtype=torch.bfloat16, device=q.device)
    _check_bf16("out", out, 4)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if lse.shape != (B, H, Nq) or not lse.is_contiguous() or lse.dtype != torch.float32:
        raise ValueError("lse must be a contiguous float32 [B, H, Nq] tensor")
    p = AttnFwdParams()
    _fill_fwd(p, q, k, v, out, lse, _strides4, scale, causal)
    p.batch, p.seqlen_q, p.seqlen_k = B, Nq, Nk
    p.rescale_stats = _ptr(rescale_stats)
    p.exp2_emu_period = int(exp2_emu_period)
    _set_score_mod(p, q, softcap, alibi_slopes)
    _set_input_dtype(p, f8, q_descale, k_descale, v_descale)
    p.cta_pair = 1 if cta_pair else 0
    ws, nbytes = _workspace(_lib.attn_fwd_workspace_size(ctypes.byref(p)), q.device)
    _abi.check(_lib.attn_fwd(ctypes.byref(p), _ptr(ws), nbytes, _stream(stream)), "attn_fwd")
    return out, lse


def _check_lists(q: torch.Tensor, kv_count: torch.Tensor, kv_index: torch.Tensor) -> Tuple[int, int]:
    """Validates the block lists of a dense [B, Nq, H, d] call; returns (max_kv, lists_per_head).
    Shared lists: kv_count [nqb], kv_index [nqb, max_kv]. Per (batch, head): kv_count [B, H, nqb],
    kv_index [B, H, nqb, max_kv]."""
    for n, t in (("kv_count", kv_count), ("kv_index", kv_index)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 CUDA tensor")
        if t.device != q.device:
            raise ValueError(f"{n} is on {t.device} but q is on {q.device}: the block lists must be on q's GPU")
    B, Nq, H = q.shape[0], q.shape[1], q.shape[2]
    nqb = (Nq + 255) // 256
    if kv_count.shape == (nqb,) and kv_index.dim() == 2 and kv_index.shape[0] == nqb:
        return int(kv_index.shape[1]), 0
    if kv_count.shape == (B, H, nqb) and kv_index.dim() == 4 and kv_index.shape[:3] == (B, H, nqb):
        return int(kv_index.shape[3]), 1
    raise ValueError(f"kv_count must be [{nqb}] and kv_index [{nqb}, max_kv], or per (batch, head) "
                     f"[{B}, {H}, {nqb}] and [{B}, {H}, {nqb}, max_kv]")


def block_lists_from_mask(block_mask: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """(kv_count, kv_index) for :func:`attn_fwd_block_sparse` from a boolean block mask
    [ceil(Nq/256), ceil(Nk/128)], or [B, H, ceil(Nq/256), ceil(Nk/128)] for lists per (batch, head)
    (True = the query block attends to the key block), key blocks in ascending order; on the mask's
    device. Argument preparation only."""
    if block_mask.dtype != torch.bool or block_mask.dim() not in (2, 4):
        raise ValueError("block_mask must be a bool tensor [query blocks, key blocks] or [B, H, query blocks, "
                         "key blocks]")
    m = block_mask.to(torch.int32)
    kv_count = m.sum(dim=-1, dtype=torch.int32)
    max_kv = max(int(kv_count.max().item()) if kv_count.numel() else 0, 1)
    # stable sort puts listed blocks first, each group in ascending key-block order
    order = torch.sort(1 - m, dim=-1, stable=True).indices.to(torch.int32)
    kv_index = order[..., :max_kv].contiguous()
    return kv_count.contiguous(), kv_index


def attn_fwd_block_sparse(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, kv_count: torch.Tensor,
                          kv_index: torch.Tensor, *, causal: bool = False, softmax_scale: Optional[float] = None,
                          out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                          softcap: Optional[float] = None, alibi_slopes: Optional[torch.Tensor] = None,
                          stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Block-sparse dense forward. q/k/v as in :func:`attn_fwd`; kv_count int32 [ceil(Nq/256)] and
    kv_index int32 [ceil(Nq/256), max_kv] (CUDA, contiguous): query block b (rows 256b..256b+255)
    attends to key blocks (of 128 keys) kv_index[b, :kv_count[b]], each listed at most once; or per
    (batch, head), kv_count [B, H, nqb] and kv_index [B, H, nqb, max_kv].
    Returns (O [B, Nq, H, d_v] bf16, LSE [B, H, Nq] fp32)."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_bf16(n, t, 4)
    B, Nq, H, dqk = q.shape
    Nk, dv = k.shape[1], v.shape[-1]
    if k.shape != (B, Nk, H, dqk) or v.shape[:3] != (B, Nk, H):
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    max_kv, per_head = _check_lists(q, kv_count, kv_index)
    scale = float(softmax_scale) if softmax_scale is not None else 1.0 / math.sqrt(dqk)
    if out is None:
        out = torch.empty((B, Nq, H, dv), dtype=torch.bfloat16, device=q.device)
    _check_bf16("out", out, 4)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if lse.shape != (B, H, Nq) or not lse.is_contiguous() or lse.dtype != torch.float32:
        raise ValueError("lse must be a contiguous float32 [B, H, Nq] tensor")
    p = AttnFwdParams()
    _fill_fwd(p, q, k, v, out, lse, _strides4, scale, causal)
    p.batch, p.seqlen_q, p.seqlen_k = B, Nq, Nk
    _set_score_mod(p, q, softcap, alibi_slopes)
    ws, nbytes = _workspace(_lib.attn_fwd_workspace_size(ctypes.byref(p)), q.device)
    _abi.check(_lib.attn_fwd_block_sparse(ctypes.byref(p), _ptr(kv_count), _ptr(kv_index), max_kv, per_head,
                                          _ptr(ws), nbytes, _stream(stream)), "attn_fwd_block_sparse")
    return out, lse


def attn_fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
                    cu_seqlens_k: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int, *, causal: bool = False,
                    softmax_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                    lse: Optional[torch.Tensor] = None, rescale_stats: Optional[torch.Tensor] = None,
                    exp2_emu_period: int = 0, softcap: Optional[float] = None,
                    alibi_slopes: Optional[torch.Tensor] = None, q_descale: float = 1.0, k_descale: float = 1.0,
                    v_descale: float = 1.0, cta_pair: bool = False,
                    stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Packed variable-length forward. q [total_q, H, d_qk], k/v [total_k, H, d]; cu_seqlens int32 on
    the device. Returns (O [total_q, H, d_v], LSE [H, total_q]). Score modifications and E4M3 inputs
    as in :func:`attn_fwd`, positions counted within each sequence."""
    f8 = _check_inputs(q, k, v, 3)
    for n, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 CUDA tensor")
    tq, H, dqk = q.shape
    tk, dv = k.shape[0], v.shape[-1]
    scale = float(softmax_scale) if softmax_scale is not None else 1.0 / math.sqrt(dqk)
    if out is None:
        out = torch.empty((tq, H, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((H, tq), dtype=torch.float32, device=q.device)
    p = AttnFwdParams()
    _fill_fwd(p, q, k, v, out, lse, _strides3, scale, causal)
    p.cu_seqlens_q, p.cu_seqlens_k = _ptr(cu_seqlens_q), _ptr(cu_seqlens_k)
    p.num_seqs = cu_seqlens_q.numel() - 1
    p.max_seqlen_q, p.max_seqlen_k = int(max_seqlen_q), int(max_seqlen_k)
    p.total_q, p.total_k = tq, tk
    p.batch = 1
    p.rescale_stats = _ptr(rescale_stats)
    p.exp2_emu_period = int(exp2_emu_period)
    _set_score_mod(p, q, softcap, alibi_slopes)
    _set_input_dtype(p, f8, q_descale, k_descale, v_descale)
    p.cta_pair = 1 if cta_pair else 0
    ws, nbytes = _workspace(_lib.attn_fwd_workspace_size(ctypes.byref(p)), q.device)
    _abi.check(_lib.attn_fwd_varlen(ctypes.byref(p), _ptr(ws), nbytes, _stream(stream)), "attn_fwd_varlen")
    return out, lse


def _fill_bwd(p: AttnBwdParams, do, dq, dk, dv, strides, deterministic, cta_pair=False, single_pass=False):
    p.dout, p.dq, p.dk, p.dv = _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv)
    (p.do_batch_stride, p.do_row_stride, p.do_head_stride) = strides(do)
    (p.dq_batch_stride, p.dq_row_stride, p.dq_head_stride) = strides(dq)
    (p.dk_batch_stride, p.dk_row_stride, p.dk_head_stride) = strides(dk)
    (p.dv_batch_stride, p.dv_row_stride, p.dv_head_stride) = strides(dv)
    p.deterministic = 1 if deterministic else 0
    p.cta_pair = 1 if cta_pair else 0
    p.single_pass = 1 if single_pass else 0


def _event_handles(events):
    if events is None:
        return None
    out = []
    for ev in events:
        if ev is None:
            out.append(None)
            continue
        if getattr(ev, "cuda_event", 0) == 0:  # torch creates the CUDA event lazily
            ev.record()
        out.append(ev.cuda_event)
    return out


def attn_bwd(q, k, v, out, lse, dout, *, causal: bool = False, softmax_scale: Optional[float] = None,
             deterministic: bool = False, dq=None, dk=None, dv=None, stream=None, phase_events=None,
             cta_pair: bool = False, softcap: Optional[float] = None, alibi_slopes: Optional[torch.Tensor] = None,
             single_pass: bool = False):
    """Dense backward: returns (dQ, dK, dV) bf16 for the loss <O, dO>. ``phase_events`` (optional, three
    torch.cuda.Event) are recorded after the D pass, the dK/dV kernel and the dQ kernel. ``cta_pair``
    selects the two-SM (cta_group::2) dK/dV kernel (d = 128); ``single_pass`` the one-kernel backward
    whose dQ partials are reduced across CTAs (d = 64; ordered by key tile when ``deterministic``).
    The score modification must be the forward's."""
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout)):
        _check_bf16(n, t, 4)
    B, Nq, H, dqk = q.shape
    Nk = k.shape[1]
    scale = float(softmax_scale) if softmax_scale is not None else 1.0 / math.sqrt(dqk)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    p = AttnBwdParams()
    _fill_fwd(p.fwd, q, k, v, out, lse, _strides4, scale, causal)
    p.fwd.batch, p.fwd.seqlen_q, p.fwd.seqlen_k = B, Nq, Nk
    _fill_bwd(p, dout, dq, dk, dv, _strides4, deterministic, cta_pair, single_pass)
    _set_score_mod(p.fwd, q, softcap, alibi_slopes)
    handles = _event_handles(phase_events)
    if handles is not None:
        for i, h in enumerate(handles):
            p.phase_events[i] = h
    ws, nbytes = _workspace(_lib.attn_bwd_workspace_size(ctypes.byref(p)), q.device)
    _abi.check(_lib.attn_bwd(ctypes.byref(p), _ptr(ws), nbytes, _stream(stream)), "attn_bwd")
    return dq, dk, dv


def attn_bwd_block_sparse(q, k, v, out, lse, dout, kv_count, kv_index, *, causal: bool = False,
                          softmax_scale: Optional[float] = None, deterministic: bool = False, dq=None, dk=None,
                          dv=None, softcap: Optional[float] = None, alibi_slopes: Optional[torch.Tensor] = None,
                          stream=None):
    """Block-sparse backward for :func:`attn_fwd_block_sparse` with the same kv_count / kv_index:
    returns (dQ, dK, dV) bf16 for the loss <O, dO>."""
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout)):
        _check_bf16(n, t, 4)
    B, Nq, H, dqk = q.shape
    Nk = k.shape[1]
    max_kv, per_head = _check_lists(q, kv_count, kv_index)
    scale = float(softmax_scale) if softmax_scale is not None else 1.0 / math.sqrt(dqk)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    p = AttnBwdParams()
    _fill_fwd(p.fwd, q, k, v, out, lse, _strides4, scale, causal)
    p.fwd.batch, p.fwd.seqlen_q, p.fwd.seqlen_k = B, Nq, Nk
    _fill_bwd(p, dout, dq, dk, dv, _strides4, deterministic)
    _set_score_mod(p.fwd, q, softcap, alibi_slopes)
    ws, nbytes = _workspace(_lib.attn_bwd_block_sparse_workspace_size(ctypes.byref(p), per_head), q.device)
    _abi.check(_lib.attn_bwd_block_sparse(ctypes.byref(p), _ptr(kv_count), _ptr(kv_index), max_kv, per_head,
                                          _ptr(ws), nbytes, _stream(stream)), "attn_bwd_block_sparse")
    return dq, dk, dv


def attn_bwd_varlen(q, k, v, out, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int, *,
                    causal: bool = False, softmax_scale: Optional[float] = None, deterministic: bool = False,
                    dq=None, dk=None, dv=None, stream=None, cta_pair: bool = False, softcap: Optional[float] = None,
                    alibi_slopes: Optional[torch.Tensor] = None, single_pass: bool = False):
    """Packed variable-length backward: returns (dQ, dK, dV) packed like q, k, v."""
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout)):
        _check_bf16(n, t, 3)
    tq, H, dqk = q.shape
    scale = float(softmax_scale) if softmax_scale is not None else 1.0 / math.sqrt(dqk)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    p = AttnBwdParams()
    _fill_fwd(p.fwd, q, k, v, out, lse, _strides3, scale, causal)
    p.fwd.cu_seqlens_q, p.fwd.cu_seqlens_k = _ptr(cu_seqlens_q), _ptr(cu_seqlens_k)
    p.fwd.num_seqs = cu_seqlens_q.numel() - 1
    p.fwd.max_seqlen_q, p.fwd.max_seqlen_k = int(max_seqlen_q), int(max_seqlen_k)
    p.fwd.total_q, p.fwd.total_k = tq, k.shape[0]
    p.fwd.batch = 1
    _fill_bwd(p, dout, dq, dk, dv, _strides3, deterministic, cta_pair, single_pass)
    _set_score_mod(p.fwd, q, softcap, alibi_slopes)
    ws, nbytes = _workspace(_lib.attn_bwd_workspace_size(ctypes.byref(p)), q.device)
    _abi.check(_lib.attn_bwd_varlen(ctypes.byref(p), _ptr(ws), nbytes, _stream(stream)), "attn_bwd_varlen")
    return dq, dk, dv


def attn_exp2_eval(x: torch.Tensor, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Evaluates the kernels' software (Cody-Waite + cubic) and hardware exp2 on a float32 CUDA tensor."""
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    yp, yh = torch.empty_like(x), torch.empty_like(x)
    _abi.check(_lib.attn_exp2_eval(_ptr(x), _ptr(yp), _ptr(yh), x.numel(), _stream(stream)), "attn_exp2_eval")
    return yp, yh


def attn_get_device_status(stream=None) -> int:
    """Synchronises the stream; raises AttnError(ATTN_ERR_TIMEOUT) if a kernel recorded a failure."""
    detail = ctypes.c_uint32(0)
    st = _lib.attn_get_device_status(_stream(stream), ctypes.byref(detail))
    if st != _abi.ATTN_OK:
        raise AttnError(st, f"device status 0x{detail.value:08x}")
    return detail.value


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, softmax_scale, deterministic, kv_count, kv_index, softcap, alibi_slopes):
        mod = dict(softcap=softcap, alibi_slopes=alibi_slopes)
        if kv_count is None:
            o, lse = attn_fwd(q, k, v, causal=causal, softmax_scale=softmax_scale, **mod)
        else:
            o, lse = attn_fwd_block_sparse(q, k, v, kv_count, kv_index, causal=causal, softmax_scale=softmax_scale,
                                           **mod)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale, ctx.det = causal, softmax_scale, deterministic
        ctx.lists = (kv_count, kv_index)
        ctx.mod = mod
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        kv_count, kv_index = ctx.lists
        if kv_count is None:
            dq, dk, dv = attn_bwd(q, k, v, o, lse, do.contiguous(), causal=ctx.causal, softmax_scale=ctx.scale,
                                  deterministic=ctx.det, **ctx.mod)
        else:
            dq, dk, dv = attn_bwd_block_sparse(q, k, v, o, lse, do.contiguous(), kv_count, kv_index,
                                               causal=ctx.causal, softmax_scale=ctx.scale, deterministic=ctx.det,
                                               **ctx.mod)
        return dq, dk, dv, None, None, None, None, None, None, None


def attention(q, k, v, causal: bool = False, softmax_scale: Optional[float] = None, deterministic: bool = False,
              block_mask: Optional[Tuple[torch.Tensor, torch.Tensor]] = None, softcap: Optional[float] = None,
              alibi_slopes: Optional[torch.Tensor] = None):
    """Autograd wrapper over attn_fwd / attn_bwd for [B, N, H, d] bf16 tensors. ``block_mask``
    = (kv_count, kv_index) selects the block-sparse pair attn_fwd_block_sparse / attn_bwd_block_sparse;
    ``softcap`` / ``alibi_slopes`` a score modification."""
    kv_count, kv_index = block_mask if block_mask is not None else (None, None)
    return _Attention.apply(q, k, v, causal, softmax_scale, deterministic, kv_count, kv_index, softcap, alibi_slopes)
