// Forward launchers (the kernel itself is in fwd_kernel.cuh), the V -> fp16
// conversion pass, the kernel for calls without keys and the exp2 diagnostic.
#include <cuda_bf16.h>

#include "fwd_kernel.cuh"

namespace gb300 {
namespace fwd {

// Fills O = 0, LSE = -inf (rows that see no key: Nk == 0).
__global__ void fwd_empty_kernel(FwdArgs a, int dv) {
  const int64_t rows = static_cast<int64_t>(a.num_units) * a.heads * a.seqlen_q;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < rows;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(idx % a.seqlen_q);
    const int64_t bh = idx / a.seqlen_q;
    const int h = static_cast<int>(bh % a.heads), b = static_cast<int>(bh / a.heads);
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.o) + b * a.o_sb + static_cast<int64_t>(r) * a.o_sn + h * a.o_sh;
    for (int c = 0; c < dv; ++c) orow[c] = __float2bfloat16_rn(0.f);
    a.lse[b * a.lse_sb + h * a.lse_sh + r] = -INFINITY;
  }
}

__global__ void exp2_eval_kernel(const float* x, float* yp, float* yh, int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float v = x[i];
    if (yp) yp[i] = ex2_emu(v);
    if (yh) yh[i] = ex2_mufu(v);
  }
}

// Merges the key ranges of a split forward: per row, LSE = ln sum_r exp(LSE_r) and
// O = sum_r exp(LSE_r - LSE) O_r (the standard merge of partial softmax results over
// disjoint key sets), the ranges taken in order, so the result does not depend on
// timing. One warp per (batch, head, row); lane l holds columns [DV/32 l, DV/32 (l+1)).
template <int DV>
__global__ void combine_kv_splits_kernel(FwdArgs a) {
  constexpr int CPL = DV / 32;
  const int lane = static_cast<int>(threadIdx.x & 31u);
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t row = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; row < a.part_rows;
       row += nwarps) {
    const float lr = lane < a.kv_split ? a.lse_part[lane * a.part_rows + row] : -INFINITY;
    float m = lr;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float w = (lr == -INFINITY) ? 0.f : expf(lr - m);
    float wsum = w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    float acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
    for (int r = 0; r < a.kv_split; ++r) {
      const float wr = __shfl_sync(0xffffffffu, w, r);
      if (wr == 0.f) continue;  // warp-uniform: a range with no visible key
      const float* src = a.o_part + (r * a.part_rows + row) * DV + lane * CPL;
      if constexpr (CPL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] = fmaf(wr, v.x, acc[0]);
        acc[1] = fmaf(wr, v.y, acc[1]);
        acc[2] = fmaf(wr, v.z, acc[2]);
        acc[3] = fmaf(wr, v.w, acc[3]);
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] = fmaf(wr, v.x, acc[0]);
        acc[1] = fmaf(wr, v.y, acc[1]);
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const int64_t q = row % a.seqlen_q, bh = row / a.seqlen_q;
    const int64_t h = bh % a.heads, b = bh / a.heads;
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.o) + b * a.o_sb + q * a.o_sn + h * a.o_sh + lane * CPL;
    if constexpr (CPL == 4) {
      *reinterpret_cast<uint2*>(orow) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                   pack_bf16x2(acc[2] * inv, acc[3] * inv));
    } else {
      *reinterpret_cast<uint32_t*>(orow) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0) a.lse[b * a.lse_sb + h * a.lse_sh + q] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
  }
}

template <int DV>
cudaError_t launch_combine(const FwdArgs& a, cudaStream_t stream) {
  if (a.kv_split < 2 || a.kv_split > 32 || a.part_rows <= 0) return cudaErrorInvalidValue;
  const int64_t blocks = (a.part_rows + 7) / 8;  // 8 warps (rows) per block of 256
  combine_kv_splits_kernel<DV><<<static_cast<unsigned>(blocks < 4864 ? blocks : 4864), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

// exp2 split: every EMU-th column of a row goes to the FMA-pipe polynomial
// (0 = all on the hardware unit). Built for 0, 4 and 8.
template <int DQK, int DV>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tv16,
                     const FwdArgs& a, cudaStream_t stream) {
  if (a.kv_split > 1) {  // split keys: dense d = 64 or 128, no exp2 emulation
    if constexpr (DQK <= 128 && DQK == DV) {
      if (a.emu_period != 0 || a.tiles != nullptr) return cudaErrorInvalidValue;
      cudaError_t e = launch_e<DQK, DV, 0, false, false, false, kModNone, false, true>(tq, tk, tv, tv16, a, stream);
      return e == cudaSuccess ? launch_combine<DV>(a, stream) : e;
    }
    return cudaErrorInvalidValue;
  }
  if (a.tiles != nullptr) {
    switch (a.emu_period) {
      case 0: return launch_e<DQK, DV, 0, false, false, true>(tq, tk, tv, tv16, a, stream);
      case 4: return launch_e<DQK, DV, 4, false, false, true>(tq, tk, tv, tv16, a, stream);
      case 8: return launch_e<DQK, DV, 8, false, false, true>(tq, tk, tv, tv16, a, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.emu_period) {
    case 0: return launch_e<DQK, DV, 0>(tq, tk, tv, tv16, a, stream);
    case 4: return launch_e<DQK, DV, 4>(tq, tk, tv, tv16, a, stream);
    case 8: return launch_e<DQK, DV, 8>(tq, tk, tv, tv16, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

// V -> fp16 copy for the PV product (contiguous [rows, heads, d_v], rows = B * N
// dense or total varlen). One warp per token row: its heads x d_v values are
// HEADS x DV / 8 units of 16 bytes, a warp-wide unit index split by constant
// shifts, the (batch, row) division done once per row. Sets *flag when a
// finite value lies outside fp16's range (|v| >= 65536, which would become
// inf); inf and NaN convert to themselves.
template <int DV>
__global__ void v_to_f16_kernel(const void* v, int64_t sb, int64_t sn, int64_t sh, int nb, int nrows, int heads,
                                void* out, uint32_t* flag) {
  constexpr int UPH = DV / 8;  // 16-byte units per (row, head)
  const int upr = heads * UPH;  // per row
  const int64_t rows = static_cast<int64_t>(nb) * nrows;
  const int lane = static_cast<int>(threadIdx.x & 31u);
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  uint32_t bad = 0;
  for (int64_t r = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; r < rows; r += nwarps) {
    const int b = static_cast<int>(r / nrows), n = static_cast<int>(r % nrows);
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(v) + b * sb + n * sn;
    uint4* dst = static_cast<uint4*>(out) + r * upr;
#pragma unroll 4
    for (int i = lane; i < upr; i += 32) {
      const uint4 x = *reinterpret_cast<const uint4*>(src + (i / UPH) * sh + 8 * (i % UPH));
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t lo = w[e] & 0x7FFFu, hi = (w[e] >> 16) & 0x7FFFu;
        bad |= static_cast<uint32_t>(lo >= 0x4780u && lo < 0x7F80u) | static_cast<uint32_t>(hi >= 0x4780u && hi < 0x7F80u);
        o[e] = pack_f16x2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
      }
      dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  if (__any_sync(0xffffffffu, bad != 0) && lane == 0) atomicOr(flag, 1u);
}

}  // namespace fwd

cudaError_t launch_fwd(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tv16, const FwdArgs& a, cudaStream_t stream) {
  if (a.kv_count != nullptr) return cudaErrorInvalidValue;
  if (a.score_mod != kModNone) return launch_fwd_mod(d_qk, d_v, tq, tk, tv, tv16, a, stream);
  if (d_qk == 64 && d_v == 64) return fwd::launch_t<64, 64>(tq, tk, tv, tv16, a, stream);
  if (d_qk == 128 && d_v == 128) return fwd::launch_t<128, 128>(tq, tk, tv, tv16, a, stream);
  if (d_qk == 192 && d_v == 128) return fwd::launch_t<192, 128>(tq, tk, tv, tv16, a, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_sparse(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tv16, const FwdArgs& a, cudaStream_t stream) {
  if (a.cu_q != nullptr || a.tiles != nullptr || a.emu_period != 0 || a.kv_count == nullptr || a.max_kv < 0)
    return cudaErrorInvalidValue;
  if (a.max_kv > 0 && a.kv_index == nullptr) return cudaErrorInvalidValue;
  if (a.score_mod != kModNone) return launch_fwd_mod(d_qk, d_v, tq, tk, tv, tv16, a, stream);
  if (d_qk == 64 && d_v == 64) return fwd::launch_e<64, 64, 0, true>(tq, tk, tv, tv16, a, stream);
  if (d_qk == 128 && d_v == 128) return fwd::launch_e<128, 128, 0, true>(tq, tk, tv, tv16, a, stream);
  if (d_qk == 192 && d_v == 128) return fwd::launch_e<192, 128, 0, true>(tq, tk, tv, tv16, a, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_diag_timeout(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                    const FwdArgs& a, cudaStream_t stream) {
  if (a.cu_q != nullptr || a.tiles != nullptr || a.kv_count != nullptr || a.spin_limit == 0 || a.v16_flag != nullptr ||
      a.score_mod != kModNone)
    return cudaErrorInvalidValue;
  return fwd::launch_e<64, 64, 0, false, true>(tq, tk, tv, tv, a, stream);
}

cudaError_t launch_v_to_f16(const void* v, int64_t sb, int64_t sn, int64_t sh, int nb, int nrows, int heads, int dv,
                            void* out, uint32_t* flag, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(nb) * nrows;
  if (rows == 0) return cudaSuccess;
  const int64_t want = (rows + 7) / 8;  // 8 warps (rows) per block and pass
  const unsigned blocks = static_cast<unsigned>(want < 152 * 8 ? want : 152 * 8);
  if (dv == 64) fwd::v_to_f16_kernel<64><<<blocks, 256, 0, stream>>>(v, sb, sn, sh, nb, nrows, heads, out, flag);
  else if (dv == 128) fwd::v_to_f16_kernel<128><<<blocks, 256, 0, stream>>>(v, sb, sn, sh, nb, nrows, heads, out, flag);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_fwd_empty(const FwdArgs& a, int d_v, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.num_units) * a.heads * a.seqlen_q;
  if (rows == 0) return cudaSuccess;
  const int blocks = static_cast<int>(rows / 256 + 1 < 4096 ? rows / 256 + 1 : 4096);
  fwd::fwd_empty_kernel<<<blocks, 256, 0, stream>>>(a, d_v);
  return cudaGetLastError();
}

cudaError_t launch_exp2_eval(const float* x, float* y_poly, float* y_hw, int64_t n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = (n + 255) / 256 < 8192 ? (n + 255) / 256 : 8192;
  fwd::exp2_eval_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, y_poly, y_hw, n);
  return cudaGetLastError();
}

}  // namespace gb300
