// Backward launchers (the dK/dV and dQ kernels are in bwd_kernels.cuh), the
// D = rowsum(dO * O) pass, the zero fill and the block-list transpose.
#include <cuda_bf16.h>

#include "bwd_kernels.cuh"

namespace gb300 {
namespace bwd {

// ===========================================================================
// Preprocess: D = rowsum(dO * O). HBM-bound: DV / 8 lanes share a row, each
// loading 16 bytes of O and of dO per access (rows and head slices start on
// 16-byte boundaries, as the TMA tensor maps already require).
// ===========================================================================
template <int DV>
__global__ void preprocess_kernel(const BwdArgs a) {
  constexpr int LPR = DV / 8;    // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp
  const int64_t rows = static_cast<int64_t>(a.batch) * a.seqlen_q * a.heads;
  const int64_t warp0 = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, l = lane % LPR;
  for (int64_t r0 = warp0 * RPW; r0 < rows; r0 += nwarps * RPW) {
    const int64_t r = r0 + sub;
    float acc = 0.f;
    int h = 0, i = 0, b = 0;
    if (r < rows) {
      h = static_cast<int>(r % a.heads);
      const int64_t bi = r / a.heads;
      i = static_cast<int>(bi % a.seqlen_q);
      b = static_cast<int>(bi / a.seqlen_q);
      const __nv_bfloat16* o = static_cast<const __nv_bfloat16*>(a.o) + b * a.o_sb + i * a.o_sn + h * a.o_sh;
      const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(a.dout) + b * a.do_sb + i * a.do_sn + h * a.do_sh;
      const uint4 ov = *reinterpret_cast<const uint4*>(o + 8 * l);
      const uint4 gv = *reinterpret_cast<const uint4*>(g + 8 * l);
      const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
        const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
        acc = fmaf(of.x, gf.x, acc);
        acc = fmaf(of.y, gf.y, acc);
      }
    }
#pragma unroll
    for (int s = LPR / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (r < rows && l == 0) a.dsum[b * a.lse_sb + h * a.lse_sh + i] = acc;
  }
}



// Zero rows: dQ (all queries) and/or dK, dV (all keys).
__global__ void zero_kernel(void* base, int64_t sb, int64_t sn, int64_t sh, int nb, int nrows, int heads, int d) {
  const int64_t total = static_cast<int64_t>(nb) * nrows * heads;
  for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r < total;
       r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int h = static_cast<int>(r % heads);
    const int64_t bi = r / heads;
    const int i = static_cast<int>(bi % nrows);
    const int b = static_cast<int>(bi / nrows);
    __nv_bfloat16* p = static_cast<__nv_bfloat16*>(base) + b * sb + i * sn + h * sh;
    for (int c = 0; c < d; ++c) p[c] = __float2bfloat16_rn(0.f);
  }
}

// Transposed block lists: one warp per (list set, key block n) scans the
// query blocks in 32-wide groups, ascending, and appends those whose list
// holds n (a block listed twice counts once). Deterministic: no atomics, fixed
// order. n_sets is 1 (lists shared by every (batch, head)) or batch * heads.
__global__ void transpose_lists_kernel(BwdArgs a, int n_kb, int n_sets) {
  const int64_t w = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = static_cast<int>(threadIdx.x & 31u);
  if (w >= static_cast<int64_t>(n_kb) * n_sets) return;  // whole warps
  const int64_t set = w / n_kb;
  const int n = static_cast<int>(w % n_kb);
  const int* cnt = a.kv_count + set * a.n_qb256;
  const int* idx = a.kv_index + set * a.n_qb256 * a.max_kv;
  int* q_index = const_cast<int*>(a.q_index) + w * a.n_qb256;
  int count = 0;
  for (int b0 = 0; b0 < a.n_qb256; b0 += 32) {
    const int b = b0 + lane;
    bool hit = false;
    if (b < a.n_qb256) {
      int c = cnt[b];
      c = c < 0 ? 0 : (c > a.max_kv ? a.max_kv : c);
      for (int j = 0; j < c && !hit; ++j) hit = idx[static_cast<int64_t>(b) * a.max_kv + j] == n;
    }
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    if (hit) q_index[count + __popc(m & ((1u << lane) - 1u))] = b;
    count += __popc(m);
  }
  if (lane == 0) const_cast<int*>(a.q_count)[w] = count;
}


}  // namespace bwd

cudaError_t launch_bwd_preprocess(int d_v, const BwdArgs& a, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.batch) * a.seqlen_q * a.heads;
  if (rows == 0) return cudaSuccess;
  const int64_t per_block = 8 * (d_v == 64 ? 4 : 2);  // 8 warps, each 32 / (d_v / 8) rows per pass
  const int64_t want = (rows + per_block - 1) / per_block;
  const int64_t blocks = want < 16384 ? want : 16384;
  if (d_v == 64) bwd::preprocess_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
  else if (d_v == 128) bwd::preprocess_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream) {
  if (a.kv_count != nullptr && (a.cu_q != nullptr || a.q_count == nullptr || a.q_index == nullptr))
    return cudaErrorInvalidValue;
  if (a.score_mod != kModNone) return launch_bwd_dkdv_mod(d_qk, d_v, tq, tk, tv, tdo, a, stream);
  if (a.kv_count != nullptr) {
    if (d_qk == 64 && d_v == 64) return bwd::launch_dkdv_t<64, 64, true>(tq, tk, tv, tdo, a, stream);
    if (d_qk == 128 && d_v == 128) return bwd::launch_dkdv_wide<true>(tq, tk, tv, tdo, a, stream);
    if (d_qk == 192 && d_v == 128) return bwd::launch_dkdv_t<192, 128, true>(tq, tk, tv, tdo, a, stream);
    return cudaErrorInvalidValue;
  }
  if (d_qk == 64 && d_v == 64) return bwd::launch_dkdv_t<64, 64, false>(tq, tk, tv, tdo, a, stream);
  if (d_qk == 128 && d_v == 128) return bwd::launch_dkdv_wide<false>(tq, tk, tv, tdo, a, stream);
  if (d_qk == 192 && d_v == 128) return bwd::launch_dkdv_t<192, 128, false>(tq, tk, tv, tdo, a, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_transpose_lists(const BwdArgs& a, int n_kb, cudaStream_t stream) {
  if (n_kb <= 0) return cudaSuccess;
  const int n_sets = a.lists_per_head ? a.batch * a.heads : 1;
  const int64_t threads = static_cast<int64_t>(n_kb) * n_sets * 32;
  const int64_t blocks = (threads + 255) / 256;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  bwd::transpose_lists_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a, n_kb, n_sets);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream) {
  if (a.kv_count != nullptr && a.cu_q != nullptr) return cudaErrorInvalidValue;
  if (a.score_mod != kModNone) return launch_bwd_dq_mod(d_qk, d_v, tq, tk, tv, tdo, a, stream);
  if (a.kv_count != nullptr) {
    if (d_qk == 64 && d_v == 64) return bwd::launch_dq_t<64, 64, true>(tq, tk, tv, tdo, a, stream);
    if (d_qk == 128 && d_v == 128) return bwd::launch_dq_t<128, 128, true>(tq, tk, tv, tdo, a, stream);
    if (d_qk == 192 && d_v == 128) return bwd::launch_dq_t<192, 128, true>(tq, tk, tv, tdo, a, stream);
    return cudaErrorInvalidValue;
  }
  if (d_qk == 64 && d_v == 64) return bwd::launch_dq_t<64, 64, false>(tq, tk, tv, tdo, a, stream);
  if (d_qk == 128 && d_v == 128) return bwd::launch_dq_t<128, 128, false>(tq, tk, tv, tdo, a, stream);
  if (d_qk == 192 && d_v == 128) return bwd::launch_dq_t<192, 128, false>(tq, tk, tv, tdo, a, stream);
  return cudaErrorInvalidValue;
}

namespace bwd {

// Split-key dQ: dQ (bf16, strided) = scale * sum_r dq_part[r], the ranges added
// in ascending order (so every call gives the same bits); one thread per 8
// elements of a (batch, head, row).
template <int D>
__global__ void dq_merge_kernel(const BwdArgs a) {
  constexpr int UPR = D / 8;
  const int64_t rows = static_cast<int64_t>(a.batch) * a.heads * a.seqlen_q;  // ((b * heads + h) * seqlen_q + row)
  const int64_t units = rows * UPR;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < units;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % UPR);
    const int64_t rh = i / UPR;
    const int row = static_cast<int>(rh % a.seqlen_q);
    const int64_t bh = rh / a.seqlen_q;
    const int h = static_cast<int>(bh % a.heads), b = static_cast<int>(bh / a.heads);
    const float* src = a.dq_part + rh * D + 8 * c;
    float4 x = __ldg(reinterpret_cast<const float4*>(src)), y = __ldg(reinterpret_cast<const float4*>(src) + 1);
    for (int r = 1; r < a.dq_split; ++r) {
      const float4* pr = reinterpret_cast<const float4*>(src + r * rows * D);
      const float4 u = __ldg(pr), w = __ldg(pr + 1);
      x = make_float4(x.x + u.x, x.y + u.y, x.z + u.z, x.w + u.w);
      y = make_float4(y.x + w.x, y.y + w.y, y.z + w.z, y.w + w.w);
    }
    const float sc = a.scale;
    const uint4 o = make_uint4(pack_bf16x2(x.x * sc, x.y * sc), pack_bf16x2(x.z * sc, x.w * sc),
                               pack_bf16x2(y.x * sc, y.y * sc), pack_bf16x2(y.z * sc, y.w * sc));
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dq) + b * a.dq_sb + static_cast<int64_t>(row) * a.dq_sn +
                         h * a.dq_sh + 8 * c;
    *reinterpret_cast<uint4*>(dst) = o;
  }
}

}  // namespace bwd

cudaError_t launch_bwd_dq_merge(const BwdArgs& a, int d_qk, cudaStream_t stream) {
  if (a.dq_split < 2 || a.dq_part == nullptr || a.cu_q != nullptr) return cudaErrorInvalidValue;
  const int64_t units = static_cast<int64_t>(a.batch) * a.heads * a.seqlen_q * (d_qk / 8);
  if (units == 0) return cudaSuccess;
  const int64_t want = (units + 255) / 256;
  const unsigned blocks = static_cast<unsigned>(want < 152 * 16 ? want : 152 * 16);
  if (d_qk == 64) bwd::dq_merge_kernel<64><<<blocks, 256, 0, stream>>>(a);
  else if (d_qk == 128) bwd::dq_merge_kernel<128><<<blocks, 256, 0, stream>>>(a);
  else if (d_qk == 192) bwd::dq_merge_kernel<192><<<blocks, 256, 0, stream>>>(a);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_bwd_zero(const BwdArgs& a, int d_qk, int d_v, bool zero_dq, bool zero_dkdv, cudaStream_t stream) {
  auto go = [&](void* p, int64_t sb, int64_t sn, int64_t sh, int nrows, int d) -> cudaError_t {
    const int64_t total = static_cast<int64_t>(a.batch) * nrows * a.heads;
    if (total == 0) return cudaSuccess;
    const int blocks = static_cast<int>(total / 256 + 1 < 4096 ? total / 256 + 1 : 4096);
    bwd::zero_kernel<<<blocks, 256, 0, stream>>>(p, sb, sn, sh, a.batch, nrows, a.heads, d);
    return cudaGetLastError();
  };
  cudaError_t e = cudaSuccess;
  if (zero_dq) e = go(a.dq, a.dq_sb, a.dq_sn, a.dq_sh, a.seqlen_q, d_qk);
  if (e == cudaSuccess && zero_dkdv) e = go(a.dk, a.dk_sb, a.dk_sn, a.dk_sh, a.seqlen_k, d_qk);
  if (e == cudaSuccess && zero_dkdv) e = go(a.dv, a.dv_sb, a.dv_sn, a.dv_sh, a.seqlen_k, d_v);
  return e;
}

}  // namespace gb300
