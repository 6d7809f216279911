// Single-pass backward for d_qk = d_v = 64 (the design of wittx
// "FlashAttention-4", 反向传播的优化): one key-stationary kernel produces dK,
// dV and, per 64-query step, the dQ partial dS K, which its softmax warps add
// into an fp32 dQ buffer in L2 (red.global.add); in deterministic mode the
// adds to each 64-row query tile are ordered by key tile through a semaphore
// per tile. A last pass writes dQ * scale in bf16.
#include <cuda_bf16.h>

#include "bwd_kernels.cuh"

namespace gb300 {
namespace bwd {

// dQ (bf16, strided) = scale * dq_acc ([units][heads][rows][D] fp32); one
// thread per 8 elements.
template <int D>
__global__ void dq_convert_kernel(const BwdArgs a) {
  constexpr int UPR = D / 8;  // 8-element units per (row, head)
  const int64_t units = static_cast<int64_t>(a.batch) * a.heads * a.seqlen_q * UPR;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < units;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % UPR);
    const int64_t rh = i / UPR;  // ((b * heads + h) * rows + row)
    const int row = static_cast<int>(rh % a.seqlen_q);
    const int64_t bh = rh / a.seqlen_q;
    const int h = static_cast<int>(bh % a.heads), b = static_cast<int>(bh / a.heads);
    const float4* src = reinterpret_cast<const float4*>(a.dq_acc + rh * D + 8 * c);
    const float4 x = src[0], y = src[1];
    const uint4 w = make_uint4(pack_bf16x2(x.x * a.scale, x.y * a.scale), pack_bf16x2(x.z * a.scale, x.w * a.scale),
                               pack_bf16x2(y.x * a.scale, y.y * a.scale), pack_bf16x2(y.z * a.scale, y.w * a.scale));
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dq) + b * a.dq_sb + static_cast<int64_t>(row) * a.dq_sn +
                         h * a.dq_sh + 8 * c;
    *reinterpret_cast<uint4*>(dst) = w;
  }
}

}  // namespace bwd

cudaError_t launch_bwd_single_pass(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                   const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream) {
  if (a.dq_acc == nullptr || a.kv_count != nullptr || a.score_mod != kModNone) return cudaErrorInvalidValue;
  return bwd::launch_dkdv_t<64, 64, false, kModNone, true>(tq, tk, tv, tdo, a, stream);
}

cudaError_t launch_bwd_dq_convert(const BwdArgs& a, int d, cudaStream_t stream) {
  if (d != 64 || a.dq_acc == nullptr) return cudaErrorInvalidValue;
  const int64_t units = static_cast<int64_t>(a.batch) * a.heads * a.seqlen_q * (64 / 8);
  if (units == 0) return cudaSuccess;
  const int64_t want = (units + 255) / 256;
  const unsigned blocks = static_cast<unsigned>(want < 152 * 16 ? want : 152 * 16);
  bwd::dq_convert_kernel<64><<<blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace gb300
