// Forward with FP8 E4M3 inputs (the FP8 path of FA3 and the lower precisions
// named for later versions: ainexis "Tri Dao FlashAttention-4", 背景; wittx
// "FlashAttention-4", closing section): S = Q K^T on the tensor core's 8-bit
// kind (twice the bf16 rate), P and V in fp16 for PV as in the bf16 forward,
// so the result carries no error beyond the bf16 path's. V is converted here
// once per call, exactly: every E4M3 value is an fp16 value.
#include <cstdint>

#include "fwd_kernel.cuh"

namespace gb300 {
namespace fwd {

// Two E4M3 codes (low byte = first) to two fp16 values (low half = first).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t x) {
  uint32_t y;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(y) : "h"(x));
  return y;
}

// One warp per token row; each lane converts 16-byte units (16 codes) into
// 32 bytes of fp16. Output layout: contiguous [rows, heads, DV] fp16.
template <int DV>
__global__ void v_e4m3_to_f16_kernel(const uint8_t* v, int64_t sb, int64_t sn, int64_t sh, int nb, int nrows,
                                     int heads, uint4* out) {
  constexpr int UPH = DV / 16;  // 16-byte input units per (row, head)
  const int upr = heads * UPH;
  const int64_t rows = static_cast<int64_t>(nb) * nrows;
  const int lane = static_cast<int>(threadIdx.x & 31u);
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; r < rows; r += nwarps) {
    const int b = static_cast<int>(r / nrows), n = static_cast<int>(r % nrows);
    const uint8_t* src = v + b * sb + n * sn;
    uint4* dst = out + r * upr * 2;
    for (int i = lane; i < upr; i += 32) {
      const uint4 x = *reinterpret_cast<const uint4*>(src + (i / UPH) * sh + 16 * (i % UPH));
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
      uint32_t o[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o[2 * e] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[e] & 0xFFFFu));
        o[2 * e + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[e] >> 16));
      }
      dst[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
}

}  // namespace fwd

cudaError_t launch_fwd_e4m3(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv16, const FwdArgs& a,
                            cudaStream_t stream) {
  if (!a.input_e4m3 || a.emu_period != 0 || a.score_mod != kModNone || a.kv_count != nullptr) return cudaErrorInvalidValue;
  if (a.tiles != nullptr)
    return fwd::launch_e<128, 128, 0, false, false, true, kModNone, true>(tq, tk, tv16, tv16, a, stream);
  return fwd::launch_e<128, 128, 0, false, false, false, kModNone, true>(tq, tk, tv16, tv16, a, stream);
}

cudaError_t launch_v_e4m3_to_f16(const void* v, int64_t sb, int64_t sn, int64_t sh, int nb, int nrows, int heads,
                                 int dv, void* out, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(nb) * nrows;
  if (rows == 0) return cudaSuccess;
  if (dv != 128) return cudaErrorInvalidValue;
  const int64_t want = (rows + 7) / 8;  // 8 warps (rows) per block and pass
  const unsigned blocks = static_cast<unsigned>(want < 152 * 8 ? want : 152 * 8);
  fwd::v_e4m3_to_f16_kernel<128><<<blocks, 256, 0, stream>>>(static_cast<const uint8_t*>(v), sb, sn, sh, nb, nrows,
                                                             heads, static_cast<uint4*>(out));
  return cudaGetLastError();
}

}  // namespace gb300
