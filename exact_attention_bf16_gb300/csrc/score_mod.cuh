// Score modifications (the FlexAttention variants built on FA4 of wittx
// "FlashAttention-4", section Python写GPU内核; newton wiki "FlashAttention-4",
// 發展歷程), applied by the forward and backward kernels to the raw logit
// s = q . k of a visible (query i, key j) pair before the softmax. The scaled
// logit is a = scale * s; each modification maps it to a', and the kernels keep
// working in raw units s' = a' / scale:
//   kModSoftcap: a' = c tanh(a / c), so s' = mod_b tanh(mod_a s) with
//                mod_a = scale / c, mod_b = c / scale; its derivative
//                da'/da = 1 - tanh^2 multiplies dS in the backward.
//   kModAlibi:   a' = a - m_h |j - (i + Nk - Nq)|, so s' = s - |slope (j - qpos)|
//                with slope = m_h / scale and qpos = i + Nk - Nq (the query's
//                position, aligned bottom-right like the causal mask).
// tanh is evaluated as 1 - 2 / (1 + e^(2x)): one hardware exp2 (relative error
// about 2^-22) and one hardware reciprocal, exact to a few fp32 ulps of 1.
#pragma once
#include "ptx_sm100.cuh"

namespace gb300 {

enum : int { kModNone = 0, kModSoftcap = 1, kModAlibi = 2 };

__device__ __forceinline__ float rcp_mufu(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tanh(mod_a * s) with k2 = 2 log2(e) mod_a.
__device__ __forceinline__ float tanh_scaled(float s, float k2) {
  return fmaf(-2.f, rcp_mufu(1.f + ex2_mufu(k2 * s)), 1.f);
}

}  // namespace gb300
