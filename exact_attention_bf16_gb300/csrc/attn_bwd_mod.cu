// Backward variants with a score modification (score_mod.cuh): the dK/dV and
// dQ kernels of bwd_kernels.cuh instantiated for soft-capping and ALiBi, dense
// or tile-list and block-sparse.
#include "bwd_kernels.cuh"

namespace gb300 {
namespace bwd {

template <int MOD, bool SPARSE>
cudaError_t dkdv_m(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                   const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream) {
  if (d_qk == 64 && d_v == 64) return launch_dkdv_t<64, 64, SPARSE, MOD>(tq, tk, tv, tdo, a, stream);
  if (d_qk == 128 && d_v == 128) return launch_dkdv_wide<SPARSE, MOD>(tq, tk, tv, tdo, a, stream);
  if (d_qk == 192 && d_v == 128) return launch_dkdv_t<192, 128, SPARSE, MOD>(tq, tk, tv, tdo, a, stream);
  return cudaErrorInvalidValue;
}

template <int MOD, bool SPARSE>
cudaError_t dq_m(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                 const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream) {
  if (d_qk == 64 && d_v == 64) return launch_dq_t<64, 64, SPARSE, MOD>(tq, tk, tv, tdo, a, stream);
  if (d_qk == 128 && d_v == 128) return launch_dq_t<128, 128, SPARSE, MOD>(tq, tk, tv, tdo, a, stream);
  if (d_qk == 192 && d_v == 128) return launch_dq_t<192, 128, SPARSE, MOD>(tq, tk, tv, tdo, a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace bwd

cudaError_t launch_bwd_dkdv_mod(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream) {
  const bool sp = a.kv_count != nullptr;
  switch (a.score_mod) {
    case kModSoftcap:
      return sp ? bwd::dkdv_m<kModSoftcap, true>(d_qk, d_v, tq, tk, tv, tdo, a, stream)
                : bwd::dkdv_m<kModSoftcap, false>(d_qk, d_v, tq, tk, tv, tdo, a, stream);
    case kModAlibi:
      return sp ? bwd::dkdv_m<kModAlibi, true>(d_qk, d_v, tq, tk, tv, tdo, a, stream)
                : bwd::dkdv_m<kModAlibi, false>(d_qk, d_v, tq, tk, tv, tdo, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_dq_mod(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream) {
  const bool sp = a.kv_count != nullptr;
  switch (a.score_mod) {
    case kModSoftcap:
      return sp ? bwd::dq_m<kModSoftcap, true>(d_qk, d_v, tq, tk, tv, tdo, a, stream)
                : bwd::dq_m<kModSoftcap, false>(d_qk, d_v, tq, tk, tv, tdo, a, stream);
    case kModAlibi:
      return sp ? bwd::dq_m<kModAlibi, true>(d_qk, d_v, tq, tk, tv, tdo, a, stream)
                : bwd::dq_m<kModAlibi, false>(d_qk, d_v, tq, tk, tv, tdo, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gb300
