// Forward variants with a score modification (score_mod.cuh): the kernel of
// fwd_kernel.cuh instantiated for soft-capping and ALiBi, dense, tile-list
// (packed variable length) and block-sparse, exp2 on the hardware unit only.
#include "fwd_kernel.cuh"

namespace gb300 {
namespace fwd {

template <int DQK, int DV, int MOD>
cudaError_t launch_m(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tv16,
                     const FwdArgs& a, cudaStream_t stream) {
  if (a.emu_period != 0) return cudaErrorInvalidValue;
  if (a.kv_count != nullptr) return launch_e<DQK, DV, 0, true, false, false, MOD>(tq, tk, tv, tv16, a, stream);
  if (a.tiles != nullptr) return launch_e<DQK, DV, 0, false, false, true, MOD>(tq, tk, tv, tv16, a, stream);
  return launch_e<DQK, DV, 0, false, false, false, MOD>(tq, tk, tv, tv16, a, stream);
}

template <int MOD>
cudaError_t launch_d(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const CUtensorMap& tv16, const FwdArgs& a, cudaStream_t stream) {
  if (d_qk == 64 && d_v == 64) return launch_m<64, 64, MOD>(tq, tk, tv, tv16, a, stream);
  if (d_qk == 128 && d_v == 128) return launch_m<128, 128, MOD>(tq, tk, tv, tv16, a, stream);
  if (d_qk == 192 && d_v == 128) return launch_m<192, 128, MOD>(tq, tk, tv, tv16, a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fwd

cudaError_t launch_fwd_mod(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tv16, const FwdArgs& a, cudaStream_t stream) {
  switch (a.score_mod) {
    case kModSoftcap: return fwd::launch_d<kModSoftcap>(d_qk, d_v, tq, tk, tv, tv16, a, stream);
    case kModAlibi: return fwd::launch_d<kModAlibi>(d_qk, d_v, tq, tk, tv, tv16, a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gb300
