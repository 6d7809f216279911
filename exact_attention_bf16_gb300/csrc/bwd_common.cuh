// Pieces shared by the backward kernels (bwd_kernels.cuh, attn_bwd_pair.cu):
// tile sizes, warp roles, row stores and the bounds of a work unit.
#pragma once
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx_sm100.cuh"

namespace gb300 {
namespace bwd {

constexpr int KB = 128;          // keys per kv tile (TMEM lanes in dkdv)
constexpr int MB = 128;          // queries per q tile in the dq kernel
constexpr int kThreads = 320;    // 8 softmax warps + TMA warp + MMA warp
constexpr int kTmaWarp = 8, kMmaWarp = 9;
constexpr int kSoftThreads = 256;

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const uint32_t (&w)[16]) { store_row64(dst, w); }

// Sequence bounds of a work unit (dense: unit = batch index; varlen: b = 0 and
// unit = the sequence).
struct Unit {
  int b, q_start, k_start, nq, nk, unit;
};
__device__ __forceinline__ Unit unit_bounds(const BwdArgs& a, int unit) {
  Unit u{unit, 0, 0, a.seqlen_q, a.seqlen_k, unit};
  if (a.cu_q != nullptr) {
    u.b = 0;
    u.q_start = a.cu_q[unit];
    u.nq = a.cu_q[unit + 1] - u.q_start;
    u.k_start = a.cu_k[unit];
    u.nk = a.cu_k[unit + 1] - u.k_start;
  }
  return u;
}

// A backward CTA's work: from the tile list of a packed variable-length
// launch (`tiles` non-null), else from the block index over nblk blocks per
// (unit, head), blocks in descending (dQ: the last query blocks are the
// heaviest under the causal mask) or ascending (dK/dV: the first key blocks)
// order. Returns false for an empty list entry (the CTA has no work).
// slot: the work item (blockIdx.x unless the kernel launches several CTAs per item).
__device__ __forceinline__ bool bwd_work(const BwdArgs& a, const TileEntry* tiles, int nblk, bool descending,
                                         Unit& U, int& h, int& blk, int slot = -1) {
  if (slot < 0) slot = static_cast<int>(blockIdx.x);
  if (tiles != nullptr) {
    const int4* te = reinterpret_cast<const int4*>(tiles + slot);
    const int4 t0 = __ldg(te), t1 = __ldg(te + 1);
    if (t1.z < 0) return false;
    U = Unit{0, t0.x, t0.z, t0.y, t0.w, t1.z};
    h = t1.x;
    blk = t1.y;
    return true;
  }
  const GridSlot g = grid_slot(slot, a.num_units * a.heads, nblk, a.n_groups);
  const int bh = g.pair;
  blk = descending ? nblk - 1 - g.rank : g.rank;
  h = bh % a.heads;
  U = unit_bounds(a, bh / a.heads);
  return true;
}

}  // namespace bwd
}  // namespace gb300
