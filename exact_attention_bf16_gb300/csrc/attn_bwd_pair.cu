// dK / dV over a pair of CTAs (d_qk = d_v = 128), the two-SM MMA of the
// backward pass (wittx "FlashAttention-4", section 反向传播的优化; newton wiki
// "FlashAttention-4", 核心技術): the two CTAs of a cluster run one MMA
// together, the accumulator split along M (keys) between them and the B
// operand (queries, or head dimensions) split along N, so that each SM keeps
// and reads only half of every B tile in its shared memory. That halves the
// B-operand reads per SM, which bound the one-SM kernel (dkdv_wide_kernel).
//
// A pair owns 256 consecutive keys, 128 per CTA (rank r: keys 256 p + 128 r);
// per step of 128 queries (all MMAs M = 256, N = 128, K = 16 per instruction):
//   S^T  = K Q^T     A = own K tile, B = Q rows [64 r, 64 r + 64) of the step
//   dP^T = V dO^T    A = own V tile, B = dO rows [64 r, 64 r + 64)
//   dV  += P^T dO    A = P^T in TMEM, B = dO columns [64 r, 64 r + 64), all rows
//   dK  += dS^T Q    A = dS^T in TMEM, B = Q columns [64 r, 64 r + 64), all rows
// so each CTA loads the step's Q and dO twice in halves (64 rows x 128
// columns for the N = query operand, 128 rows x 64 columns for the N = head
// dimension operand): the same 64 KB per step as the one-SM kernel.
//
// Roles per CTA (320 threads): warps 0..7 compute P^T and dS^T of their own
// 128 keys exactly as in the one-SM kernel (same TMEM regions, same 16x256b
// fragment layout), warp 8 issues the CTA's TMA copies, warp 9 of rank 0
// issues every MMA of the pair from one thread; warp 9 of rank 1 relays the
// completion of its CTA's copies to rank 0 (a remote mbarrier arrive), so rank
// 0's MMA thread waits for both halves of every operand.
//
// Cross-CTA signals: MMA completions are committed to the same barrier in both
// CTAs (multicast); the softmax warps of both CTAs arrive on rank 0's
// barriers. Every wait is bounded; both CTAs always reach the final cluster
// barrier before TMEM is released.
#include <cuda_bf16.h>

#include "bwd_common.cuh"
#include "kernels.h"
#include "ptx_sm100.cuh"

namespace gb300 {
namespace bwd {

struct DkdvPCfg {
  static constexpr int QB = 128, D = 128;
  static constexpr uint32_t tR0 = 0, tR1 = 128, tdV = 256, tdK = 384;
  static constexpr int TILE = 128 * 128 * 2;    // own K or V tile (32 KB, two 64-column chunks)
  static constexpr int ROWH = 64 * 128 * 2;     // 64 rows x 128 columns: two 8 KB chunks
  static constexpr int COLH = 128 * 64 * 2;     // 128 rows x 64 columns: one 16 KB chunk
  static constexpr int SLOT = ROWH + COLH;      // one Q or dO stage: [row half | column half]
  static constexpr int NQ = 3, NG = 2, NVEC = 2;
  static constexpr int OFF_K = 0, OFF_V = TILE, OFF_Q = 2 * TILE;
  static constexpr int OFF_G = OFF_Q + NQ * SLOT;
  static constexpr int OFF_VEC = OFF_G + NG * SLOT;  // [NVEC][2][QB] floats: -LSE*log2e, -D
  static constexpr int OFF_BAR = OFF_VEC + NVEC * 2 * QB * 4;
  static constexpr int SMEM = OFF_BAR + 256;         // the base is 1024-byte aligned (checked)
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct DkdvPBars {
  uint64_t kv_full, kv_full_peer;         // own K/V landed; rank 1's K/V landed (relayed)
  uint64_t q_full[3], q_full_peer[3], q_empty[3];
  uint64_t g_full[2], g_full_peer[2], g_empty[2];
  uint64_t v_full[2], v_empty[2];         // per CTA: the (-LSE*log2e, -D) vectors
  uint64_t s_full, dp_full, acc_full, mma_done;  // pair MMA commits (both CTAs)
  uint64_t sp_free, ds_full;              // rank 0: softmax warps of both CTAs
  uint32_t tmem_base;
};
static_assert(sizeof(DkdvPBars) <= 256, "pair barriers must fit their reserved bytes");

__device__ __forceinline__ bool wait_c_warp(uint64_t* bar, uint32_t parity, uint32_t* status, uint32_t where) {
  return __all_sync(0xffffffffu, mbar_wait_cluster(bar, parity, status, where));
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    dkdv_pair_kernel(const __grid_constant__ CUtensorMap tmq_r, const __grid_constant__ CUtensorMap tmq_c,
                     const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tmdo_r, const __grid_constant__ CUtensorMap tmdo_c,
                     const BwdArgs a) {
  using C = DkdvPCfg;
  constexpr int QB = C::QB;
  extern __shared__ __align__(1024) uint8_t smem_p[];
  if ((smem_u32(smem_p) & 1023u) != 0u) {  // same layout in both CTAs: both leave here, before any cluster barrier
    if (threadIdx.x == 0) record_error(a.status, DEV_BAD_CONFIG, 0x1800);
    return;
  }
  uint8_t* sK = smem_p + C::OFF_K;
  uint8_t* sV = smem_p + C::OFF_V;
  uint8_t* sQ = smem_p + C::OFF_Q;
  uint8_t* sG = smem_p + C::OFF_G;
  float* sVec = reinterpret_cast<float*>(smem_p + C::OFF_VEC);
  DkdvPBars* bar = reinterpret_cast<DkdvPBars*>(smem_p + C::OFF_BAR);

  const uint32_t rank = cluster_ctarank();
  // Pairs walk (unit, head) slowest and, within a head, the heaviest key
  // blocks (the first, under the causal mask) first.
  const int n_pair = (a.n_kblk + 1) / 2;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int bh = pair / n_pair;
  const int n = pair % n_pair;
  const int h = bh % a.heads;
  const Unit U = unit_bounds(a, bh / a.heads);
  const int kp = 256 * n;                            // the pair's first key
  if (kp >= U.nk) return;                            // pair-uniform: both CTAs leave together
  const int k0 = kp + 128 * static_cast<int>(rank);  // this CTA's first key
  int m_begin = 0;
  if (a.causal) {
    const int i_min = kp - (U.nk - U.nq);  // first query row that sees the pair's first key
    m_begin = i_min > 0 ? i_min / QB : 0;
  }
  const int m_end = ceil_div(U.nq, QB);
  const int T = m_end > m_begin ? m_end - m_begin : 0;  // the same in both CTAs
  auto q_row = [&](int t) -> int { return (m_begin + t) * QB; };

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(&bar->kv_full, 1);
    mbar_init(&bar->kv_full_peer, 1);
    for (int s = 0; s < C::NQ; ++s) {
      mbar_init(&bar->q_full[s], 1);
      mbar_init(&bar->q_full_peer[s], 1);
      mbar_init(&bar->q_empty[s], 1);
    }
    for (int s = 0; s < C::NG; ++s) {
      mbar_init(&bar->g_full[s], 1);
      mbar_init(&bar->g_full_peer[s], 1);
      mbar_init(&bar->g_empty[s], 1);
    }
    for (int s = 0; s < C::NVEC; ++s) {
      mbar_init(&bar->v_full[s], 32);
      mbar_init(&bar->v_empty[s], kSoftThreads / 32);
    }
    mbar_init(&bar->s_full, 1);
    mbar_init(&bar->dp_full, 1);
    mbar_init(&bar->acc_full, 1);
    mbar_init(&bar->mma_done, 1);
    mbar_init(&bar->sp_free, 2 * kSoftThreads / 32);  // eight warps in each CTA
    mbar_init(&bar->ds_full, 2 * kSoftThreads / 32);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {  // one warp of each CTA allocates the pair's TMEM together
    tmem_alloc_pair(&bar->tmem_base, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tbase = bar->tmem_base;
  auto region = [](int t) { return (t & 1) ? C::tR1 : C::tR0; };  // R(t): S^T(t), then P^T/dS^T(t)
  auto other = [](int t) { return (t & 1) ? C::tR0 : C::tR1; };   // R'(t): dP^T(t)

  if (warp == kTmaWarp) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar->kv_full, 2 * C::TILE);
      for (int c = 0; c < 2; ++c) tma_load_4d(sK + c * KB * 128, &tmk, &bar->kv_full, c * 64, h, U.k_start + k0, U.b);
      for (int c = 0; c < 2; ++c) tma_load_4d(sV + c * KB * 128, &tmv, &bar->kv_full, c * 64, h, U.k_start + k0, U.b);
    }
    int nq_issued = 0, ng_issued = 0;
    bool ok = true;
    const int rh = 64 * static_cast<int>(rank);  // this CTA's row half and column half
    for (int t = 0; t < T && ok; ++t) {
      const int tile = q_row(t);
      const int row = U.q_start + tile;
      float nl[QB / 32], nd[QB / 32];
#pragma unroll
      for (int u = 0; u < QB / 32; ++u) {
        const int r = static_cast<int>(lane) + 32 * u;
        nl[u] = -INFINITY;  // rows past the end: P = 0
        nd[u] = 0.f;
        if (tile + r < U.nq) {
          const int64_t idx = U.b * a.lse_sb + h * a.lse_sh + U.q_start + tile + r;
          const float l = a.lse[idx];
          nl[u] = (l == -INFINITY) ? -INFINITY : -l * 1.4426950408889634f;
          nd[u] = -a.dsum[idx];
        }
      }
      const int qs = t % C::NQ, gs = t % C::NG, vs = t % C::NVEC;
      ok = mbar_wait_cluster(&bar->q_empty[qs], (static_cast<uint32_t>(t / C::NQ) & 1u) ^ 1u, a.status, 0x1800 + qs);
      if (!ok) break;
      if (lane == 0) {
        uint8_t* dst = sQ + qs * C::SLOT;
        mbar_arrive_expect_tx(&bar->q_full[qs], C::SLOT);
        for (int c = 0; c < 2; ++c) tma_load_4d(dst + c * (C::ROWH / 2), &tmq_r, &bar->q_full[qs], c * 64, h, row + rh, U.b);
        tma_load_4d(dst + C::ROWH, &tmq_c, &bar->q_full[qs], rh, h, row, U.b);
      }
      ++nq_issued;
      ok = mbar_wait_cluster(&bar->g_empty[gs], (static_cast<uint32_t>(t / C::NG) & 1u) ^ 1u, a.status, 0x1808 + gs);
      if (!ok) break;
      if (lane == 0) {
        uint8_t* dst = sG + gs * C::SLOT;
        mbar_arrive_expect_tx(&bar->g_full[gs], C::SLOT);
        for (int c = 0; c < 2; ++c)
          tma_load_4d(dst + c * (C::ROWH / 2), &tmdo_r, &bar->g_full[gs], c * 64, h, row + rh, U.b);
        tma_load_4d(dst + C::ROWH, &tmdo_c, &bar->g_full[gs], rh, h, row, U.b);
      }
      ++ng_issued;
      ok = mbar_wait(&bar->v_empty[vs], (static_cast<uint32_t>(t / C::NVEC) & 1u) ^ 1u, a.status, 0x1810 + vs);
      if (!ok) break;
      float* vec = sVec + vs * 2 * QB;
#pragma unroll
      for (int u = 0; u < QB / 32; ++u) {
        vec[lane + 32 * u] = nl[u];
        vec[QB + lane + 32 * u] = nd[u];
      }
      mbar_arrive(&bar->v_full[vs]);
    }
    if (lane == 0) {
      if (!ok) {  // let the copies in flight land before the CTA leaves
        for (int t = nq_issued - 1; t >= 0 && t >= nq_issued - C::NQ; --t)
          mbar_wait(&bar->q_full[t % C::NQ], static_cast<uint32_t>(t / C::NQ) & 1u, nullptr, 0);
        for (int t = ng_issued - 1; t >= 0 && t >= ng_issued - C::NG; --t)
          mbar_wait(&bar->g_full[t % C::NG], static_cast<uint32_t>(t / C::NG) & 1u, nullptr, 0);
      }
      mbar_wait(&bar->kv_full, 0, nullptr, 0);
    }
  } else if (warp == kMmaWarp && rank == 1) {
    // ---- relay: tell rank 0 when this CTA's halves of each operand landed
    if (lane == 0) {
      bool ok = mbar_wait(&bar->kv_full, 0, a.status, 0x1820);
      if (ok) mbar_arrive_cluster(&bar->kv_full_peer, 0);
      for (int t = 0; t < T && ok; ++t) {
        ok = mbar_wait(&bar->q_full[t % C::NQ], static_cast<uint32_t>(t / C::NQ) & 1u, a.status, 0x1821);
        if (!ok) break;
        mbar_arrive_cluster(&bar->q_full_peer[t % C::NQ], 0);
        ok = mbar_wait(&bar->g_full[t % C::NG], static_cast<uint32_t>(t / C::NG) & 1u, a.status, 0x1822);
        if (!ok) break;
        mbar_arrive_cluster(&bar->g_full_peer[t % C::NG], 0);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---- rank 0: the pair's MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(256, QB, false, false);  // S^T, dP^T: B = Q / dO rows, K-major
      constexpr uint32_t idA = idesc_bf16_f32(256, 128, false, true);  // dV, dK: B = dO / Q columns, MN-major
      const uint64_t dKd = smem_desc(smem_u32(sK), 16, 1024, SWZ_128B);
      const uint64_t dVd = smem_desc(smem_u32(sV), 16, 1024, SWZ_128B);
      auto q_slot = [&](int t) { return smem_u32(sQ + (t % C::NQ) * C::SLOT); };
      auto g_slot = [&](int t) { return smem_u32(sG + (t % C::NG) * C::SLOT); };
      auto q_ready = [&](int t) {
        const uint32_t ph = static_cast<uint32_t>(t / C::NQ) & 1u;
        return mbar_wait(&bar->q_full[t % C::NQ], ph, a.status, 0x1830) &&
               mbar_wait_cluster(&bar->q_full_peer[t % C::NQ], ph, a.status, 0x1831);
      };
      auto g_ready = [&](int t) {
        const uint32_t ph = static_cast<uint32_t>(t / C::NG) & 1u;
        return mbar_wait(&bar->g_full[t % C::NG], ph, a.status, 0x1832) &&
               mbar_wait_cluster(&bar->g_full_peer[t % C::NG], ph, a.status, 0x1833);
      };
      // A: 128 key rows per CTA, 64-column chunks 16 KB apart; B row half:
      // 64 query rows per CTA, chunks 8 KB apart
      auto issue_s = [&](int t) {  // S^T(t) = K Q^T -> R(t)
        const uint64_t bq = smem_desc(q_slot(t), 16, 1024, SWZ_128B);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss_pair(tbase + region(t), desc_add(dKd, (kk / 4) * KB * 128 + (kk % 4) * 32),
                      desc_add(bq, (kk / 4) * (C::ROWH / 2) + (kk % 4) * 32), idS, kk > 0 ? 1u : 0u);
      };
      auto issue_dp = [&](int t) {  // dP^T(t) = V dO^T -> R'(t)
        const uint64_t bg = smem_desc(g_slot(t), 16, 1024, SWZ_128B);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss_pair(tbase + other(t), desc_add(dVd, (kk / 4) * KB * 128 + (kk % 4) * 32),
                      desc_add(bg, (kk / 4) * (C::ROWH / 2) + (kk % 4) * 32), idS, kk > 0 ? 1u : 0u);
      };
      bool ok = mbar_wait(&bar->kv_full, 0, a.status, 0x1838) &&
                mbar_wait_cluster(&bar->kv_full_peer, 0, a.status, 0x1839);
      if (ok && T > 0) {
        ok = q_ready(0);
        if (ok) {
          tc_fence_after();
          issue_s(0);
          mma_commit_pair(&bar->s_full);
          ok = g_ready(0);
        }
        if (ok) {
          tc_fence_after();
          issue_dp(0);
          mma_commit_pair(&bar->dp_full);
        }
      }
      for (int t = 0; t < T && ok; ++t) {
        if (t + 1 < T) {  // S^T(t+1) into R'(t) once both CTAs' softmax warps hold dP^T(t)
          ok = mbar_wait_cluster(&bar->sp_free, static_cast<uint32_t>(t) & 1u, a.status, 0x1840) && q_ready(t + 1);
          if (!ok) break;
          tc_fence_after();
          issue_s(t + 1);
          mma_commit_pair(&bar->s_full);
        }
        ok = mbar_wait_cluster(&bar->ds_full, static_cast<uint32_t>(t) & 1u, a.status, 0x1841);
        if (!ok) break;
        tc_fence_after();
        // dV += P^T dO and dK += dS^T Q: A from R(t) (k-step kk = 16 queries of
        // warpgroup kk / 4: P^T in its first 32 columns, dS^T in the last 32),
        // B = this CTA's 64-column half of the step's dO / Q rows, MN-major
        const uint64_t mg = smem_desc(g_slot(t) + C::ROWH, C::COLH, 1024, SWZ_128B);
        const uint64_t mq = smem_desc(q_slot(t) + C::ROWH, C::COLH, 1024, SWZ_128B);
        const uint32_t acc0 = t > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < QB / 16; ++kk) {
          const uint32_t pa = tbase + region(t) + 64 * (kk / 4) + 8 * (kk % 4);
          mma_ts_pair(tbase + C::tdV, pa, desc_add(mg, kk * 2048), idA, kk > 0 ? 1u : acc0);
        }
        mma_commit_pair(&bar->g_empty[t % C::NG]);
#pragma unroll
        for (int kk = 0; kk < QB / 16; ++kk) {
          const uint32_t da = tbase + region(t) + 64 * (kk / 4) + 32 + 8 * (kk % 4);
          mma_ts_pair(tbase + C::tdK, da, desc_add(mq, kk * 2048), idA, kk > 0 ? 1u : acc0);
        }
        mma_commit_pair(&bar->q_empty[t % C::NQ]);
        if (t + 1 < T) {  // dP^T(t+1) into R(t), after the reads above in issue order
          ok = g_ready(t + 1);
          if (!ok) break;
          tc_fence_after();
          issue_dp(t + 1);
          mma_commit_pair(&bar->dp_full);
        }
      }
      mma_commit_pair(&bar->acc_full);
      mma_commit_pair(&bar->mma_done);
      mbar_wait(&bar->mma_done, 0, a.status, 0x18ff);
    }
  } else if (warp < kTmaWarp) {
    // ================= softmax gradient (each CTA: its own 128 keys) =========
    // The same fragment layout and arithmetic as dkdv_wide_kernel.
    const int wg = static_cast<int>(warp) / 4;
    const uint32_t quarter = warp & 3u;
    const int g = static_cast<int>(lane >> 2), c = static_cast<int>(lane & 3u);
    int vis[2][2];
    bool kok[2][2];
#pragma unroll
    for (int lg = 0; lg < 2; ++lg)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int kj = k0 + static_cast<int>(quarter) * 32 + 16 * lg + 8 * hh + g;
        vis[lg][hh] = a.causal ? kj - (U.nk - U.nq) : -0x40000000;
        kok[lg][hh] = kj < U.nk;
      }
    const bool all_keys = kok[0][0] && kok[0][1] && kok[1][0] && kok[1][1];
    const int vis_max = max(max(vis[0][0], vis[0][1]), max(vis[1][0], vis[1][1]));
    const float2 sl2v = make_float2(a.scale_log2, a.scale_log2);
    auto lanes = [&](int lg) { return tbase + ((quarter * 32u + 16u * static_cast<uint32_t>(lg)) << 16); };
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      const int q0 = q_row(t) + 64 * wg;
      const uint32_t col = region(t) + 64 * wg;
      // ---- phase A: P from S^T(t), written over S^T(t) as bf16 P^T
      ok = wait_c_warp(&bar->s_full, static_cast<uint32_t>(t) & 1u, a.status, 0x1850) &&
           mbar_wait_warp(&bar->v_full[t % C::NVEC], static_cast<uint32_t>(t / C::NVEC) & 1u, a.status, 0x1851);
      if (!ok) break;
      tc_fence_after();
      const float* vL = sVec + (t % C::NVEC) * 2 * QB + 64 * wg + 2 * c;
      const float* vD = vL + QB;
      const bool full = all_keys && q0 >= vis_max;
      float2 nlv[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) nlv[r] = *reinterpret_cast<const float2*>(vL + 8 * r);
      float p[2][32];
#pragma unroll
      for (int lg = 0; lg < 2; ++lg) {
        uint32_t sv[32], pw[16];
        tmem_ld16x256b_x8(lanes(lg) + col, sv);
        tmem_wait_ld();
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float2 nl = nlv[r];
          const float2 x0 = ffma2(make_float2(__uint_as_float(sv[4 * r]), __uint_as_float(sv[4 * r + 1])), sl2v, nl);
          const float2 x1 = ffma2(make_float2(__uint_as_float(sv[4 * r + 2]), __uint_as_float(sv[4 * r + 3])), sl2v, nl);
          float* pp = &p[lg][4 * r];
          pp[0] = ex2_mufu(x0.x);
          pp[1] = ex2_mufu(x0.y);
          pp[2] = ex2_mufu(x1.x);
          pp[3] = ex2_mufu(x1.y);
          if (!full) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int qi = q0 + 8 * r + 2 * c + (u & 1);
              if (!(kok[lg][u >> 1] && qi >= vis[lg][u >> 1])) pp[u] = 0.f;
            }
          }
          pw[2 * r] = pack_bf16x2(pp[0], pp[1]);
          pw[2 * r + 1] = pack_bf16x2(pp[2], pp[3]);
        }
        tmem_st16x128b_x8(lanes(lg) + col, pw);
      }
      // ---- phase B: dS = P (dP - D) from dP^T(t), written next to P^T
      ok = wait_c_warp(&bar->dp_full, static_cast<uint32_t>(t) & 1u, a.status, 0x1852);
      if (!ok) break;
      tc_fence_after();
      uint32_t dp[2][32];
      tmem_ld16x256b_x8(lanes(0) + other(t) + 64 * wg, dp[0]);
      tmem_ld16x256b_x8(lanes(1) + other(t) + 64 * wg, dp[1]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(&bar->sp_free, 0);
      float2 ndv[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) ndv[r] = *reinterpret_cast<const float2*>(vD + 8 * r);
#pragma unroll
      for (int lg = 0; lg < 2; ++lg) {
        uint32_t dw[16];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float2 nd = ndv[r];
          const float2 d0 = fmul2(make_float2(p[lg][4 * r], p[lg][4 * r + 1]),
                                  fadd2(make_float2(__uint_as_float(dp[lg][4 * r]), __uint_as_float(dp[lg][4 * r + 1])), nd));
          const float2 d1 = fmul2(make_float2(p[lg][4 * r + 2], p[lg][4 * r + 3]),
                                  fadd2(make_float2(__uint_as_float(dp[lg][4 * r + 2]), __uint_as_float(dp[lg][4 * r + 3])), nd));
          dw[2 * r] = pack_bf16x2(d0.x, d0.y);
          dw[2 * r + 1] = pack_bf16x2(d1.x, d1.y);
        }
        tmem_st16x128b_x8(lanes(lg) + col + 32, dw);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_cluster(&bar->ds_full, 0);
        mbar_arrive(&bar->v_empty[t % C::NVEC]);
      }
    }
    // ---- epilogue: warpgroup 0 writes dV, warpgroup 1 writes scale * dK (one key row per thread)
    if (ok && T > 0) {
      ok = wait_c_warp(&bar->acc_full, 0, a.status, 0x1860);
      tc_fence_after();
    }
    const int kj = k0 + static_cast<int>(quarter * 32 + lane);
    const uint32_t lane_base = tbase + ((quarter * 32u) << 16);
    const bool store = kj < U.nk;
    __nv_bfloat16* dst = wg == 0 ? static_cast<__nv_bfloat16*>(a.dv) + U.b * a.dv_sb +
                                       static_cast<int64_t>(U.k_start + kj) * a.dv_sn + h * a.dv_sh
                                 : static_cast<__nv_bfloat16*>(a.dk) + U.b * a.dk_sb +
                                       static_cast<int64_t>(U.k_start + kj) * a.dk_sn + h * a.dk_sh;
    const uint32_t acc = wg == 0 ? C::tdV : C::tdK;
    const float mul = wg == 0 ? 1.f : a.scale;
#pragma unroll
    for (int cc = 0; cc < C::D / 32; ++cc) {
      uint32_t v[32], w[16];
      if (T > 0) {
        tmem_ld32(lane_base + acc + cc * 32, v);
        tmem_wait_ld();
      }
#pragma unroll
      for (int e = 0; e < 16; ++e)
        w[e] = T > 0 ? pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul) : 0u;
      if (store) store_row_bf16(dst + cc * 32, w);
    }
  }

  // Neither CTA may release TMEM or leave while the other's MMAs, remote
  // arrivals or reads of its memory can still be in flight.
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc_pair(tbase, 512);
}

}  // namespace bwd

cudaError_t launch_bwd_dkdv_pair(const CUtensorMap& tq_r, const CUtensorMap& tq_c, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo_r, const CUtensorMap& tdo_c,
                                 const BwdArgs& a, cudaStream_t stream) {
  using namespace bwd;
  // block-sparse lists use the one-SM kernel; a packed batch's pairs are decoded from the grid
  if (a.kv_count != nullptr || a.tiles_kv != nullptr) return cudaErrorInvalidValue;
  static PerDeviceOnce once;
  cudaError_t e = once.run([] {
    return cudaFuncSetAttribute(dkdv_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DkdvPCfg::SMEM);
  });
  if (e != cudaSuccess) return e;
  const int64_t grid = 2 * static_cast<int64_t>((a.n_kblk + 1) / 2) * a.num_units * a.heads;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  dkdv_pair_kernel<<<static_cast<unsigned>(grid), kThreads, DkdvPCfg::SMEM, stream>>>(tq_r, tq_c, tk, tv, tdo_r,
                                                                                     tdo_c, a);
  return cudaGetLastError();
}

}  // namespace gb300
