// Backward attention kernels for GB300 (sm_103a).
//
// Gradients of the loss <O, dO> (dQ, dK, dV; wittx "FlashAttention-4",
// section 反向传播的优化) with P recomputed from the forward's LSE:
//   P = 2^(scale*log2e * Q K^T - LSE*log2e),  dP = dO V^T,  D_i = dO_i . O_i,
//   dS = P * (dP - D),  dV = P^T dO,  dK = scale * dS^T Q,  dQ = scale * dS K.
//
// Three launches:
//   preprocess  D_i = sum_d dO_id O_id (fp32) into the workspace.
//   dkdv        one CTA per 128-key tile (K, V stay in shared memory), looping
//               over query tiles: S^T = K Q^T and dP^T = V dO^T into Tensor
//               Memory, P^T / dS^T computed one key row per thread, then
//               dV += P^T dO (P^T read straight from TMEM) and dK += dS^T Q
//               with both accumulators resident in TMEM for the whole loop.
//   dq          one CTA per 128-query tile (Q, dO stay in shared memory),
//               looping over key tiles: S, dP, dS as above, dQ += dS K in TMEM.
// Every output element is produced by exactly one CTA with a fixed summation
// order, so results are bitwise reproducible run to run (the deterministic
// mode costs nothing here). This trades the pages' single-pass design (dQ
// partials reduced across CTAs with global atomics, or semaphore-ordered adds
// in deterministic mode) for two extra GEMMs per tile pair (S and dP are
// recomputed by the dq kernel) and no atomics at all.
//
// Roles: warps 0..7 are two softmax-gradient warpgroups (each TMEM lane =
// one row, the two groups split the columns), warp 8 issues TMA copies,
// warp 9 allocates TMEM and issues every tcgen05.mma from one thread.
//
// This header holds the dK/dV and dQ kernel templates and their launch
// templates; attn_bwd.cu instantiates them without a score modification,
// attn_bwd_mod.cu with one, attn_bwd_fused.cu the single-pass d = 64 kernel.
#pragma once
#include <cuda_bf16.h>

#include "bwd_common.cuh"
#include "kernels.h"
#include "ptx_sm100.cuh"
#include "score_mod.cuh"

namespace gb300 {
namespace bwd {

// Copies row `row` of a K-major 128-byte-swizzled tile (64-column chunks
// `chunk_bytes` apart) into registers as packed bf16 pairs: 32 words per chunk.
__device__ __forceinline__ void smem_row_chunk(const uint8_t* tile, int chunk_bytes, int row, int chunk,
                                               uint32_t (&w)[32]) {
  const uint8_t* base = tile + chunk * chunk_bytes + row * 128;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint4 v = *reinterpret_cast<const uint4*>(base + ((u ^ (row & 7)) * 16));
    w[4 * u] = v.x;
    w[4 * u + 1] = v.y;
    w[4 * u + 2] = v.z;
    w[4 * u + 3] = v.w;
  }
}

// Stores this thread's row of a 128-row operand tile (d columns) into TMEM as
// an MMA A operand: lane = row, column c = elements (2c, 2c+1).
__device__ __forceinline__ void tile_row_to_tmem(const uint8_t* tile, int chunks, int row, uint32_t taddr) {
  for (int c = 0; c < chunks; ++c) {
    uint32_t w[32];
    smem_row_chunk(tile, KB * 128, row, c, w);
    tmem_st32(taddr + 32 * c, w);
  }
}

// ===========================================================================
// dK / dV kernel (key-stationary)
// ===========================================================================
// Per step one 64-row query tile. S^T = K Q^T and dP^T = V dO^T go to TMEM;
// the softmax warps turn them into P^T and dS^T (bf16 pairs) in a TMEM region
// of their own, which feeds dV += P^T dO and dK += dS^T Q directly. Because
// P^T/dS^T do not overwrite S^T, the next tile's S^T and dP^T are issued as
// soon as the softmax warps have copied this tile's out of TMEM, so the
// tensor core computes them while the softmax runs. V (and for d_qk = 64 also
// K) sits in TMEM as an MMA A operand; the rest is read from shared memory.
//
// FUSED (single pass, d = 64): the softmax warps also write dS^T into a
// swizzled [128 keys][64 queries] shared-memory tile, the MMA warp adds
// dQ(t) = dS K (M = 64 queries, both operands MN-major) into 64 more TMEM
// columns, and the softmax warps add each partial into the fp32 dQ buffer
// one step later (the dQ reduction across CTAs of wittx "FlashAttention-4",
// 反向传播的优化), in key-tile order when a semaphore per query tile is given.
template <int DQK, int DV, bool FUSED = false>
struct DkdvCfg {
  static constexpr int QB = 64;                     // query rows per step
  // TMEM columns: S^T | dP^T | P^T,dS^T | dV | dK | [V] | [K]
  static constexpr uint32_t tS = 0, tdP = QB, tPdS = 2 * QB, tdV = 3 * QB, tdK = 3 * QB + DV;
  static constexpr uint32_t BASE = tdK + DQK;
  static constexpr bool V_TMEM = BASE + DV / 2 <= 512;
  static constexpr uint32_t tV = BASE;
  static constexpr uint32_t tK = BASE + (V_TMEM ? DV / 2 : 0);
  static constexpr bool K_TMEM = tK + DQK / 2 <= 512;
  static constexpr int QCH = DQK / 64, VCH = DV / 64;
  static constexpr int K_BYTES = QCH * KB * 128;
  static constexpr int V_BYTES = VCH * KB * 128;
  static constexpr int QT_BYTES = QCH * QB * 128;   // one query tile of Q
  static constexpr int DOT_BYTES = VCH * QB * 128;  // one query tile of dO
  static constexpr int NST = DQK == 192 ? 3 : 4;  // query-tile stages (as many as shared memory holds)
  static constexpr int STAGE = QT_BYTES + DOT_BYTES;
  static constexpr int OFF_V = K_BYTES;
  static constexpr int OFF_ST = OFF_V + V_BYTES;
  static constexpr int OFF_VEC = OFF_ST + NST * STAGE;  // per stage: [QB] -LSE*log2e, [QB] -D
  static constexpr int OFF_DS = (OFF_VEC + NST * 2 * QB * 4 + 1023) / 1024 * 1024;  // FUSED: dS^T tile
  static constexpr int OFF_BAR = FUSED ? OFF_DS + KB * QB * 2 : OFF_VEC + NST * 2 * QB * 4;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  // FUSED: the 64 x DQK dQ partial (M = 64: row m in lane 32 (m / 16) + m % 16)
  static constexpr uint32_t tdQ = tK + (K_TMEM ? DQK / 2 : 0);
  static_assert(!FUSED || (DQK == 64 && DV == 64 && tdQ + DQK <= 512), "single pass: d = 64");
  static_assert(BASE <= 512, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct DkdvBars {
  uint64_t kv_full;
  uint64_t kv_tmem;
  uint64_t st_full[4];
  uint64_t st_empty[4];
  uint64_t s_full;
  uint64_t sp_free;   // softmax warps hold S^T(t), dP^T(t) in registers
  uint64_t pds_free;  // dV(t), dK(t) have read P^T(t), dS^T(t)
  uint64_t ds_full;
  uint64_t acc_full;
  uint64_t mma_done;
  uint32_t tmem_base;
};

// Waits until *sem >= target (acquire). Gives up like mbar_wait (10 s and
// 2^22 polls, or at once when another wait already failed), recording
// DEV_TIMEOUT_SEM at `where`.
__device__ __forceinline__ bool sem_wait(const int* sem, int target, uint32_t* status, uint32_t where) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(sem) : "memory");
    if (v >= target) return true;
    if (i > 64) __nanosleep(128);
    if ((i & 0xFFu) == 0xFFu) {
      if (status && *reinterpret_cast<volatile uint32_t*>(status) != 0) return false;
      if (i > kMinPolls && globaltimer_ns() - t0 > kWaitNs) break;
    }
  }
  record_error(status, DEV_TIMEOUT_SEM, where);
  return false;
}

// SPARSE: the key block's query tiles are those of the query blocks in its
// transposed block-sparse list (a.q_index), not m_begin .. m_end - 1.
template <int DQK, int DV, bool SPARSE = false, int MOD = 0, bool FUSED = false>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo, const BwdArgs a) {
  using C = DkdvCfg<DQK, DV, FUSED>;
  constexpr int QB = C::QB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sST = smem + C::OFF_ST;
  float* sVec = reinterpret_cast<float*>(smem + C::OFF_VEC);  // [NST][2][QB], beside the stages
  uint8_t* sDS = smem + C::OFF_DS;                             // FUSED only
  DkdvBars* bar = reinterpret_cast<DkdvBars*>(smem + C::OFF_BAR);

  // (unit, head) is the slow index so that resident CTAs share a few heads'
  // Q/dO in L2; within a head the heaviest key tiles (tile 0 sees every query
  // under the causal mask) come first.
  Unit U;
  int h, n;
  // FUSED with semaphores: key tiles in descending order, the shortest (fewest
  // query tiles under the causal mask) first, matching the adds' order below
  if (!bwd_work(a, a.tiles_kv, a.n_kblk, FUSED && a.dq_sem != nullptr, U, h, n)) return;
  const int k0 = n * KB;
  if (k0 >= U.nk) return;
  int m_begin = 0;
  if (a.causal) {
    const int i_min = k0 - (U.nk - U.nq);  // first query row that sees key k0
    m_begin = i_min > 0 ? i_min / QB : 0;
  }
  const int m_end = ceil_div(U.nq, QB);
  int T = m_end > m_begin ? m_end - m_begin : 0;
  // block-sparse: this key block's row of the transposed lists (per (batch, head) or shared)
  const int64_t kv_list = SPARSE ? (a.lists_per_head ? (static_cast<int64_t>(U.b) * a.heads + h) * a.n_kblk : 0) + n
                                 : 0;
  if constexpr (SPARSE) T = __ldg(a.q_count + kv_list) * (256 / QB);
  // first query row of step t
  auto q_row = [&](int t) -> int {
    if constexpr (SPARSE) {
      constexpr int R = 256 / QB;  // query tiles per 256-row block
      return __ldg(a.q_index + (kv_list * a.n_qb256 + t / R)) * 256 + (t % R) * QB;
    } else {
      return (m_begin + t) * QB;
    }
  };

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(&bar->kv_full, 1);
    mbar_init(&bar->kv_tmem, kSoftThreads / 32);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&bar->st_full[s], 1 + 32);  // the TMA bytes plus one arrival per loader lane
      mbar_init(&bar->st_empty[s], 1);
    }
    mbar_init(&bar->s_full, 1);
    mbar_init(&bar->sp_free, kSoftThreads / 32);
    mbar_init(&bar->pds_free, 1);
    mbar_init(&bar->ds_full, kSoftThreads / 32);
    mbar_init(&bar->acc_full, 1);
    mbar_init(&bar->mma_done, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bar->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bar->tmem_base;

  if (warp == kTmaWarp) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar->kv_full, C::K_BYTES + C::V_BYTES);
      for (int c = 0; c < C::QCH; ++c)
        tma_load_4d(sK + c * KB * 128, &tmk, &bar->kv_full, c * 64, h, U.k_start + k0, U.b);
      for (int c = 0; c < C::VCH; ++c)
        tma_load_4d(sV + c * KB * 128, &tmv, &bar->kv_full, c * 64, h, U.k_start + k0, U.b);
    }
    // Lane 0 streams the Q and dO tiles; every lane also writes two of the
    // tile's 64 (-LSE*log2e, -D) pairs next to the stage and arrives on the
    // stage's barrier, so the softmax warps find them there with no barrier
    // of their own (the slot is recycled only after dV, dK of that tile ran).
    int issued = 0;
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      const int st = t % C::NST;
      const uint32_t use = static_cast<uint32_t>(t / C::NST);
      const int tile = q_row(t);
      // fetch the vectors first, so their latency overlaps the wait for the slot
      float nl[QB / 32], nd[QB / 32];
#pragma unroll
      for (int u = 0; u < QB / 32; ++u) {
        const int r = static_cast<int>(lane) + 32 * u;
        nl[u] = -INFINITY;  // rows past the end: P = 0
        nd[u] = 0.f;
        if (tile + r < U.nq) {
          const int64_t idx = U.b * a.lse_sb + h * a.lse_sh + U.q_start + tile + r;
          const float l = a.lse[idx];
          nl[u] = (l == -INFINITY) ? -INFINITY : -l * 1.4426950408889634f;  // P = 2^(S * scale * log2e + nl)
          nd[u] = -a.dsum[idx];
        }
      }
      ok = mbar_wait(&bar->st_empty[st], (use & 1u) ^ 1u, a.status, 0x1100 + st);
      if (!ok) break;
      if (lane == 0) {
        uint8_t* dst = sST + st * C::STAGE;
        const int row = U.q_start + tile;
        mbar_arrive_expect_tx(&bar->st_full[st], C::STAGE);
        for (int c = 0; c < C::QCH; ++c) tma_load_4d(dst + c * QB * 128, &tmq, &bar->st_full[st], c * 64, h, row, U.b);
        for (int c = 0; c < C::VCH; ++c)
          tma_load_4d(dst + C::QT_BYTES + c * QB * 128, &tmdo, &bar->st_full[st], c * 64, h, row, U.b);
      }
      float* vec = sVec + st * 2 * QB;
#pragma unroll
      for (int u = 0; u < QB / 32; ++u) {
        vec[lane + 32 * u] = nl[u];
        vec[QB + lane + 32 * u] = nd[u];
      }
      mbar_arrive(&bar->st_full[st]);
      ++issued;
    }
    if (lane == 0) {
      if (!ok)
        for (int t = issued - 1; t >= 0 && t >= issued - C::NST; --t)
          mbar_wait(&bar->st_full[t % C::NST], static_cast<uint32_t>(t / C::NST) & 1u, nullptr, 0);
      mbar_wait(&bar->kv_full, 0, nullptr, 0);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(KB, QB, false, false);  // S^T, dP^T: B = Q / dO tile, K-major
      constexpr uint32_t idV = idesc_bf16_f32(KB, DV, false, true);   // dV: B = dO tile, MN-major
      constexpr uint32_t idK = idesc_bf16_f32(KB, DQK, false, true);  // dK: B = Q tile, MN-major
      bool ok = mbar_wait(&bar->kv_tmem, 0, a.status, 0x1200);
      const uint32_t kb = smem_u32(sK);
      auto stage_q = [&](int t) { return smem_u32(sST + (t % C::NST) * C::STAGE); };
      auto wait_stage = [&](int t) {
        return mbar_wait(&bar->st_full[t % C::NST], static_cast<uint32_t>(t / C::NST) & 1u, a.status, 0x1210);
      };
      // Descriptors are built once (K, V) or once per tile (Q, dO) and advanced
      // per k-step with desc_add, which keeps the single issuing thread's
      // instruction stream short between MMAs.
      const uint64_t dK = smem_desc(kb, 16, 1024, SWZ_128B);
      const uint64_t dV0 = smem_desc(smem_u32(sV), 16, 1024, SWZ_128B);
      auto issue_s = [&](int t) {  // S^T = K Q^T  (M = 128 keys, N = 64 queries, K = d_qk)
        const uint64_t dq = smem_desc(stage_q(t), 16, 1024, SWZ_128B);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint64_t bd = desc_add(dq, (kk / 4) * QB * 128 + (kk % 4) * 32);
          if constexpr (C::K_TMEM) {
            mma_ts(tbase + C::tS, tbase + C::tK + kk * 8, bd, idS, kk > 0 ? 1u : 0u);
          } else {
            mma_ss(tbase + C::tS, desc_add(dK, (kk / 4) * KB * 128 + (kk % 4) * 32), bd, idS, kk > 0 ? 1u : 0u);
          }
        }
      };
      auto issue_dp = [&](int t) {  // dP^T = V dO^T  (K = d_v)
        const uint64_t dg = smem_desc(stage_q(t) + C::QT_BYTES, 16, 1024, SWZ_128B);
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
          const uint64_t bd = desc_add(dg, (kk / 4) * QB * 128 + (kk % 4) * 32);
          if constexpr (C::V_TMEM) {
            mma_ts(tbase + C::tdP, tbase + C::tV + kk * 8, bd, idS, kk > 0 ? 1u : 0u);
          } else {
            mma_ss(tbase + C::tdP, desc_add(dV0, (kk / 4) * KB * 128 + (kk % 4) * 32), bd, idS, kk > 0 ? 1u : 0u);
          }
        }
      };
      if (ok) ok = mbar_wait(&bar->kv_full, 0, a.status, 0x1201);
      if (ok && T > 0) {
        ok = wait_stage(0);
        if (ok) {
          tc_fence_after();
          issue_s(0);
          issue_dp(0);
          mma_commit(&bar->s_full);
        }
      }
      for (int t = 0; t < T && ok; ++t) {
        if (t + 1 < T) {  // next S^T, dP^T as soon as the softmax warps hold this tile's
          ok = mbar_wait(&bar->sp_free, static_cast<uint32_t>(t) & 1u, a.status, 0x1215) && wait_stage(t + 1);
          if (!ok) break;
          tc_fence_after();
          issue_s(t + 1);
          issue_dp(t + 1);
          mma_commit(&bar->s_full);
        }
        ok = mbar_wait(&bar->ds_full, static_cast<uint32_t>(t) & 1u, a.status, 0x1220);
        if (!ok) break;
        tc_fence_after();
        const uint64_t mq = smem_desc(stage_q(t), QB * 128, 1024, SWZ_128B);           // Q tile, MN-major
        const uint64_t mg = smem_desc(stage_q(t) + C::QT_BYTES, QB * 128, 1024, SWZ_128B);  // dO tile, MN-major
        const uint32_t acc0 = t > 0 ? 1u : 0u;
        // dV += P^T dO and dK += dS^T Q, A from TMEM: warpgroup w's 32 queries are
        // in columns tPdS + [32w, 32w+32): P^T in the first 16, dS^T in the last 16
#pragma unroll
        for (int kk = 0; kk < QB / 16; ++kk) {
          const uint32_t pa = tbase + C::tPdS + 32 * (kk / 2) + (kk % 2) * 8;
          mma_ts(tbase + C::tdV, pa, desc_add(mg, kk * 2048), idV, kk > 0 ? 1u : acc0);
        }
#pragma unroll
        for (int kk = 0; kk < QB / 16; ++kk) {
          const uint32_t da = tbase + C::tPdS + 32 * (kk / 2) + 16 + (kk % 2) * 8;
          mma_ts(tbase + C::tdK, da, desc_add(mq, kk * 2048), idK, kk > 0 ? 1u : acc0);
        }
        if constexpr (FUSED) {  // dQ(t) = dS K over the tile's 128 keys, 16 keys (16 rows of both tiles) per k-step
          constexpr uint32_t idQ = idesc_bf16_f32(QB, DQK, true, true);
          const uint64_t dsa = smem_desc(smem_u32(sDS), KB * 128, 1024, SWZ_128B);
          const uint64_t kmn = smem_desc(kb, KB * 128, 1024, SWZ_128B);  // K as the MN-major B operand
#pragma unroll
          for (int kk = 0; kk < KB / 16; ++kk)
            mma_ss(tbase + C::tdQ, desc_add(dsa, kk * 2048), desc_add(kmn, kk * 2048), idQ, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar->pds_free);
        mma_commit(&bar->st_empty[t % C::NST]);
      }
      mma_commit(&bar->acc_full);
      mma_commit(&bar->mma_done);
      mbar_wait(&bar->mma_done, 0, a.status, 0x12ff);
    }
  } else {
    // ================= softmax gradient: one key row per thread ============
    const int wg = static_cast<int>(warp) / 4;           // which 32 of the 64 query columns
    const uint32_t quarter = warp & 3u;
    const int j = static_cast<int>(quarter * 32 + lane);  // key row within the tile
    const int kj = k0 + j;                                // key index within the sequence
    const uint32_t lane_base = tbase + ((quarter * 32u) << 16);
    // query rows i that see key kj: i >= i_vis (and kj < nk)
    const int i_vis = a.causal ? kj - (U.nk - U.nq) : -0x40000000;
    const bool key_ok = kj < U.nk;
    const float sl2 = a.scale_log2;
    const float alibi_slope = MOD == kModAlibi ? __ldg(a.alibi_slopes + h) * a.inv_scale : 0.f;  // raw units
    const uint32_t my_cols = C::tS + 32 * wg;     // this warpgroup's S^T columns
    const uint32_t my_pds = C::tPdS + 32 * wg;    // its P^T (16) and dS^T (16) columns
    bool ok = mbar_wait_warp(&bar->kv_full, 0, a.status, 0x1301);
    // K (warpgroup 0) and V (warpgroup 1) rows into TMEM as MMA A operands, where they fit
    if (ok) {
      if (wg == 0) {
        if constexpr (C::K_TMEM) tile_row_to_tmem(sK, C::QCH, j, lane_base + C::tK);
      } else {
        if constexpr (C::V_TMEM) tile_row_to_tmem(sV, C::VCH, j, lane_base + C::tV);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar->kv_tmem);
    const float2 sl2v = make_float2(sl2, sl2);
    // FUSED: adds this warp's part of the dQ partial of the query tile at tq0 (lanes
    // 0-15 hold rows 16 * quarter + lane, columns 32 * wg ...) into the fp32 buffer.
    // With semaphores the adds to a query tile go from the highest contributing key
    // tile down (SPT order: wittx "FlashAttention-4", 反向传播的优化): the key tiles
    // that see query tile m are 0 .. n_m - 1 (a prefix, since m_begin grows with
    // n), so each warp waits until the eight warps of each of the n_m - 1 - n tiles
    // above it have added this tile, and counts itself in afterwards.
    auto reduce_dq = [&](const uint32_t (&qv)[32], int tq0) -> bool {
      bool good = true;
      int* sem = a.dq_sem ? a.dq_sem + (static_cast<int64_t>(U.unit) * a.heads + h) * a.n_qt64 + tq0 / QB : nullptr;
      if (sem != nullptr) {
        int n_m = ceil_div(U.nk, KB);
        if (a.causal) {  // key tiles with 128 n - (nk - nq) <= the tile's last row
          const int lim = tq0 + QB - 1 + (U.nk - U.nq);
          n_m = min(n_m, lim / KB + 1);  // lim >= 0: this tile sees key tile n
        }
        if (lane == 0) good = sem_wait(sem, (n_m - 1 - n) * (kSoftThreads / 32), a.status, 0x1320);
        good = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
      }
      const int m = 16 * static_cast<int>(quarter) + static_cast<int>(lane);
      if (lane < 16 && tq0 + m < U.nq) {
        float* dst = a.dq_acc + ((static_cast<int64_t>(U.b) * a.heads + h) * a.seqlen_q + U.q_start + tq0 + m) * DQK +
                     32 * wg;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4 * c),
                       "f"(__uint_as_float(qv[4 * c])), "f"(__uint_as_float(qv[4 * c + 1])),
                       "f"(__uint_as_float(qv[4 * c + 2])), "f"(__uint_as_float(qv[4 * c + 3]))
                       : "memory");
      }
      if (sem != nullptr) {
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(sem, 1);
      }
      return good;
    };
    for (int t = 0; t < T && ok; ++t) {
      const int q0 = q_row(t);
      ok = mbar_wait_warp(&bar->s_full, static_cast<uint32_t>(t) & 1u, a.status, 0x1300);
      // this tile's (-LSE*log2e, -D) vectors, written by the loader lanes
      if (ok) ok = mbar_wait_warp(&bar->st_full[t % C::NST], static_cast<uint32_t>(t / C::NST) & 1u, a.status, 0x1302);
      if (!ok) break;
      tc_fence_after();
      const float* vL = sVec + (t % C::NST) * 2 * QB + 32 * wg;
      const float* vD = vL + QB;
      uint32_t s[32], dp[32];
      tmem_ld32(lane_base + my_cols, s);
      tmem_ld32(lane_base + C::tdP + 32 * wg, dp);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar->sp_free);
      uint32_t pw[16], dw[16];
      // ALiBi: slope * (kj - qpos) of this warpgroup's first query column
      const float abase = alibi_slope * static_cast<float>(kj - q0 - 32 * wg - (U.nk - U.nq));
      auto pair = [&](int e, float2 nl, float2 nd, bool mask) {
        const int col = 32 * wg + e;
        float s0 = __uint_as_float(s[e]), s1 = __uint_as_float(s[e + 1]);
        float2 f = make_float2(1.f, 1.f);  // derivative of the score modification
        if constexpr (MOD == kModSoftcap) {
          const float t0 = tanh_scaled(s0, a.mod_k2), t1 = tanh_scaled(s1, a.mod_k2);
          s0 = a.mod_b * t0;
          s1 = a.mod_b * t1;
          f = make_float2(fmaf(-t0, t0, 1.f), fmaf(-t1, t1, 1.f));
        } else if constexpr (MOD == kModAlibi) {
          s0 -= fabsf(fmaf(-alibi_slope, static_cast<float>(e), abase));
          s1 -= fabsf(fmaf(-alibi_slope, static_cast<float>(e + 1), abase));
        }
        const float2 x = ffma2(make_float2(s0, s1), sl2v, nl);
        float2 p = make_float2(ex2_mufu(x.x), ex2_mufu(x.y));
        if (mask) {
          if (!(key_ok && q0 + col >= i_vis)) p.x = 0.f;
          if (!(key_ok && q0 + col + 1 >= i_vis)) p.y = 0.f;
        }
        float2 ds = fmul2(p, fadd2(make_float2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), nd));
        if constexpr (MOD == kModSoftcap) ds = fmul2(ds, f);
        pw[e / 2] = pack_bf16x2(p.x, p.y);
        dw[e / 2] = pack_bf16x2(ds.x, ds.y);
      };
      auto row = [&](bool mask) {
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 nl = *reinterpret_cast<const float4*>(vL + e);
          const float4 nd = *reinterpret_cast<const float4*>(vD + e);
          pair(e, make_float2(nl.x, nl.y), make_float2(nd.x, nd.y), mask);
          pair(e + 2, make_float2(nl.z, nl.w), make_float2(nd.z, nd.w), mask);
        }
      };
      // Queries past the end already give P = 0 through -LSE*log2e = -inf, so only
      // the causal boundary and a key row past the end need the per-element test.
      if (key_ok && q0 + 32 * wg >= i_vis) row(false);
      else row(true);
      if (t > 0) {  // dV(t-1), dK(t-1) (and dQ(t-1)) must have read the previous P^T, dS^T
        ok = mbar_wait_warp(&bar->pds_free, static_cast<uint32_t>(t - 1) & 1u, a.status, 0x1305);
        if (!ok) break;
        tc_fence_after();
      }
      uint32_t qv[32];  // FUSED: dQ(t-1), complete once pds_free(t-1) has
      if constexpr (FUSED) {
        if (t > 0) {
          tmem_ld32(lane_base + C::tdQ + 32 * wg, qv);
          tmem_wait_ld();
        }
      }
      tmem_st16(lane_base + my_pds, pw);
      tmem_st16(lane_base + my_pds + 16, dw);
      if constexpr (FUSED) {  // key row j of dS^T: query columns 32 wg .. 32 wg + 31, 16-byte chunks swizzled by j
        uint8_t* rowp = sDS + j * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4*>(rowp + (((4 * wg + u) ^ (j & 7)) << 4)) =
              make_uint4(dw[4 * u], dw[4 * u + 1], dw[4 * u + 2], dw[4 * u + 3]);
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar->ds_full);
      if constexpr (FUSED) {
        if (t > 0) ok = reduce_dq(qv, q_row(t - 1)) && ok;
      }
    }
    // ---- epilogue: warpgroup 0 writes dV, warpgroup 1 writes scale * dK
    if (ok && T > 0) {
      ok = mbar_wait_warp(&bar->acc_full, 0, a.status, 0x1310);
      tc_fence_after();
    }
    if constexpr (FUSED) {  // the last step's dQ partial
      if (ok && T > 0) {
        uint32_t qv[32];
        tmem_ld32(lane_base + C::tdQ + 32 * wg, qv);
        tmem_wait_ld();
        ok = reduce_dq(qv, q_row(T - 1));
      }
    }
    const bool store = key_ok;
    if (wg == 0) {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dv) + U.b * a.dv_sb +
                           static_cast<int64_t>(U.k_start + kj) * a.dv_sn + h * a.dv_sh;
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t v[32], w[16];
        if (T > 0) {
          tmem_ld32(lane_base + C::tdV + c * 32, v);
          tmem_wait_ld();
        }
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = T > 0 ? pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])) : 0u;
        if (store) store_row_bf16(dst + c * 32, w);
      }
    } else {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dk) + U.b * a.dk_sb +
                           static_cast<int64_t>(U.k_start + kj) * a.dk_sn + h * a.dk_sh;
#pragma unroll
      for (int c = 0; c < DQK / 32; ++c) {
        uint32_t v[32], w[16];
        if (T > 0) {
          tmem_ld32(lane_base + C::tdK + c * 32, v);
          tmem_wait_ld();
        }
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = T > 0 ? pack_bf16x2(__uint_as_float(v[2 * e]) * a.scale, __uint_as_float(v[2 * e + 1]) * a.scale)
                       : 0u;
        if (store) store_row_bf16(dst + c * 32, w);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tbase, 512);
}

// ===========================================================================
// dK / dV kernel for d_qk = d_v = 128: 128 query rows per step
// ===========================================================================
// With 64-row steps the S^T and dP^T MMAs are only N = 64 wide, and the one
// thread that issues MMAs cannot keep the tensor core busy with them. Here a
// step is 128 queries, so every MMA is N = 128. TMEM then holds two 128-column
// regions besides the dV and dK accumulators (512 columns in all):
//   S^T(t) -> R(t) and dP^T(t) -> R'(t), the other region;
//   the softmax warps write P^T(t) and dS^T(t) over S^T(t) in R(t);
//   S^T(t+1) -> R'(t) once they have copied dP^T(t) out (sp_free);
//   dP^T(t+1) -> R(t), issued after dV(t) and dK(t), which read R(t): MMAs run
//   in issue order, so the overwrite comes after those reads.
// The softmax work of a step is split: P from S^T (phase A) needs only S^T and
// the LSE vector, so it runs while the tensor core computes dV, dK of the
// previous step and dP^T of this one; dS from dP^T (phase B) follows.
struct DkdvWCfg {
  static constexpr int QB = 128, D = 128;
  static constexpr uint32_t tR0 = 0, tR1 = 128, tdV = 256, tdK = 384;
  static constexpr int TILE = QB * D * 2;            // one 128 x 128 bf16 tile: 32 KB
  static constexpr int NQ = 3, NG = 2, NVEC = 2;     // Q, dO and vector ring slots
  static constexpr int OFF_K = 0, OFF_V = TILE, OFF_Q = 2 * TILE;
  static constexpr int OFF_G = OFF_Q + NQ * TILE;
  static constexpr int OFF_VEC = OFF_G + NG * TILE;  // [NVEC][2][QB] floats: -LSE*log2e, -D
  static constexpr int OFF_BAR = OFF_VEC + NVEC * 2 * QB * 4;
  static constexpr int SMEM = OFF_BAR + 256;         // the base is 1024-byte aligned (checked)
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct DkdvWBars {
  uint64_t kv_full;
  uint64_t q_full[3], q_empty[3];
  uint64_t g_full[2], g_empty[2];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full;    // S^T(t) in TMEM
  uint64_t dp_full;   // dP^T(t) in TMEM
  uint64_t sp_free;   // softmax warps hold dP^T(t) in registers
  uint64_t ds_full;   // P^T(t), dS^T(t) written
  uint64_t acc_full;
  uint64_t mma_done;
  uint32_t tmem_base;
};
static_assert(sizeof(DkdvWBars) <= 256, "dK/dV barriers must fit their reserved bytes");

// Slot of query q (0..127) in a (-LSE*log2e) or (-D) vector of the wide dK/dV
// kernel's ring. Within each 64-query half, queries 8r + 2c + j and
// 8(r + 4) + 2c + j (r < 4, c < 4, j < 2) share the 16 bytes at slot
// 16r + 4c, so the thread with fragment column pair c reads its 16 queries'
// values in four 16-byte loads, a warp's four addresses spanning 64 bytes.
__device__ __forceinline__ int vec_slot(int q) {
  const int r = (q >> 3) & 7, c = (q >> 1) & 3, j = q & 1;
  return (q & 64) + ((r & 3) * 4 + c) * 4 + (r >> 2) * 2 + j;
}

template <bool SPARSE = false, int MOD = 0>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_wide_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo, const BwdArgs a) {
  using C = DkdvWCfg;
  constexpr int QB = C::QB;
  extern __shared__ __align__(1024) uint8_t smem_w[];
  if ((smem_u32(smem_w) & 1023u) != 0u) {  // the 128-byte-swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) record_error(a.status, DEV_BAD_CONFIG, 0x1400);
    return;
  }
  uint8_t* sK = smem_w + C::OFF_K;
  uint8_t* sV = smem_w + C::OFF_V;
  uint8_t* sQ = smem_w + C::OFF_Q;
  uint8_t* sG = smem_w + C::OFF_G;
  float* sVec = reinterpret_cast<float*>(smem_w + C::OFF_VEC);
  DkdvWBars* bar = reinterpret_cast<DkdvWBars*>(smem_w + C::OFF_BAR);

  // same work order as dkdv_kernel: (unit, head) slow, key tile 0 (the heaviest under causal) first
  Unit U;
  int h, n;
  if (!bwd_work(a, a.tiles_kv, a.n_kblk, false, U, h, n)) return;
  const int k0 = n * KB;
  if (k0 >= U.nk) return;
  int m_begin = 0;
  if (a.causal) {
    const int i_min = k0 - (U.nk - U.nq);  // first query row that sees key k0
    m_begin = i_min > 0 ? i_min / QB : 0;
  }
  const int m_end = ceil_div(U.nq, QB);
  int T = m_end > m_begin ? m_end - m_begin : 0;
  // block-sparse: this key block's row of the transposed lists (per (batch, head) or shared)
  const int64_t kv_list = SPARSE ? (a.lists_per_head ? (static_cast<int64_t>(U.b) * a.heads + h) * a.n_kblk : 0) + n
                                 : 0;
  if constexpr (SPARSE) T = __ldg(a.q_count + kv_list) * (256 / QB);
  // first query row of step t
  auto q_row = [&](int t) -> int {
    if constexpr (SPARSE) {
      constexpr int R = 256 / QB;  // query tiles per 256-row block
      return __ldg(a.q_index + (kv_list * a.n_qb256 + t / R)) * 256 + (t % R) * QB;
    } else {
      return (m_begin + t) * QB;
    }
  };

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(&bar->kv_full, 1);
    for (int s = 0; s < C::NQ; ++s) {
      mbar_init(&bar->q_full[s], 1);
      mbar_init(&bar->q_empty[s], 1);
    }
    for (int s = 0; s < C::NG; ++s) {
      mbar_init(&bar->g_full[s], 1);
      mbar_init(&bar->g_empty[s], 1);
    }
    for (int s = 0; s < C::NVEC; ++s) {
      mbar_init(&bar->v_full[s], 32);                 // every loader lane
      mbar_init(&bar->v_empty[s], kSoftThreads / 32);  // every softmax warp
    }
    mbar_init(&bar->s_full, 1);
    mbar_init(&bar->dp_full, 1);
    mbar_init(&bar->sp_free, kSoftThreads / 32);
    mbar_init(&bar->ds_full, kSoftThreads / 32);
    mbar_init(&bar->acc_full, 1);
    mbar_init(&bar->mma_done, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bar->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bar->tmem_base;
  auto region = [](int t) { return (t & 1) ? C::tR1 : C::tR0; };        // R(t): S^T(t), then P^T/dS^T(t)
  auto other = [](int t) { return (t & 1) ? C::tR0 : C::tR1; };         // R'(t): dP^T(t)

  if (warp == kTmaWarp) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar->kv_full, 2 * C::TILE);
      for (int c = 0; c < 2; ++c) tma_load_4d(sK + c * KB * 128, &tmk, &bar->kv_full, c * 64, h, U.k_start + k0, U.b);
      for (int c = 0; c < 2; ++c) tma_load_4d(sV + c * KB * 128, &tmv, &bar->kv_full, c * 64, h, U.k_start + k0, U.b);
    }
    // Lane 0 streams the Q and dO tiles; every lane writes four of the tile's
    // 128 (-LSE*log2e, -D) pairs into the vector ring and arrives on its barrier.
    int nq_issued = 0, ng_issued = 0;
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      const int tile = q_row(t);
      const int row = U.q_start + tile;
      float nl[QB / 32], nd[QB / 32];  // fetched first, so their latency overlaps the waits below
#pragma unroll
      for (int u = 0; u < QB / 32; ++u) {
        const int r = static_cast<int>(lane) + 32 * u;
        nl[u] = -INFINITY;  // rows past the end: P = 0
        nd[u] = 0.f;
        if (tile + r < U.nq) {
          const int64_t idx = U.b * a.lse_sb + h * a.lse_sh + U.q_start + tile + r;
          const float l = a.lse[idx];
          nl[u] = (l == -INFINITY) ? -INFINITY : -l * 1.4426950408889634f;  // P = 2^(S * scale * log2e + nl)
          nd[u] = -a.dsum[idx];
        }
      }
      const int qs = t % C::NQ, gs = t % C::NG, vs = t % C::NVEC;
      ok = mbar_wait(&bar->q_empty[qs], (static_cast<uint32_t>(t / C::NQ) & 1u) ^ 1u, a.status, 0x1400 + qs);
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar->q_full[qs], C::TILE);
        for (int c = 0; c < 2; ++c)
          tma_load_4d(sQ + qs * C::TILE + c * QB * 128, &tmq, &bar->q_full[qs], c * 64, h, row, U.b);
      }
      ++nq_issued;
      ok = mbar_wait(&bar->g_empty[gs], (static_cast<uint32_t>(t / C::NG) & 1u) ^ 1u, a.status, 0x1408 + gs);
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar->g_full[gs], C::TILE);
        for (int c = 0; c < 2; ++c)
          tma_load_4d(sG + gs * C::TILE + c * QB * 128, &tmdo, &bar->g_full[gs], c * 64, h, row, U.b);
      }
      ++ng_issued;
      ok = mbar_wait(&bar->v_empty[vs], (static_cast<uint32_t>(t / C::NVEC) & 1u) ^ 1u, a.status, 0x1410 + vs);
      if (!ok) break;
      float* vec = sVec + vs * 2 * QB;
#pragma unroll
      for (int u = 0; u < QB / 32; ++u) {
        const int p = vec_slot(static_cast<int>(lane) + 32 * u);
        vec[p] = nl[u];
        vec[QB + p] = nd[u];
      }
      mbar_arrive(&bar->v_full[vs]);
    }
    if (lane == 0) {
      if (!ok) {  // let the copies in flight land before the CTA exits
        for (int t = nq_issued - 1; t >= 0 && t >= nq_issued - C::NQ; --t)
          mbar_wait(&bar->q_full[t % C::NQ], static_cast<uint32_t>(t / C::NQ) & 1u, nullptr, 0);
        for (int t = ng_issued - 1; t >= 0 && t >= ng_issued - C::NG; --t)
          mbar_wait(&bar->g_full[t % C::NG], static_cast<uint32_t>(t / C::NG) & 1u, nullptr, 0);
      }
      mbar_wait(&bar->kv_full, 0, nullptr, 0);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(KB, QB, false, false);  // S^T, dP^T: B = Q / dO tile, K-major
      constexpr uint32_t idA = idesc_bf16_f32(KB, 128, false, true);  // dV, dK: B = dO / Q tile, MN-major
      const uint64_t dKd = smem_desc(smem_u32(sK), 16, 1024, SWZ_128B);
      const uint64_t dVd = smem_desc(smem_u32(sV), 16, 1024, SWZ_128B);
      auto q_tile = [&](int t) { return smem_u32(sQ + (t % C::NQ) * C::TILE); };
      auto g_tile = [&](int t) { return smem_u32(sG + (t % C::NG) * C::TILE); };
      auto issue_s = [&](int t) {  // S^T(t) = K Q^T -> R(t)
        const uint64_t bq = smem_desc(q_tile(t), 16, 1024, SWZ_128B);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk / 4) * KB * 128 + (kk % 4) * 32;
          mma_ss(tbase + region(t), desc_add(dKd, off), desc_add(bq, off), idS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_dp = [&](int t) {  // dP^T(t) = V dO^T -> R'(t)
        const uint64_t bg = smem_desc(g_tile(t), 16, 1024, SWZ_128B);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk / 4) * KB * 128 + (kk % 4) * 32;
          mma_ss(tbase + other(t), desc_add(dVd, off), desc_add(bg, off), idS, kk > 0 ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(&bar->kv_full, 0, a.status, 0x1420);
      if (ok && T > 0) {
        ok = mbar_wait(&bar->q_full[0], 0, a.status, 0x1421);
        if (ok) {
          tc_fence_after();
          issue_s(0);
          mma_commit(&bar->s_full);
          ok = mbar_wait(&bar->g_full[0], 0, a.status, 0x1422);
        }
        if (ok) {
          tc_fence_after();
          issue_dp(0);
          mma_commit(&bar->dp_full);
        }
      }
      for (int t = 0; t < T && ok; ++t) {
        if (t + 1 < T) {  // S^T(t+1) into R'(t) once the softmax warps hold dP^T(t)
          ok = mbar_wait(&bar->sp_free, static_cast<uint32_t>(t) & 1u, a.status, 0x1425) &&
               mbar_wait(&bar->q_full[(t + 1) % C::NQ], static_cast<uint32_t>((t + 1) / C::NQ) & 1u, a.status, 0x1426);
          if (!ok) break;
          tc_fence_after();
          issue_s(t + 1);
          mma_commit(&bar->s_full);
        }
        ok = mbar_wait(&bar->ds_full, static_cast<uint32_t>(t) & 1u, a.status, 0x1428);
        if (!ok) break;
        tc_fence_after();
        // dV += P^T dO and dK += dS^T Q, A from R(t): the 16 queries of k-step kk
        // belong to warpgroup kk/4, whose 64 columns hold P^T (bf16 pairs) in the
        // first 32 and dS^T in the last 32
        const uint64_t mg = smem_desc(g_tile(t), QB * 128, 1024, SWZ_128B);
        const uint64_t mq = smem_desc(q_tile(t), QB * 128, 1024, SWZ_128B);
        const uint32_t acc0 = t > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < QB / 16; ++kk) {
          const uint32_t pa = tbase + region(t) + 64 * (kk / 4) + 8 * (kk % 4);
          mma_ts(tbase + C::tdV, pa, desc_add(mg, kk * 2048), idA, kk > 0 ? 1u : acc0);
        }
        mma_commit(&bar->g_empty[t % C::NG]);
#pragma unroll
        for (int kk = 0; kk < QB / 16; ++kk) {
          const uint32_t da = tbase + region(t) + 64 * (kk / 4) + 32 + 8 * (kk % 4);
          mma_ts(tbase + C::tdK, da, desc_add(mq, kk * 2048), idA, kk > 0 ? 1u : acc0);
        }
        mma_commit(&bar->q_empty[t % C::NQ]);
        if (t + 1 < T) {  // dP^T(t+1) into R(t), after the reads above in issue order
          ok = mbar_wait(&bar->g_full[(t + 1) % C::NG], static_cast<uint32_t>((t + 1) / C::NG) & 1u, a.status, 0x142a);
          if (!ok) break;
          tc_fence_after();
          issue_dp(t + 1);
          mma_commit(&bar->dp_full);
        }
      }
      mma_commit(&bar->acc_full);
      mma_commit(&bar->mma_done);
      mbar_wait(&bar->mma_done, 0, a.status, 0x14ff);
    }
  } else {
    // ================= softmax gradient ====================================
    // Warp w reads its lane quarter in the 16x256b fragment layout: per 16-lane
    // group lg, thread (g, c) = (lane / 4, lane % 4) holds key rows g and g + 8
    // at query columns 8r + 2c and 8r + 2c + 1 (r = 0..7) of its warpgroup's 64.
    // A thread so needs the LSE and D of only 16 queries per step (8 float2
    // loads each), and each adjacent pair packs into the bf16x2 column 4r + c
    // that the 16x128b store writes.
    const int wg = static_cast<int>(warp) / 4;  // which 64 of the 128 query columns
    const uint32_t quarter = warp & 3u;
    const int g = static_cast<int>(lane >> 2), c = static_cast<int>(lane & 3u);
    int vis[2][2];    // [lane group][row g or g + 8]: queries i >= vis see the key
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
    const float alibi_slope = MOD == kModAlibi ? __ldg(a.alibi_slopes + h) * a.inv_scale : 0.f;  // raw units
    auto lanes = [&](int lg) { return tbase + ((quarter * 32u + 16u * static_cast<uint32_t>(lg)) << 16); };
    bool ok = true;
    for (int t = 0; t < T && ok; ++t) {
      const int q0 = q_row(t) + 64 * wg;  // this warpgroup's first query
      const uint32_t col = region(t) + 64 * wg;
      // ---- phase A: P from S^T(t), written over S^T(t) as bf16 P^T
      ok = mbar_wait_warp(&bar->s_full, static_cast<uint32_t>(t) & 1u, a.status, 0x1430) &&
           mbar_wait_warp(&bar->v_full[t % C::NVEC], static_cast<uint32_t>(t / C::NVEC) & 1u, a.status, 0x1431);
      if (!ok) break;
      tc_fence_after();
      const float4* vL = reinterpret_cast<const float4*>(sVec + (t % C::NVEC) * 2 * QB + 64 * wg) + c;
      const float4* vD = vL + QB / 4;
      const bool full = all_keys && q0 >= vis_max;  // every (key, query) cell of this thread is visible
      float2 nlv[8];  // -LSE*log2e of this thread's 16 queries (the same for both lane groups)
#pragma unroll
      for (int r = 0; r < 4; ++r) {  // queries 8r + 2c, +1 and 8(r + 4) + 2c, +1 in one 16-byte load
        const float4 x = vL[4 * r];
        nlv[r] = make_float2(x.x, x.y);
        nlv[r + 4] = make_float2(x.z, x.w);
      }
      float p[2][32];
#pragma unroll
      for (int lg = 0; lg < 2; ++lg) {
        uint32_t sv[32], pw[16];
        tmem_ld16x256b_x8(lanes(lg) + col, sv);
        tmem_wait_ld();
        // ALiBi: slope * (kj - qpos) of key rows g, g + 8 at query column 2c
        float abase[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int kj = k0 + static_cast<int>(quarter) * 32 + 16 * lg + 8 * hh + g;
          abase[hh] = alibi_slope * static_cast<float>(kj - q0 - 2 * c - (U.nk - U.nq));
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float2 nl = nlv[r];
          float sm[4], fz[4];  // modified logits and the modification's derivative
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float sx = __uint_as_float(sv[4 * r + u]);
            fz[u] = 1.f;
            if constexpr (MOD == kModSoftcap) {
              const float tt = tanh_scaled(sx, a.mod_k2);
              sx = a.mod_b * tt;
              fz[u] = fmaf(-tt, tt, 1.f);
            } else if constexpr (MOD == kModAlibi) {
              sx -= fabsf(fmaf(-alibi_slope, static_cast<float>(8 * r + (u & 1)), abase[u >> 1]));
            }
            sm[u] = sx;
          }
          const float2 x0 = ffma2(make_float2(sm[0], sm[1]), sl2v, nl);
          const float2 x1 = ffma2(make_float2(sm[2], sm[3]), sl2v, nl);
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
          if constexpr (MOD == kModSoftcap) {  // phase B then computes dS = P f (dP - D)
#pragma unroll
            for (int u = 0; u < 4; ++u) pp[u] *= fz[u];
          }
        }
        tmem_st16x128b_x8(lanes(lg) + col, pw);
      }
      // ---- phase B: dS = P (dP - D) from dP^T(t), written next to P^T
      ok = mbar_wait_warp(&bar->dp_full, static_cast<uint32_t>(t) & 1u, a.status, 0x1432);
      if (!ok) break;
      tc_fence_after();
      uint32_t dp[2][32];
      tmem_ld16x256b_x8(lanes(0) + other(t) + 64 * wg, dp[0]);
      tmem_ld16x256b_x8(lanes(1) + other(t) + 64 * wg, dp[1]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar->sp_free);
      float2 ndv[8];  // -D of the same 16 queries
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float4 x = vD[4 * r];
        ndv[r] = make_float2(x.x, x.y);
        ndv[r + 4] = make_float2(x.z, x.w);
      }
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
        mbar_arrive(&bar->ds_full);
        mbar_arrive(&bar->v_empty[t % C::NVEC]);
      }
    }
    // ---- epilogue: warpgroup 0 writes dV, warpgroup 1 writes scale * dK (one key row per thread)
    if (ok && T > 0) {
      ok = mbar_wait_warp(&bar->acc_full, 0, a.status, 0x1440);
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
    for (int c = 0; c < C::D / 32; ++c) {
      uint32_t v[32], w[16];
      if (T > 0) {
        tmem_ld32(lane_base + acc + c * 32, v);
        tmem_wait_ld();
      }
#pragma unroll
      for (int e = 0; e < 16; ++e)
        w[e] = T > 0 ? pack_bf16x2(__uint_as_float(v[2 * e]) * mul, __uint_as_float(v[2 * e + 1]) * mul) : 0u;
      if (store) store_row_bf16(dst + c * 32, w);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tbase, 512);
}

// ===========================================================================
// dQ kernel (query-stationary)
// ===========================================================================
// S = Q K^T and dP = dO V^T go to TMEM; the softmax warps write dS (bf16
// pairs) to a TMEM region of its own that feeds dQ += dS K directly. Because
// dS does not overwrite S, the next tile's S and dP are issued as soon as the
// softmax warps have copied this tile's out of TMEM. dO sits in TMEM as the A
// operand of dP where it fits (d_qk <= 128); Q is read from shared memory.
template <int DQK, int DV>
struct DqCfg {
  static constexpr bool DO_TMEM = DQK <= 128;
  static constexpr int QCH = DQK / 64, VCH = DV / 64;
  static constexpr int Q_BYTES = QCH * MB * 128;
  static constexpr int DO_BYTES = VCH * MB * 128;
  static constexpr int K_BYTES = QCH * KB * 128;
  static constexpr int V_BYTES = VCH * KB * 128;
  // Separate K and V rings: V(t) is free once dP(t) has read it, K(t) only
  // after dQ(t), so K gets the extra slot that lets its load start two steps
  // ahead (one K/V pair per step is more than an SM fetches in one step's time).
  static constexpr int KST = DQK == 64 ? 4 : DQK == 128 ? 3 : 2;
  static constexpr int VST = DQK == 64 ? 3 : DQK == 128 ? 2 : 1;
  // d_qk = 192: S and dP hand off through barriers of their own (s_full, s_free;
  // dp_full, dp_free), so the softmax warps start on S(t) while dP(t) runs and
  // S(t+1) is issued once they hold S(t). At d_qk <= 128 both go together
  // (s_full, sp_free), measured faster there.
  static constexpr bool SPLIT_SDP = KST < 3;
  static constexpr int OFF_DO = Q_BYTES;
  static constexpr int OFF_K = OFF_DO + DO_BYTES;
  static constexpr int OFF_V = OFF_K + KST * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + VST * V_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  // TMEM columns: S | dP | dS | dQ | [dO]
  static constexpr uint32_t tS = 0, tdP = 128, tdS = 256, tdQ = 320, tdO = 320 + DQK;
  static_assert(tdO + (DO_TMEM ? DV / 2 : 0) <= 512, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct DqBars {
  uint64_t q_full;
  uint64_t qd_tmem;
  uint64_t k_full[4];
  uint64_t k_empty[4];
  uint64_t v_full[3];
  uint64_t v_empty[3];
  uint64_t s_full;    // S(t) (and, unless SPLIT_SDP, dP(t)) has landed
  uint64_t sp_free;   // softmax warps hold S(t), dP(t) in registers
  uint64_t dp_full;   // SPLIT_SDP: dP(t) has landed
  uint64_t s_free;    // SPLIT_SDP: softmax warps hold S(t) in registers
  uint64_t dp_free;   // SPLIT_SDP: softmax warps hold dP(t) in registers
  uint64_t ds_free;   // dQ(t) has read dS(t)
  uint64_t ds_full;
  uint64_t acc_full;
  uint64_t mma_done;
  uint32_t tmem_base;
};

static_assert(sizeof(DqBars) <= 256, "dQ barriers must fit their reserved bytes");
static_assert(sizeof(DkdvBars) <= 256, "dK/dV barriers must fit their reserved bytes");

__device__ __forceinline__ int key_limit(int row, int nq, int nk, int causal) {
  if (!causal) return nk;
  int lim = row + (nk - nq) + 1;
  return lim < 0 ? 0 : (lim > nk ? nk : lim);
}

// SPARSE: the query tile's key blocks are its 256-row query block's list
// (a.kv_index), not 0 .. T - 1; an index outside [0, ceil(nk / KB)) becomes a
// block past the last key (zero loads, every key masked).
template <int DQK, int DV, bool SPARSE = false, int MOD = 0>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
              const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo, const BwdArgs a) {
  using C = DqCfg<DQK, DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sdO = smem + C::OFF_DO;
  uint8_t* sKr = smem + C::OFF_K;
  uint8_t* sVr = smem + C::OFF_V;
  DqBars* bar = reinterpret_cast<DqBars*>(smem + C::OFF_BAR);

  // (unit, head) slow for L2 sharing of K/V; heaviest (last) query tiles first within a head
  Unit U;
  int h, m;
  // split keys (dense, no block lists): range `split` of this query tile's key blocks
  const bool split = !SPARSE && a.dq_split > 1;
  const int range = split ? static_cast<int>(blockIdx.x % static_cast<unsigned>(a.dq_split)) : 0;
  if (!bwd_work(a, a.tiles_q, a.n_qblk, true, U, h, m,
                split ? static_cast<int>(blockIdx.x / static_cast<unsigned>(a.dq_split)) : -1))
    return;
  const int q0 = m * MB;
  if (q0 >= U.nq) return;
  const int last = min(q0 + MB - 1, U.nq - 1);
  int T = ceil_div(key_limit(last, U.nq, U.nk, a.causal), KB);
  const int kb0 = split ? range * a.dq_kb_per_split : 0;  // first key block of the range
  if (split) T = max(0, min(T, kb0 + a.dq_kb_per_split) - kb0);
  // block-sparse: this query block's list (per (batch, head) or shared)
  const int64_t q_list = SPARSE ? (a.lists_per_head ? (static_cast<int64_t>(U.b) * a.heads + h) * a.n_qb256 : 0) +
                                      (q0 >> 8)
                                : 0;
  if constexpr (SPARSE) {
    const int c = __ldg(a.kv_count + q_list);
    T = c < 0 ? 0 : (c > a.max_kv ? a.max_kv : c);
  }
  // key block of step t
  auto key_block = [&](int t) -> int {
    if constexpr (SPARSE) {
      const int n_kb = ceil_div(U.nk, KB);
      const int kb = __ldg(a.kv_index + (q_list * a.max_kv + t));
      return (kb < 0 || kb >= n_kb) ? n_kb : kb;
    } else {
      return kb0 + t;
    }
  };

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(&bar->q_full, 1);
    mbar_init(&bar->qd_tmem, kSoftThreads / 32);
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(&bar->k_full[s], 1);
      mbar_init(&bar->k_empty[s], 1);
    }
    for (int s = 0; s < C::VST; ++s) {
      mbar_init(&bar->v_full[s], 1);
      mbar_init(&bar->v_empty[s], 1);
    }
    mbar_init(&bar->s_full, 1);
    mbar_init(&bar->sp_free, kSoftThreads / 32);
    mbar_init(&bar->dp_full, 1);
    mbar_init(&bar->s_free, kSoftThreads / 32);
    mbar_init(&bar->dp_free, kSoftThreads / 32);
    mbar_init(&bar->ds_free, 1);
    mbar_init(&bar->ds_full, kSoftThreads / 32);  // one arrival per softmax warp
    mbar_init(&bar->acc_full, 1);
    mbar_init(&bar->mma_done, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bar->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bar->tmem_base;

  if (warp == kTmaWarp) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar->q_full, C::Q_BYTES + C::DO_BYTES);
      for (int c = 0; c < C::QCH; ++c)
        tma_load_4d(sQ + c * MB * 128, &tmq, &bar->q_full, c * 64, h, U.q_start + q0, U.b);
      for (int c = 0; c < C::VCH; ++c)
        tma_load_4d(sdO + c * MB * 128, &tmdo, &bar->q_full, c * 64, h, U.q_start + q0, U.b);
      int nk_issued = 0, nv_issued = 0;
      bool ok = true;
      for (int t = 0; t < T && ok; ++t) {
        const int row = U.k_start + key_block(t) * KB;
        const int ks = t % C::KST, vs = t % C::VST;
        ok = mbar_wait(&bar->k_empty[ks], (static_cast<uint32_t>(t / C::KST) & 1u) ^ 1u, a.status, 0x2100 + ks);
        if (!ok) break;
        mbar_arrive_expect_tx(&bar->k_full[ks], C::K_BYTES);
        for (int c = 0; c < C::QCH; ++c)
          tma_load_4d(sKr + ks * C::K_BYTES + c * KB * 128, &tmk, &bar->k_full[ks], c * 64, h, row, U.b);
        ++nk_issued;
        ok = mbar_wait(&bar->v_empty[vs], (static_cast<uint32_t>(t / C::VST) & 1u) ^ 1u, a.status, 0x2108 + vs);
        if (!ok) break;
        mbar_arrive_expect_tx(&bar->v_full[vs], C::V_BYTES);
        for (int c = 0; c < C::VCH; ++c)
          tma_load_4d(sVr + vs * C::V_BYTES + c * KB * 128, &tmv, &bar->v_full[vs], c * 64, h, row, U.b);
        ++nv_issued;
      }
      if (!ok) {  // let the copies in flight land before the CTA exits
        for (int t = nk_issued - 1; t >= 0 && t >= nk_issued - C::KST; --t)
          mbar_wait(&bar->k_full[t % C::KST], static_cast<uint32_t>(t / C::KST) & 1u, nullptr, 0);
        for (int t = nv_issued - 1; t >= 0 && t >= nv_issued - C::VST; --t)
          mbar_wait(&bar->v_full[t % C::VST], static_cast<uint32_t>(t / C::VST) & 1u, nullptr, 0);
      }
      mbar_wait(&bar->q_full, 0, nullptr, 0);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(MB, KB, false, false);
      constexpr uint32_t idQ = idesc_bf16_f32(MB, DQK, false, true);  // B = K tile, MN-major
      bool ok = mbar_wait(&bar->qd_tmem, 0, a.status, 0x2200);
      const uint32_t qb = smem_u32(sQ);
      auto stage_k = [&](int t) { return smem_u32(sKr + (t % C::KST) * C::K_BYTES); };
      auto stage_v = [&](int t) { return smem_u32(sVr + (t % C::VST) * C::V_BYTES); };
      auto wait_stage = [&](int t) {  // K(t) and V(t) have landed
        return mbar_wait(&bar->k_full[t % C::KST], static_cast<uint32_t>(t / C::KST) & 1u, a.status, 0x2210) &&
               mbar_wait(&bar->v_full[t % C::VST], static_cast<uint32_t>(t / C::VST) & 1u, a.status, 0x2211);
      };
      // descriptors built once (Q, dO) or once per tile (K, V), advanced per k-step
      const uint64_t dQd = smem_desc(qb, 16, 1024, SWZ_128B);
      const uint64_t dOd = smem_desc(smem_u32(sdO), 16, 1024, SWZ_128B);
      auto issue_s = [&](int t) {  // S = Q K^T
        const uint64_t dk = smem_desc(stage_k(t), 16, 1024, SWZ_128B);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint32_t off = (kk / 4) * KB * 128 + (kk % 4) * 32;
          mma_ss(tbase + C::tS, desc_add(dQd, off), desc_add(dk, off), idS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_dp = [&](int t) {  // dP = dO V^T
        const uint64_t dv = smem_desc(stage_v(t), 16, 1024, SWZ_128B);
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
          const uint32_t off = (kk / 4) * KB * 128 + (kk % 4) * 32;
          const uint64_t bd = desc_add(dv, off);
          if constexpr (C::DO_TMEM) {
            mma_ts(tbase + C::tdP, tbase + C::tdO + kk * 8, bd, idS, kk > 0 ? 1u : 0u);
          } else {
            mma_ss(tbase + C::tdP, desc_add(dOd, off), bd, idS, kk > 0 ? 1u : 0u);
          }
        }
      };
      auto commit_s = [&](int t) {  // SPLIT_SDP
        tc_fence_after();
        issue_s(t);
        mma_commit(&bar->s_full);
      };
      auto commit_dp = [&](int t) {  // SPLIT_SDP
        tc_fence_after();
        issue_dp(t);
        mma_commit(&bar->dp_full);
        mma_commit(&bar->v_empty[t % C::VST]);  // V(t) has no other reader
      };
      if (ok) ok = mbar_wait(&bar->q_full, 0, a.status, 0x2201);
      if (ok && T > 0) {
        ok = wait_stage(0);
        if (ok) {
          if constexpr (C::SPLIT_SDP) {
            commit_s(0);
            commit_dp(0);
          } else {
            tc_fence_after();
            issue_s(0);
            issue_dp(0);
            mma_commit(&bar->s_full);
            mma_commit(&bar->v_empty[0]);
          }
        }
      }
      for (int t = 0; t < T && ok; ++t) {
        auto issue_next = [&]() {  // S, dP of tile t + 1 into the regions the softmax warps have read
          tc_fence_after();
          issue_s(t + 1);
          issue_dp(t + 1);
          mma_commit(&bar->s_full);
          mma_commit(&bar->v_empty[(t + 1) % C::VST]);
        };
        auto issue_dq = [&]() {
          tc_fence_after();
          const uint64_t mk = smem_desc(stage_k(t), KB * 128, 1024, SWZ_128B);
          const uint32_t acc0 = t > 0 ? 1u : 0u;
          // dQ += dS K: A = dS from TMEM (warpgroup w's 64 keys in columns tdS + [32w, 32w+32)),
          // B = K tile read as [d][kv], MN-major
#pragma unroll
          for (int kk = 0; kk < KB / 16; ++kk) {
            const uint32_t da = tbase + C::tdS + 32 * (kk / 4) + (kk % 4) * 8;
            mma_ts(tbase + C::tdQ, da, desc_add(mk, kk * 2048), idQ, kk > 0 ? 1u : acc0);
          }
          mma_commit(&bar->ds_free);
          mma_commit(&bar->k_empty[t % C::KST]);  // K(t) read for the last time: K(t + KST) may load
        };
        if constexpr (C::SPLIT_SDP) {
          // Two K slots (d_qk = 192): K(t + 2) is copied only once dQ(t) has read K(t), so
          // dQ(t) must not wait behind tile t + 1's S and dP when K(t + 1) is late.
          // dQ(t), S(t + 1) and dP(t + 1) touch disjoint TMEM and any order is valid:
          // issue each as soon as its inputs are ready (bounded like mbar_wait).
          const uint32_t ph = static_cast<uint32_t>(t) & 1u;
          bool s_todo = t + 1 < T, dp_todo = t + 1 < T, dq_todo = true;
          const uint64_t t0 = globaltimer_ns();
          for (uint32_t polls = 0; (s_todo || dp_todo || dq_todo) && ok; ++polls) {
            bool progressed = false;
            if (s_todo && mbar_test(&bar->s_free, ph) &&
                mbar_test(&bar->k_full[(t + 1) % C::KST], static_cast<uint32_t>((t + 1) / C::KST) & 1u)) {
              commit_s(t + 1);
              s_todo = false;
              progressed = true;
            }
            if (dp_todo && mbar_test(&bar->dp_free, ph) &&
                mbar_test(&bar->v_full[(t + 1) % C::VST], static_cast<uint32_t>((t + 1) / C::VST) & 1u)) {
              commit_dp(t + 1);
              dp_todo = false;
              progressed = true;
            }
            if (dq_todo && mbar_test(&bar->ds_full, ph)) {
              issue_dq();
              dq_todo = false;
              progressed = true;
            }
            if (!progressed && polls > (1u << 20)) __nanosleep(256);  // as mbar_wait: back off only when stuck
            if (!progressed && (polls & 0xFFFu) == 0xFFFu) {
              if (polls > (1u << 16) && *reinterpret_cast<volatile uint32_t*>(a.status) != 0) ok = false;
              if (polls > kMinPolls && globaltimer_ns() - t0 > kWaitNs) {
                record_error(a.status, DEV_TIMEOUT_MBAR, s_todo ? 0x2215 : (dp_todo ? 0x2216 : 0x2220));
                ok = false;
              }
            }
          }
          if (!ok) break;
        } else {
          if (t + 1 < T) {  // next S, dP as soon as the softmax warps hold this tile's
            ok = mbar_wait(&bar->sp_free, static_cast<uint32_t>(t) & 1u, a.status, 0x2215) && wait_stage(t + 1);
            if (!ok) break;
            issue_next();
          }
          ok = mbar_wait(&bar->ds_full, static_cast<uint32_t>(t) & 1u, a.status, 0x2220);
          if (!ok) break;
          issue_dq();
        }
      }
      mma_commit(&bar->acc_full);
      mma_commit(&bar->mma_done);
      mbar_wait(&bar->mma_done, 0, a.status, 0x22ff);
    }
  } else {
    // ================= softmax gradient: one query row per thread ==========
    const int wg = static_cast<int>(warp) / 4;
    const uint32_t quarter = warp & 3u;
    const int r = static_cast<int>(quarter * 32 + lane);  // query row within the tile
    const int i = q0 + r;
    const uint32_t lane_base = tbase + ((quarter * 32u) << 16);
    const int lim = key_limit(i, U.nq, U.nk, a.causal);
    float lse2 = INFINITY, dsum = 0.f;
    if (i < U.nq) {
      const float l = a.lse[U.b * a.lse_sb + h * a.lse_sh + U.q_start + i];
      lse2 = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
      dsum = a.dsum[U.b * a.lse_sb + h * a.lse_sh + U.q_start + i];
    }
    const float sl2 = a.scale_log2;
    const float alibi_slope = MOD == kModAlibi ? __ldg(a.alibi_slopes + h) * a.inv_scale : 0.f;  // raw units
    bool ok = mbar_wait_warp(&bar->q_full, 0, a.status, 0x2301);
    // dO rows into TMEM as the A operand of dP, where it fits
    if (ok && wg == 1) {
      if constexpr (C::DO_TMEM) tile_row_to_tmem(sdO, C::VCH, r, lane_base + C::tdO);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar->qd_tmem);
    const float2 sl2v = make_float2(sl2, sl2), nl = make_float2(-lse2, -lse2), nd = make_float2(-dsum, -dsum);
    for (int t = 0; t < T && ok; ++t) {
      ok = mbar_wait_warp(&bar->s_full, static_cast<uint32_t>(t) & 1u, a.status, 0x2300);
      if (!ok) break;
      tc_fence_after();
      const int cnt = lim - key_block(t) * KB;  // visible keys of this row in tile t
      uint32_t s[64], dp[64], dw[32];
      // ALiBi: slope * (key - qpos) of this warpgroup's first key column
      const float abase = alibi_slope * static_cast<float>(key_block(t) * KB + wg * 64 - i - (U.nk - U.nq));
      // P of columns e, e + 1 (zero where masked) and the score modification's derivative f there
      auto prob2 = [&](int e, bool mask, float2& f) -> float2 {
        const int col = wg * 64 + e;
        float s0 = __uint_as_float(s[e]), s1 = __uint_as_float(s[e + 1]);
        f = make_float2(1.f, 1.f);
        if constexpr (MOD == kModSoftcap) {
          const float t0 = tanh_scaled(s0, a.mod_k2), t1 = tanh_scaled(s1, a.mod_k2);
          s0 = a.mod_b * t0;
          s1 = a.mod_b * t1;
          f = make_float2(fmaf(-t0, t0, 1.f), fmaf(-t1, t1, 1.f));
        } else if constexpr (MOD == kModAlibi) {
          s0 -= fabsf(fmaf(alibi_slope, static_cast<float>(e), abase));
          s1 -= fabsf(fmaf(alibi_slope, static_cast<float>(e + 1), abase));
        }
        const float2 x = ffma2(make_float2(s0, s1), sl2v, nl);
        float2 p = make_float2(ex2_mufu(x.x), ex2_mufu(x.y));
        if (mask) {
          if (col >= cnt) p.x = 0.f;
          if (col + 1 >= cnt) p.y = 0.f;
        }
        return p;
      };
      const bool full = cnt >= wg * 64 + 64;  // every key of this warpgroup's half is visible
      if constexpr (C::SPLIT_SDP) {
        // this warpgroup's 64 columns of S out of TMEM, then S released
        tmem_ld32(lane_base + C::tS + wg * 64, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld32(lane_base + C::tS + wg * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar->s_free);
        // P times f, in place of S, while dP(t) runs
        auto prob = [&](bool mask) {
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            float2 f;
            float2 p = prob2(e, mask, f);
            if constexpr (MOD == kModSoftcap) p = fmul2(p, f);
            s[e] = __float_as_uint(p.x);
            s[e + 1] = __float_as_uint(p.y);
          }
        };
        if (full) prob(false);
        else prob(true);
        ok = mbar_wait_warp(&bar->dp_full, static_cast<uint32_t>(t) & 1u, a.status, 0x2302);
        if (!ok) break;
        tc_fence_after();
        tmem_ld32(lane_base + C::tdP + wg * 64, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
        tmem_ld32(lane_base + C::tdP + wg * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar->dp_free);
#pragma unroll
        for (int e = 0; e < 64; e += 2) {  // dS = P f (dP - D)
          const float2 ds = fmul2(make_float2(__uint_as_float(s[e]), __uint_as_float(s[e + 1])),
                                  fadd2(make_float2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), nd));
          dw[e / 2] = pack_bf16x2(ds.x, ds.y);
        }
      } else {
        // this warpgroup's 64 columns of S and dP out of TMEM, then both released
        tmem_ld32(lane_base + C::tS + wg * 64, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tmem_ld32(lane_base + C::tS + wg * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tmem_ld32(lane_base + C::tdP + wg * 64, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
        tmem_ld32(lane_base + C::tdP + wg * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar->sp_free);
        auto row = [&](bool mask) {  // dS = P (dP - D) f
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            float2 f;
            const float2 p = prob2(e, mask, f);
            float2 ds = fmul2(p, fadd2(make_float2(__uint_as_float(dp[e]), __uint_as_float(dp[e + 1])), nd));
            if constexpr (MOD == kModSoftcap) ds = fmul2(ds, f);
            dw[e / 2] = pack_bf16x2(ds.x, ds.y);
          }
        };
        if (full) row(false);
        else row(true);
      }
      if (t > 0) {  // dQ(t-1) must have read the previous dS
        ok = mbar_wait_warp(&bar->ds_free, static_cast<uint32_t>(t - 1) & 1u, a.status, 0x2305);
        if (!ok) break;
        tc_fence_after();
      }
      tmem_st32(lane_base + C::tdS + wg * 32, dw);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar->ds_full);
    }
    if (ok && T > 0) {
      ok = mbar_wait_warp(&bar->acc_full, 0, a.status, 0x2310);
      tc_fence_after();
    }
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.dq) + U.b * a.dq_sb +
                         static_cast<int64_t>(U.q_start + i) * a.dq_sn + h * a.dq_sh;
    constexpr int CPW = DQK / 2;  // dQ columns per warpgroup (32, 64 or 96)
    // split keys: this range's unscaled fp32 dQ row (zero when the range sees no key)
    float* part = split ? a.dq_part + ((static_cast<int64_t>(range) * a.batch + U.b) * a.heads + h) *
                                          static_cast<int64_t>(a.seqlen_q) * DQK +
                              static_cast<int64_t>(i) * DQK
                        : nullptr;
#pragma unroll
    for (int c = 0; c < CPW / 32; ++c) {
      const int col0 = wg * CPW + c * 32;
      uint32_t v[32], w[16];
      if (T > 0) {
        tmem_ld32(lane_base + C::tdQ + col0, v);
        tmem_wait_ld();
      }
      if (split) {
        if (i < U.nq) {
          float4* pv = reinterpret_cast<float4*>(part + col0);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            pv[e] = T > 0 ? make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                        __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        continue;
      }
#pragma unroll
      for (int e = 0; e < 16; ++e)
        w[e] = T > 0 ? pack_bf16x2(__uint_as_float(v[2 * e]) * a.scale, __uint_as_float(v[2 * e + 1]) * a.scale) : 0u;
      if (i < U.nq) store_row_bf16(dst + col0, w);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tbase, 512);
}

template <typename K>
cudaError_t set_smem(K kern, int bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int DQK, int DV, bool SPARSE, int MOD = 0, bool FUSED = false>
cudaError_t launch_dkdv_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                          const BwdArgs& a, cudaStream_t stream) {
  using C = DkdvCfg<DQK, DV, FUSED>;
  auto kern = dkdv_kernel<DQK, DV, SPARSE, MOD, FUSED>;
  static PerDeviceOnce once;
  cudaError_t e = once.run([&] { return set_smem(kern, C::SMEM); });
  if (e != cudaSuccess) return e;
  const int64_t grid = a.tiles_kv ? a.n_tiles_kv : static_cast<int64_t>(a.n_kblk) * a.num_units * a.heads;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  kern<<<static_cast<unsigned>(grid), kThreads, C::SMEM, stream>>>(tq, tk, tv, tdo, a);
  return cudaGetLastError();
}

template <bool SPARSE, int MOD = 0>
cudaError_t launch_dkdv_wide(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream) {
  static PerDeviceOnce once;
  cudaError_t e = once.run([] { return set_smem(dkdv_wide_kernel<SPARSE, MOD>, DkdvWCfg::SMEM); });
  if (e != cudaSuccess) return e;
  const int64_t grid = a.tiles_kv ? a.n_tiles_kv : static_cast<int64_t>(a.n_kblk) * a.num_units * a.heads;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  dkdv_wide_kernel<SPARSE, MOD><<<static_cast<unsigned>(grid), kThreads, DkdvWCfg::SMEM, stream>>>(tq, tk, tv, tdo, a);
  return cudaGetLastError();
}

template <int DQK, int DV, bool SPARSE, int MOD = 0>
cudaError_t launch_dq_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                        const BwdArgs& a, cudaStream_t stream) {
  using C = DqCfg<DQK, DV>;
  auto kern = dq_kernel<DQK, DV, SPARSE, MOD>;
  static PerDeviceOnce once;
  cudaError_t e = once.run([&] { return set_smem(kern, C::SMEM); });
  if (e != cudaSuccess) return e;
  const int split = (!SPARSE && a.dq_split > 1) ? a.dq_split : 1;
  if (split > 1 && (a.tiles_q != nullptr || a.dq_part == nullptr || a.dq_kb_per_split < 1))
    return cudaErrorInvalidValue;
  const int64_t grid = (a.tiles_q ? a.n_tiles_q : static_cast<int64_t>(a.n_qblk) * a.num_units * a.heads) * split;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  kern<<<static_cast<unsigned>(grid), kThreads, C::SMEM, stream>>>(tq, tk, tv, tdo, a);
  return cudaGetLastError();
}

}  // namespace bwd
}  // namespace gb300
