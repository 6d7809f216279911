// Forward attention kernel for GB300 (sm_103a): TMA-staged Q/K/V tiles,
// tcgen05 MMAs accumulating S = Q K^T and O += P V in Tensor Memory, and a
// warp-specialised pipeline:
//   warp 0        TMA producer (Q once, then K_j / V_j through a shared-memory ring)
//   warp 1        TMEM allocator and single-thread MMA issuer
//   warps 4..7    softmax + correction for query tile 0 (one thread per row)
//   warps 8..11   softmax + correction for query tile 1
// Each CTA owns 256 query rows (two 128-row tiles) of one (batch|sequence,
// head); while one tile's softmax runs the tensor core works on the other's
// MMAs (the asynchronous pipeline of newton wiki "FlashAttention-4", 核心技術,
// and jsqmd "GPU 算力翻倍…", section 四.2; TMEM-resident accumulators of
// section 四.4).
//
// Online softmax with conditional rescaling (wittx "FlashAttention-4",
// section 90%的rescaling都是白干的): scores are kept in log2 units; a row's
// running max m_used is replaced only when a new tile's row max exceeds it by
// more than 8.0, in which case O and l are multiplied by 2^(m_old - m_new);
// otherwise the stale max is kept (p <= 2^8). The epilogue divides by the
// exact row sum, which makes the result independent of the skipped rescales.
// exp2 runs on the hardware unit for most columns and on the FMA pipe
// (exp2_emu.cuh) for a fixed 1/EMU_PERIOD of them (same page, section
// 用软件"伪造"硬件指令).
//
// P enters the PV MMA in fp16 (11 significant bits) rather than bf16 (8):
// under a stale max a row's largest weights reach 2^8 and carry their own
// rounding, which with bf16 moves O by up to ~2e-2 on rows that concentrate on
// a few keys. The MMA takes A and B of one type, so V is read from an fp16 copy
// made by v_to_f16_kernel before the launch (exact for |v| < 65536). When that
// pass found a finite value outside fp16's range (a.v16_flag != 0), or no copy
// was made (a.v16_flag == nullptr), V and P stay bf16 for the whole call.
//
// This header holds the kernel template and its launch template; the
// translation units that instantiate it are attn_fwd.cu (no score
// modification), attn_fwd_mod.cu (the score-modification variants) and
// attn_fwd_fp8.cu (E4M3 inputs). The two-SM forward is attn_fwd_pair.cu.
#pragma once
#include <cuda_bf16.h>

#include <type_traits>

#include "exp2_emu.cuh"
#include "kernels.h"
#include "ptx_sm100.cuh"
#include "score_mod.cuh"

namespace gb300 {
namespace fwd {

constexpr int BM = 128;         // query rows per tile (= TMEM lanes)
constexpr int BN = 128;         // keys per KV tile
constexpr int QT = 2;           // query tiles per CTA
constexpr int kThreads = 384;   // 12 warps
constexpr int kChunk = BM * 128;  // bytes of one 64-column (128-byte) swizzled chunk of a 128-row tile
constexpr float kThreshold = 8.0f;  // log2 units (factor 256)


// TMEM column map (512 columns allocated): S/P for tile i at tS(i), O at tO(i).
__host__ __device__ constexpr uint32_t tS(int i) { return 128u * i; }
__host__ __device__ constexpr uint32_t tO(int i) { return 256u + 128u * i; }

// F8: Q and K are E4M3 bytes, so a 128-byte swizzled chunk holds 128 columns
// instead of 64 (V is always the fp16 copy or bf16: 64 columns per chunk).
template <int DQK, int DV, bool F8 = false>
struct Cfg {
  static constexpr int QX = F8 ? 128 : 64;  // Q/K columns per 128-byte chunk
  static constexpr int QCH = DQK / QX;      // 128-byte chunks of a Q/K row
  static constexpr int VCH = DV / 64;
  static constexpr int Q_BYTES = QCH * kChunk;
  static constexpr int K_BYTES = QCH * kChunk;
  static constexpr int V_BYTES = VCH * kChunk;
  static constexpr int SLOT = K_BYTES > V_BYTES ? K_BYTES : V_BYTES;
  // d_qk = 192: K and V in rings of their own, two 48 KB K slots and one 32 KB V
  // slot (barriers 0, 1 and 2), so that the next K is copied while the current
  // S runs; otherwise one ring of NSLOT slots taking K and V in turn.
  static constexpr bool SPLIT = DQK == 192;
  static constexpr int NSLOT = SPLIT ? 3 : (DQK <= 64 ? 8 : 4);
  static constexpr int BAR_OFF = QT * Q_BYTES + (SPLIT ? 2 * K_BYTES + V_BYTES : NSLOT * SLOT);
  static constexpr int SMEM = BAR_OFF + 256 + 1024;  // barriers + alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
  // Register split: warpgroup 0 (TMA, MMA, two idle warps) gives registers to
  // the two softmax warpgroups. 128*REG_LO + 256*REG_HI must fit in the
  // 384 * (launch registers per thread) the CTA starts with (checked on the host).
  static constexpr uint32_t REG_LO = DQK == 192 ? 72 : 56;
  static constexpr uint32_t REG_HI = DQK == 192 ? 192 : 200;
  static constexpr int REG_BUDGET = 128 * REG_LO + 256 * REG_HI;
};

struct Bars {
  uint64_t q_full[QT];
  uint64_t s_full[QT];
  uint64_t p_full[QT];
  uint64_t o_full[QT];
  uint64_t kv_full[8];
  uint64_t kv_empty[8];
  uint64_t mma_done;
  uint32_t tmem_base;
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// V (and so P) in fp16 for this call: a copy was made and every value fit.
__device__ __forceinline__ bool v_is_f16(const FwdArgs& a) { return a.v16_flag != nullptr && __ldg(a.v16_flag) == 0u; }

// Number of visible keys of query row `row` (0-based within its sequence).
__device__ __forceinline__ int key_limit(int row, int nq, int nk, int causal) {
  if (!causal) return nk;
  int lim = row + (nk - nq) + 1;
  return lim < 0 ? 0 : (lim > nk ? nk : lim);
}

// SPARSE: the CTA's key blocks are the list a.kv_index[mblk * a.max_kv + j],
// j < a.kv_count[mblk], instead of 0 .. nkv-1 (block-sparse masks, the
// FlexAttention / block-sparse variants of wittx "FlashAttention-4", section
// Python写GPU内核); the causal mask still applies inside the listed blocks.
//
// DIAG (diagnostic only, attn_diag_wait_timeout): the loader issues no copies
// and every wait gives up after a.spin_limit polls, so the MMA and softmax
// waits run out, record DEV_TIMEOUT_MBAR and the kernel returns with nothing
// in flight (no copy or MMA was ever issued).
//
// LIST (packed variable length): the CTA's (sequence, head, block) comes from
// the tile list in a.tiles instead of the block index. A variant of its own, so
// that the dense kernels keep their bounds in the constant bank rather than in
// registers.
//
// MOD: the score modification (score_mod.cuh) applied to every raw logit of a
// tile before the mask and the row max; 0 for none.
//
// F8: Q and K are FP8 E4M3 and S = Q K^T runs as tcgen05 kind::f8f6f4 (32
// columns per k-step, the same 32 bytes of each swizzled row as a bf16 k-step);
// their descale factors are folded into a.scale_log2 by the host, V is the
// exact fp16 copy and O is multiplied by a.v_descale in the epilogue.
//
// SPLITKV (dense): the key blocks are cut into a.kv_split ranges of
// a.kv_blocks_per_split; CTA (x, y) takes range y of the block that x names and
// writes its normalised fp32 O and its LSE over that range to a.o_part and
// a.lse_part ([range][batch, head, row]); combine_kv_splits_kernel merges them.
template <int DQK, int DV, int EMU_PERIOD, bool SPARSE = false, bool DIAG = false, bool LIST = false, int MOD = 0,
          bool F8 = false, bool SPLITKV = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmv16,
                    const FwdArgs a) {
  using C = Cfg<DQK, DV, F8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + QT * C::Q_BYTES;
  Bars* bar = reinterpret_cast<Bars*>(smem + C::BAR_OFF);

  // ---- work unit ------------------------------------------------------------
  // (unit, head) is the slow index so that the CTAs resident at any time share
  // a few heads' K/V in L2 (all heads' K/V together exceed it); within a head
  // the heaviest (last, under the causal mask) 256-row blocks come first.
  int mblk, h, q_start = 0, k_start = 0, nq = a.seqlen_q, nk = a.seqlen_k, b;
  int kv_part = 0;  // SPLITKV: this CTA's key range
  if constexpr (LIST) {
    // packed variable length: this CTA's entry of the tile list (longest sequences first)
    const int4* te = reinterpret_cast<const int4*>(a.tiles + blockIdx.x);
    const int4 t0 = __ldg(te), t1 = __ldg(te + 1);
    if (t1.z < 0) return;  // an empty entry past the real ones
    q_start = t0.x, nq = t0.y, k_start = t0.z, nk = t0.w, h = t1.x, mblk = t1.y, b = 0;
  } else {
    if constexpr (SPLITKV) kv_part = static_cast<int>(blockIdx.y);
    const GridSlot g = grid_slot(static_cast<int>(blockIdx.x), a.num_units * a.heads, a.n_mblk, a.n_groups);
    const int bh = g.pair;
    mblk = a.n_mblk - 1 - g.rank;
    const int unit = bh / a.heads;
    h = bh % a.heads;
    b = unit;
    if (a.cu_q != nullptr) {
      q_start = a.cu_q[unit];
      nq = a.cu_q[unit + 1] - q_start;
      k_start = a.cu_k[unit];
      nk = a.cu_k[unit + 1] - k_start;
      b = 0;
    }
  }
  const int row0 = mblk * (QT * BM);
  if (row0 >= nq) return;  // block-uniform: this unit is shorter than the grid's longest

  int nkv[QT];
  // block-sparse: this CTA's list (one set for all (batch, head), or one per (batch, head))
  const int64_t list_row = SPARSE ? (a.lists_per_head ? (static_cast<int64_t>(b) * a.heads + h) * a.n_mblk : 0) + mblk
                                  : 0;
  if constexpr (SPARSE) {
    int n = a.kv_count[list_row];
    n = n < 0 ? 0 : (n > a.max_kv ? a.max_kv : n);
#pragma unroll
    for (int i = 0; i < QT; ++i) nkv[i] = row0 + i * BM < nq ? n : 0;
  } else {
#pragma unroll
    for (int i = 0; i < QT; ++i) {
      const int r = row0 + i * BM;
      if (r >= nq) {
        nkv[i] = 0;
      } else {
        const int last = min(r + BM - 1, nq - 1);
        nkv[i] = ceil_div(key_limit(last, nq, nk, a.causal), BN);
      }
    }
  }
  // SPLITKV: key blocks [kb_lo, kb_lo + a.kv_blocks_per_split) only
  const int kb_lo = SPLITKV ? kv_part * a.kv_blocks_per_split : 0;
  if constexpr (SPLITKV) {
#pragma unroll
    for (int i = 0; i < QT; ++i) nkv[i] = max(0, min(nkv[i], kb_lo + a.kv_blocks_per_split) - kb_lo);
  }
  // Key block of step j: j itself, or the j-th listed block. A listed index
  // outside [0, ceil(nk / BN)) becomes ceil(nk / BN), a block past the last
  // key: its loads read zeros and every key in it is masked. (Addresses and
  // bounds are rebuilt from the kernel arguments to keep registers free.)
  auto key_block = [&](int j) -> int {
    if constexpr (SPARSE) {
      const int n_kblk = ceil_div(a.seqlen_k, BN);
      const int kb = __ldg(a.kv_index + (list_row * a.max_kv + j));
      return (kb < 0 || kb >= n_kblk) ? n_kblk : kb;
    } else {
      return j + kb_lo;
    }
  };
  const int nkv_max = max(nkv[0], nkv[1]);
  // Ring position of copy u (K of step u / 2 when u is even, V when odd): its
  // barrier pair, the how-manieth copy into that slot it is, and its address.
  auto ring_slot = [](int u) -> int {
    if constexpr (C::SPLIT) return (u & 1) ? 2 : (u >> 1) & 1;
    else return u % C::NSLOT;
  };
  auto ring_use = [](int u) -> uint32_t {
    if constexpr (C::SPLIT) return static_cast<uint32_t>((u & 1) ? (u >> 1) : (u >> 2));
    else return static_cast<uint32_t>(u / C::NSLOT);
  };
  auto ring_addr = [&](int u) -> uint8_t* {
    if constexpr (C::SPLIT) return sKV + ((u & 1) ? 2 * C::K_BYTES : ((u >> 1) & 1) * C::K_BYTES);
    else return sKV + (u % C::NSLOT) * C::SLOT;
  };
  const PollLimit poll_lim = DIAG ? PollLimit{a.spin_limit} : kNoPollLimit;  // of the waits below

  // Early copies by thread 0 for dense d_qk <= 128 without a score
  // modification. Otherwise (d_qk = 192: measured faster; block-sparse and
  // score modifications: fewer spills) the producer copies Q first, then the
  // K/V ring, after the block barrier.
  constexpr bool kEarlyQ = DQK <= 128 && !SPARSE && MOD == kModNone, kEarlyK = kEarlyQ;
  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    for (int i = 0; i < QT; ++i) {
      mbar_init(&bar->q_full[i], 1);
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->p_full[i], 4);  // one arrival per softmax warp
      mbar_init(&bar->o_full[i], 1);
    }
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&bar->kv_full[s], 1);
      mbar_init(&bar->kv_empty[s], 1);
    }
    mbar_init(&bar->mma_done, 1);
    fence_barrier_init();
    if (!DIAG && kEarlyQ) {
      // Q (and, dense, K of the first step right behind Q tile 0: all the first S
      // needs) copied before the TMEM allocation and the block barrier
      tma_prefetch_desc(&tmq);
      for (int i = 0; i < QT; ++i) {
        mbar_arrive_expect_tx(&bar->q_full[i], C::Q_BYTES);
        for (int c = 0; c < C::QCH; ++c)
          tma_load_4d(sQ + i * C::Q_BYTES + c * kChunk, &tmq, &bar->q_full[i], c * C::QX, h, q_start + row0 + i * BM, b);
        if (kEarlyK && i == 0 && nkv_max > 0) {
          const int kb0 = key_block(0);
          mbar_arrive_expect_tx(&bar->kv_full[0], C::K_BYTES);
          for (int c = 0; c < C::QCH; ++c)
            tma_load_4d(sKV + c * kChunk, &tmk, &bar->kv_full[0], c * C::QX, h, k_start + kb0 * BN, b);
        }
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(&bar->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bar->tmem_base;

  if (warp < 4) {
  regs_dec<C::REG_LO>();
  if (warp == 0) {
    // ======================= TMA producer ===================================
    if (lane == 0 && !DIAG) {
      if constexpr (!kEarlyQ) {
        tma_prefetch_desc(&tmq);
        for (int i = 0; i < QT; ++i) {
          mbar_arrive_expect_tx(&bar->q_full[i], C::Q_BYTES);
          for (int c = 0; c < C::QCH; ++c)
            tma_load_4d(sQ + i * C::Q_BYTES + c * kChunk, &tmq, &bar->q_full[i], c * C::QX, h, q_start + row0 + i * BM, b);
        }
      }
      tma_prefetch_desc(&tmk);
      // read while the Q copies fly: V from the fp16 copy, or the bf16 original
      const CUtensorMap* tmvv = v_is_f16(a) ? &tmv16 : &tmv;
      tma_prefetch_desc(tmvv);
      if constexpr (C::SPLIT) {
        // Split rings: K0, then K(j+1) before V(j), since a K slot frees a step
        // before the V slot does.
        int last_use[C::NSLOT];  // per slot, the latest copy issued into it (for the drain)
#pragma unroll
        for (int s2 = 0; s2 < C::NSLOT; ++s2) last_use[s2] = -1;
        const int n_copies = 2 * nkv_max;
        bool ok = true;
        for (int n = 0; n < n_copies + 1 && ok; ++n) {
          const int u = n == 0 ? 0 : ((n & 1) ? n + 1 : n - 1);
          if (u >= n_copies) continue;  // K of the step past the last
          const int slot = ring_slot(u);
          const uint32_t use = ring_use(u);
          ok = mbar_wait(&bar->kv_empty[slot], (use & 1u) ^ 1u, a.status, 0x100 + slot);
          if (!ok) break;
          const int kb = key_block(u >> 1);
          uint8_t* dst = ring_addr(u);
          if ((u & 1) == 0) {
            mbar_arrive_expect_tx(&bar->kv_full[slot], C::K_BYTES);
            for (int c = 0; c < C::QCH; ++c)
              tma_load_4d(dst + c * kChunk, &tmk, &bar->kv_full[slot], c * C::QX, h, k_start + kb * BN, b);
          } else {
            mbar_arrive_expect_tx(&bar->kv_full[slot], C::V_BYTES);
            for (int c = 0; c < C::VCH; ++c)
              tma_load_4d(dst + c * kChunk, tmvv, &bar->kv_full[slot], c * 64, h, k_start + kb * BN, b);
          }
          last_use[slot] = static_cast<int>(use);
        }
        if (!ok) {
          // Drain: wait (bounded) for the copies still in flight into this CTA's shared memory.
#pragma unroll
          for (int s2 = 0; s2 < C::NSLOT; ++s2)
            if (last_use[s2] >= 0) mbar_wait(&bar->kv_full[s2], static_cast<uint32_t>(last_use[s2]) & 1u, nullptr, 0);
        }
      } else {  // one ring: K0, V0, K1, V1, ...
        int issued = (kEarlyK && nkv_max > 0) ? 1 : 0;
        bool ok = true;
        for (int j = 0; j < nkv_max && ok; ++j) {
          const int kb = key_block(j);
          for (int which = (kEarlyK && j == 0) ? 1 : 0; which < 2 && ok; ++which) {  // K0 may be copied already
            const int u = 2 * j + which;
            const int slot = u % C::NSLOT;
            const uint32_t use = static_cast<uint32_t>(u / C::NSLOT);
            ok = mbar_wait(&bar->kv_empty[slot], (use & 1u) ^ 1u, a.status, 0x100 + slot);
            if (!ok) break;
            uint8_t* dst = sKV + slot * C::SLOT;
            if (which == 0) {
              mbar_arrive_expect_tx(&bar->kv_full[slot], C::K_BYTES);
              for (int c = 0; c < C::QCH; ++c)
                tma_load_4d(dst + c * kChunk, &tmk, &bar->kv_full[slot], c * C::QX, h, k_start + kb * BN, b);
            } else {
              mbar_arrive_expect_tx(&bar->kv_full[slot], C::V_BYTES);
              for (int c = 0; c < C::VCH; ++c)
                tma_load_4d(dst + c * kChunk, tmvv, &bar->kv_full[slot], c * 64, h, k_start + kb * BN, b);
            }
            ++issued;
          }
        }
        if (!ok) {
          // Drain: wait (bounded) for the copies still in flight into this CTA's shared memory.
          for (int u = issued - 1; u >= 0 && u >= issued - C::NSLOT; --u)
            mbar_wait(&bar->kv_full[u % C::NSLOT], static_cast<uint32_t>(u / C::NSLOT) & 1u, nullptr, 0);
        }
      }
      mbar_wait(&bar->q_full[0], 0, nullptr, 0);
      mbar_wait(&bar->q_full[1], 0, nullptr, 0);
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =====================================
    if (lane == 0) {
      constexpr uint32_t idS = F8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN, false, false);
      const uint32_t idO = v_is_f16(a) ? idesc_f16_f32(BM, DV, false, true) : idesc_bf16_f32(BM, DV, false, true);
      // Q tile 0 first (copied before K0), tile 1 only before its first S
      bool ok = mbar_wait(&bar->q_full[0], 0, a.status, 0x200, poll_lim);
      for (int j = 0; j <= nkv_max && ok; ++j) {
        const bool haveK = j < nkv_max;
        const bool haveV = j > 0;
        const int uK = 2 * j, uV = 2 * (j - 1) + 1;
        const int sK = ring_slot(uK), sV = ring_slot(haveV ? uV : 1);
        const uint32_t js = (static_cast<uint32_t>(j) & 0xFFFu) << 12;  // the step, in the site's bits 12..23
        if (haveK) ok = mbar_wait(&bar->kv_full[sK], ring_use(uK) & 1u, a.status, 0x210 | js, poll_lim);
        if (ok && haveV)
          ok = mbar_wait(&bar->kv_full[sV], ring_use(uV) & 1u, a.status, 0x211 | js, poll_lim);
        if (!ok) break;
        tc_fence_after();
        // descriptors built once per tile, advanced per k-step with one add
        const uint64_t dk = smem_desc(smem_u32(ring_addr(uK)), 16, 1024, SWZ_128B);
        const uint64_t dv = smem_desc(smem_u32(ring_addr(haveV ? uV : 1)), kChunk, 1024, SWZ_128B);
#pragma unroll
        for (int i = 0; i < QT; ++i) {
          if (haveV && j - 1 < nkv[i]) {
            // O_i (+)= P_i(j-1) V_{j-1}: P from TMEM (aliasing S_i), V MN-major in shared memory
            ok = mbar_wait(&bar->p_full[i], static_cast<uint32_t>(j - 1) & 1u, a.status, (0x220u + i) | js, poll_lim);
            if (!ok) break;
            tc_fence_after();
            const uint32_t acc0 = j - 1 > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
              mma_ts(tbase + tO(i), tbase + tS(i) + kk * 8, desc_add(dv, kk * 2048), idO, kk > 0 ? 1u : acc0);
            }
            if (j == nkv[i]) mma_commit(&bar->o_full[i]);
            // split rings: the V slot is free once the step's last PV (tile 1's,
            // or tile 0's when tile 1 has no such step) has completed
            if (C::SPLIT && (i == QT - 1 || j - 1 >= nkv[QT - 1])) mma_commit(&bar->kv_empty[sV]);
          }
          if (j < nkv[i]) {
            if (j == 0 && i > 0) {
              ok = mbar_wait(&bar->q_full[i], 0, a.status, 0x200u + i, poll_lim);
              if (!ok) break;
              tc_fence_after();
            }
            // S_i = Q_i K_j^T, both K-major, 16-wide k-steps walking the 128-byte swizzle atoms
            const uint64_t dq = smem_desc(smem_u32(sQ + i * C::Q_BYTES), 16, 1024, SWZ_128B);
#pragma unroll
            for (int kk = 0; kk < C::QCH * 4; ++kk) {  // 32-byte k-steps of the swizzled rows
              const uint32_t off = (kk / 4) * kChunk + (kk % 4) * 32;
              if constexpr (F8) mma_ss_f8(tbase + tS(i), desc_add(dq, off), desc_add(dk, off), idS, kk > 0 ? 1u : 0u);
              else mma_ss(tbase + tS(i), desc_add(dq, off), desc_add(dk, off), idS, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bar->s_full[i]);
          }
        }
        if (!ok) break;
        if (!C::SPLIT && haveV) mma_commit(&bar->kv_empty[sV]);
        if (haveK) mma_commit(&bar->kv_empty[sK]);
      }
      // Commits complete in order: once this one lands, every earlier MMA and
      // barrier arrival of this CTA has too, so teardown cannot race them.
      mma_commit(&bar->mma_done);
      mbar_wait(&bar->mma_done, 0, a.status, 0x2ff);
    }
  }
  } else {
    regs_inc<C::REG_HI>();
    // ======================= softmax + correction ===========================
    const int i = (warp - 4) / 4;          // query tile
    const uint32_t quarter = warp & 3u;    // TMEM lane quarter this warp may access
    const int row_in_tile = static_cast<int>(quarter * 32 + lane);
    const int row = row0 + i * BM + row_in_tile;
    // keys visible to this row (SPLITKV: counted from the range's first key, so that
    // step j is key block j of the range and kb_lo need not stay live in the loop)
    const int klim = key_limit(row, nq, nk, a.causal) - (SPLITKV ? kb_lo * BN : 0);
    const float alibi_slope = MOD == kModAlibi ? __ldg(a.alibi_slopes + h) * a.inv_scale : 0.f;  // raw units
    const int qpos = row + (nk - nq);  // the row's position among the keys (bottom-right aligned)
    const uint32_t lane_base = tbase + ((quarter * 32u) << 16);
    const float sl2 = a.scale_log2;
    const bool f16 = v_is_f16(a);  // P packed as fp16 (V's copy) or bf16
    float m_used = -INFINITY;  // log2 units
    float l = 0.f;  // row sum of the fp32 weights
    int n_rescale = 0, n_opp = 0;
    bool ok = true;
    for (int j = 0; j < nkv[i]; ++j) {
      const int kb = SPLITKV ? j : key_block(j);  // read before the wait, off the critical path
      // site: 0x300 + tile, the step in bits 12..23 (a timeout then says where it stopped)
      ok = mbar_wait_warp(&bar->s_full[i], static_cast<uint32_t>(j) & 1u, a.status,
                          0x300u + i + ((static_cast<uint32_t>(j) & 0xFFFu) << 12), poll_lim);
      if (!ok) break;
      tc_fence_after();
      uint32_t s[BN];
      tmem_ld32(lane_base + tS(i) + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tmem_ld32(lane_base + tS(i) + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      tmem_ld32(lane_base + tS(i) + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
      tmem_ld32(lane_base + tS(i) + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
      tmem_wait_ld();
      if constexpr (MOD == kModSoftcap) {
#pragma unroll
        for (int c = 0; c < BN; ++c) s[c] = __float_as_uint(a.mod_b * tanh_scaled(__uint_as_float(s[c]), a.mod_k2));
      } else if constexpr (MOD == kModAlibi) {
        const float base = alibi_slope * static_cast<float>(kb * BN - qpos);  // slope * (first key - qpos)
#pragma unroll
        for (int c = 0; c < BN; ++c)
          s[c] = __float_as_uint(__uint_as_float(s[c]) - fabsf(fmaf(alibi_slope, static_cast<float>(c), base)));
      }
      const int cnt = klim - kb * BN;  // visible keys of this row inside the tile
      if (cnt < BN) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= cnt) s[c] = __float_as_uint(-INFINITY);
      }
      // row max: 8 independent chains of three-input max, then a tree
      float mp[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) mp[c] = fmaxf(__uint_as_float(s[c]), __uint_as_float(s[c + 8]));
#pragma unroll
      for (int c = 16; c < BN; c += 16)
#pragma unroll
        for (int z = 0; z < 8; ++z) mp[z] = fmax3(mp[z], __uint_as_float(s[c + z]), __uint_as_float(s[c + 8 + z]));
      const float mx = fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
      const float m_tile = mx * sl2;
      const bool need = m_tile > m_used + kThreshold;
      float alpha = 1.f;
      if (need) {
        alpha = (m_used == -INFINITY) ? 0.f : ex2_mufu(m_used - m_tile);
        m_used = m_tile;
      }
      if (j > 0 && row < nq) {
        n_opp += (cnt > 0);
        n_rescale += need;
      }
      l *= alpha;
      const float mu = (m_used == -INFINITY) ? 0.f : m_used;
      // p = 2^(s * scale * log2e - m_used), packed to fp16 (or bf16) pairs in place
      uint32_t pk[BN / 2];
      float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // partial row sums (packed pairs)
      const float2 sl2v = make_float2(sl2, sl2), negmu = make_float2(-mu, -mu);
      auto exp_row = [&](auto f16_tag) {
        constexpr bool F16 = decltype(f16_tag)::value;
#pragma unroll
        for (int c = 0; c < BN / 2; ++c) {
          const float2 x = ffma2(make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), sl2v, negmu);
          float2 p;
          if constexpr (EMU_PERIOD > 0) {
            if (((2 * c) % EMU_PERIOD) == EMU_PERIOD - 2) {
              p = make_float2(ex2_mufu(x.x), ex2_emu(x.y));
            } else {
              p = make_float2(ex2_mufu(x.x), ex2_mufu(x.y));
            }
          } else {
            p = make_float2(ex2_mufu(x.x), ex2_mufu(x.y));
          }
          pk[c] = F16 ? pack_f16x2(p.x, p.y) : pack_bf16x2(p.x, p.y);
          rs[c & 1] = fadd2(rs[c & 1], p);
        }
      };
      if (f16) exp_row(std::true_type{});
      else exp_row(std::false_type{});
      l += (rs[0].x + rs[0].y) + (rs[1].x + rs[1].y);
      tmem_st32(lane_base + tS(i) + 0, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st32(lane_base + tS(i) + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      // correction: rescale this tile's O rows whose max moved (warp-uniform branch)
      if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + tO(i) + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
          tmem_st32(lane_base + tO(i) + c * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar->p_full[i]);
    }
    if (a.stats != nullptr) {
      int r = __reduce_add_sync(0xffffffffu, n_rescale), o = __reduce_add_sync(0xffffffffu, n_opp);
      if (lane == 0 && (r | o) != 0) {
        atomicAdd(&a.stats[0], static_cast<unsigned long long>(r));
        atomicAdd(&a.stats[1], static_cast<unsigned long long>(o));
      }
    }
    // ---- epilogue: O = acc / l (exact normalisation), LSE = ln2 * (m + log2 l)
    if (ok && nkv[i] > 0) {
      ok = mbar_wait_warp(&bar->o_full[i], 0, a.status, 0x310 + i, poll_lim);
      tc_fence_after();
    }
    float inv_l = (l > 0.f) ? 1.f / l : 0.f;
    if constexpr (F8) inv_l *= a.v_descale;
    const bool store = row < nq;
    if constexpr (SPLITKV) {
      // this range's O (normalised over its keys, fp32) and LSE; -inf where it has no key
      const int64_t prow = static_cast<int64_t>(blockIdx.y) * a.part_rows +
                           (static_cast<int64_t>(b) * a.heads + h) * a.seqlen_q + q_start + row;
      float4* op = reinterpret_cast<float4*>(a.o_part + prow * DV);
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t o[32];
        if (nkv[i] > 0) {
          tmem_ld32(lane_base + tO(i) + c * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = 0u;
        }
        if (store) {
#pragma unroll
          for (int t = 0; t < 8; ++t)
            op[c * 8 + t] = make_float4(__uint_as_float(o[4 * t]) * inv_l, __uint_as_float(o[4 * t + 1]) * inv_l,
                                        __uint_as_float(o[4 * t + 2]) * inv_l, __uint_as_float(o[4 * t + 3]) * inv_l);
        }
      }
      if (store) a.lse_part[prow] = (l > 0.f) ? (m_used + log2f(l)) * 0.69314718055994531f : -INFINITY;
    } else {
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.o) + static_cast<int64_t>(b) * a.o_sb +
                          static_cast<int64_t>(q_start + row) * a.o_sn + static_cast<int64_t>(h) * a.o_sh;
#pragma unroll
    for (int c = 0; c < DV / 32; ++c) {
      uint32_t o[32];
      if (nkv[i] > 0) {
        tmem_ld32(lane_base + tO(i) + c * 32, o);
        tmem_wait_ld();
      }
      uint32_t w[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float v0 = nkv[i] > 0 ? __uint_as_float(o[2 * t]) * inv_l : 0.f;
        const float v1 = nkv[i] > 0 ? __uint_as_float(o[2 * t + 1]) * inv_l : 0.f;
        w[t] = pack_bf16x2(v0, v1);
      }
      if (store) store_row64(orow + c * 32, w);
    }
    if (store) {
      const float lse = (l > 0.f) ? (m_used + log2f(l)) * 0.69314718055994531f : -INFINITY;
      a.lse[static_cast<int64_t>(b) * a.lse_sb + static_cast<int64_t>(h) * a.lse_sh + q_start + row] = lse;
    }
    }
  }

  // ---- teardown ------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

template <int DQK, int DV, int EMU, bool SPARSE = false, bool DIAG = false, bool LIST = false, int MOD = 0,
          bool F8 = false, bool SPLITKV = false>
cudaError_t launch_e(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tv16,
                     const FwdArgs& a, cudaStream_t stream) {
  using C = Cfg<DQK, DV, F8>;
  auto kern = attn_fwd_kernel<DQK, DV, EMU, SPARSE, DIAG, LIST, MOD, F8, SPLITKV>;
  static PerDeviceOnce once;
  cudaError_t e = once.run([&]() -> cudaError_t {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (r != cudaSuccess) return r;
    cudaFuncAttributes fa{};
    r = cudaFuncGetAttributes(&fa, kern);
    if (r != cudaSuccess) return r;
    // The setmaxnreg split must fit in the registers the CTA is launched with.
    return fa.numRegs * kThreads < C::REG_BUDGET ? cudaErrorInvalidConfiguration : cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  if (LIST != (a.tiles != nullptr) || MOD != a.score_mod || SPARSE != (a.kv_count != nullptr) ||
      F8 != (a.input_e4m3 != 0) || SPLITKV != (a.kv_split > 1))
    return cudaErrorInvalidValue;
  if (SPLITKV && (a.o_part == nullptr || a.lse_part == nullptr || a.kv_blocks_per_split < 1 || LIST || SPARSE))
    return cudaErrorInvalidValue;
  const int64_t grid = LIST ? a.n_tiles : static_cast<int64_t>(a.n_mblk) * a.num_units * a.heads;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffff || (SPLITKV && a.kv_split > 65535)) return cudaErrorInvalidConfiguration;
  const dim3 g3(static_cast<unsigned>(grid), SPLITKV ? static_cast<unsigned>(a.kv_split) : 1u);
  kern<<<g3, kThreads, C::SMEM, stream>>>(tq, tk, tv, tv16, a);
  return cudaGetLastError();
}

}  // namespace fwd
}  // namespace gb300
