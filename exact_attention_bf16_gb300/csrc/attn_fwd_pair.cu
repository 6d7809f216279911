// Forward over a pair of CTAs (d_qk = d_v = 128), the two-SM MMA (M = 256 pair)
// of wittx "FlashAttention-4", sections 反向传播的优化 and Blackwell的跛脚问题
// (the shared-memory co-bottleneck that the pair halves): the two CTAs of a
// cluster run every MMA together, the accumulator split along M (queries)
// between them and the B operand split along N, so each SM loads and reads
// half of every K and V tile.
//
// A pair owns 512 query rows; its query tile i (i = 0, 1) is the 256 rows
// [512 p + 256 i, +256), 128 per CTA (rank r: rows + 128 r), held in each
// CTA's TMEM exactly as the one-SM kernel holds its two tiles. Per key block j
// (128 keys):
//   S_i = Q_i K_j^T    A = own Q tile, B = K_j rows (keys) [64 r, 64 r + 64)
//   O_i += P_i V_j     A = P_i in TMEM, B = V_j columns [64 r, 64 r + 64)
// so each CTA copies 32 KB per key block instead of 64 KB. The softmax, the
// conditional rescale and the epilogue are the one-SM kernel's (fp16 P and V,
// bf16 when V does not fit fp16), each CTA on its own rows; the number of key
// blocks is the pair tile's (its later CTA's), the earlier CTA's extra block
// under the causal mask being fully masked.
//
// Roles per CTA (384 threads): warp 0 issues the CTA's TMA copies; warp 1 of
// rank 0 issues every MMA of the pair from one thread; warp 2 of rank 1 relays
// the completion of its CTA's copies to rank 0 (a remote mbarrier arrive);
// warps 4..11 run the softmax of the CTA's two tiles. MMA completions are
// committed to the same barrier in both CTAs (multicast); the softmax warps of
// both CTAs arrive on rank 0's barriers. Every wait is bounded, and both CTAs
// reach the final cluster barrier before TMEM is released.
#include <cuda_bf16.h>

#include "fwd_kernel.cuh"

namespace gb300 {
namespace fwd {

constexpr int kDP = 128;  // d_qk = d_v

struct PairCfg {
  static constexpr int Q_BYTES = 2 * kChunk;      // one 128-row tile: two 64-column chunks (32 KB)
  static constexpr int KH_BYTES = 2 * 64 * 128;   // half a K tile: 64 keys x 128 columns, two 8 KB chunks
  static constexpr int VH_BYTES = 128 * 128;      // half a V tile: 128 keys x 64 columns, one 16 KB chunk
  static constexpr int SLOT = 16384;
  static constexpr int NSLOT = 8;
  static constexpr int BAR_OFF = QT * Q_BYTES + NSLOT * SLOT;
  static constexpr int SMEM = BAR_OFF + 512 + 1024;  // barriers + alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
  static constexpr uint32_t REG_LO = 56, REG_HI = 200;
  static constexpr int REG_BUDGET = 128 * REG_LO + 256 * REG_HI;
};

struct PairBars {
  uint64_t q_full[QT], q_full_peer[QT];      // own Q tile landed; rank 1's landed (relayed)
  uint64_t s_full[QT], p_full[QT], o_full[QT];
  uint64_t kv_full[PairCfg::NSLOT], kv_full_peer[PairCfg::NSLOT], kv_empty[PairCfg::NSLOT];
  uint64_t mma_done;
  uint32_t tmem_base;
};
static_assert(sizeof(PairBars) <= 512, "pair barriers must fit their reserved bytes");

__device__ __forceinline__ bool wait_c(uint64_t* bar, uint32_t parity, uint32_t* status, uint32_t where) {
  return mbar_wait_cluster(bar, parity, status, where);
}
__device__ __forceinline__ bool wait_c_warp(uint64_t* bar, uint32_t parity, uint32_t* status, uint32_t where) {
  return __all_sync(0xffffffffu, mbar_wait_cluster(bar, parity, status, where));
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk_h,
                         const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmv16,
                         const FwdArgs a) {
  using C = PairCfg;
  extern __shared__ uint8_t smem_raw[];
  // the same offset in both CTAs (same kernel), so barrier offsets match for remote arrivals
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + QT * C::Q_BYTES;
  PairBars* bar = reinterpret_cast<PairBars*>(smem + C::BAR_OFF);

  // ---- work unit: (unit, head) slow, heaviest 512-row blocks first ---------
  const uint32_t rank = cluster_ctarank();
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int bh = pair / a.n_mblk;
  const int pblk = a.n_mblk - 1 - pair % a.n_mblk;
  const int unit = bh / a.heads, h = bh % a.heads;
  int q_start = 0, k_start = 0, nq = a.seqlen_q, nk = a.seqlen_k, b = unit;
  if (a.cu_q != nullptr) {
    q_start = a.cu_q[unit];
    nq = a.cu_q[unit + 1] - q_start;
    k_start = a.cu_k[unit];
    nk = a.cu_k[unit + 1] - k_start;
    b = 0;
  }
  const int prow0 = pblk * (2 * QT * BM);
  if (prow0 >= nq) return;  // pair-uniform: both CTAs leave, before any cluster barrier
  int nkv[QT];              // key blocks of pair tile i: the same in both CTAs
#pragma unroll
  for (int i = 0; i < QT; ++i) {
    const int r = prow0 + 2 * BM * i;
    nkv[i] = r >= nq ? 0 : ceil_div(key_limit(min(r + 2 * BM - 1, nq - 1), nq, nk, a.causal), BN);
  }
  const int nkv_max = max(nkv[0], nkv[1]);
  auto own_row0 = [&](int i) { return prow0 + 2 * BM * i + BM * static_cast<int>(rank); };

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    for (int i = 0; i < QT; ++i) {
      mbar_init(&bar->q_full[i], 1);
      mbar_init(&bar->q_full_peer[i], 1);
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->p_full[i], 8);  // four softmax warps in each CTA
      mbar_init(&bar->o_full[i], 1);
    }
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&bar->kv_full[s], 1);
      mbar_init(&bar->kv_full_peer[s], 1);
      mbar_init(&bar->kv_empty[s], 1);
    }
    mbar_init(&bar->mma_done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {  // one warp of each CTA allocates the pair's TMEM together
    tmem_alloc_pair(&bar->tmem_base, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tbase = bar->tmem_base;
  const bool f16 = v_is_f16(a);  // P and V in fp16, or both bf16

  if (warp < 4) {
    regs_dec<C::REG_LO>();
    if (warp == 0) {
      // ==================== TMA producer (each CTA) ===========================
      if (lane == 0) {
        for (int i = 0; i < QT; ++i) {
          mbar_arrive_expect_tx(&bar->q_full[i], C::Q_BYTES);
          for (int c = 0; c < 2; ++c)
            tma_load_4d(sQ + i * C::Q_BYTES + c * kChunk, &tmq, &bar->q_full[i], c * 64, h, q_start + own_row0(i), b);
        }
        const CUtensorMap* tmvv = f16 ? &tmv16 : &tmv;
        int issued = 0;
        bool ok = true;
        for (int j = 0; j < nkv_max && ok; ++j) {
          for (int which = 0; which < 2 && ok; ++which) {
            const int u = 2 * j + which;
            const int slot = u % C::NSLOT;
            ok = wait_c(&bar->kv_empty[slot], (static_cast<uint32_t>(u / C::NSLOT) & 1u) ^ 1u, a.status, 0x1900 + slot);
            if (!ok) break;
            uint8_t* dst = sKV + slot * C::SLOT;
            if (which == 0) {  // keys [128 j + 64 r, +64), all 128 columns
              mbar_arrive_expect_tx(&bar->kv_full[slot], C::KH_BYTES);
              for (int c = 0; c < 2; ++c)
                tma_load_4d(dst + c * (C::KH_BYTES / 2), &tmk_h, &bar->kv_full[slot], c * 64, h,
                            k_start + j * BN + 64 * static_cast<int>(rank), b);
            } else {  // all 128 keys, columns [64 r, +64)
              mbar_arrive_expect_tx(&bar->kv_full[slot], C::VH_BYTES);
              tma_load_4d(dst, tmvv, &bar->kv_full[slot], 64 * static_cast<int>(rank), h, k_start + j * BN, b);
            }
            ++issued;
          }
        }
        if (!ok)  // let the copies in flight land before the CTA leaves
          for (int u = issued - 1; u >= 0 && u >= issued - C::NSLOT; --u)
            mbar_wait(&bar->kv_full[u % C::NSLOT], static_cast<uint32_t>(u / C::NSLOT) & 1u, nullptr, 0);
        mbar_wait(&bar->q_full[0], 0, nullptr, 0);
        mbar_wait(&bar->q_full[1], 0, nullptr, 0);
      }
    } else if (warp == 2 && rank == 1) {
      // ==================== relay: rank 1's copies landed ======================
      if (lane == 0) {
        bool ok = true;
        for (int i = 0; i < QT && ok; ++i) {
          ok = mbar_wait(&bar->q_full[i], 0, a.status, 0x1910 + i);
          if (ok) mbar_arrive_cluster(&bar->q_full_peer[i], 0);
        }
        for (int u = 0; u < 2 * nkv_max && ok; ++u) {
          ok = mbar_wait(&bar->kv_full[u % C::NSLOT], static_cast<uint32_t>(u / C::NSLOT) & 1u, a.status, 0x1912);
          if (ok) mbar_arrive_cluster(&bar->kv_full_peer[u % C::NSLOT], 0);
        }
      }
    } else if (warp == 1 && rank == 0) {
      // ==================== the pair's MMA issuer ==============================
      if (lane == 0) {
        constexpr uint32_t idS = idesc_bf16_f32(2 * BM, BN, false, false);  // M = 256 pair, N = 128 keys
        const uint32_t idO = f16 ? idesc_f16_f32(2 * BM, kDP, false, true) : idesc_bf16_f32(2 * BM, kDP, false, true);
        auto both = [&](uint64_t* own, uint64_t* peer, uint32_t ph, uint32_t where) {
          return wait_c(own, ph, a.status, where) && wait_c(peer, ph, a.status, where + 1);
        };
        bool ok = both(&bar->q_full[0], &bar->q_full_peer[0], 0, 0x1920) &&
                  both(&bar->q_full[1], &bar->q_full_peer[1], 0, 0x1922);
        for (int j = 0; j <= nkv_max && ok; ++j) {
          const bool haveK = j < nkv_max, haveV = j > 0;
          const int uK = 2 * j, uV = 2 * (j - 1) + 1;
          const int sK = uK % C::NSLOT, sV = (uV + C::NSLOT) % C::NSLOT;
          const uint32_t js = (static_cast<uint32_t>(j) & 0xFFFu) << 12;
          if (haveK)
            ok = both(&bar->kv_full[sK], &bar->kv_full_peer[sK], static_cast<uint32_t>(uK / C::NSLOT) & 1u, 0x1930 | js);
          if (ok && haveV)
            ok = both(&bar->kv_full[sV], &bar->kv_full_peer[sV], static_cast<uint32_t>(uV / C::NSLOT) & 1u, 0x1932 | js);
          if (!ok) break;
          tc_fence_after();
          // K half: 64 rows per chunk (8 KB apart); V half: one 64-column chunk, MN-major
          const uint64_t dk = smem_desc(smem_u32(sKV + sK * C::SLOT), 16, 1024, SWZ_128B);
          const uint64_t dv = smem_desc(smem_u32(sKV + sV * C::SLOT), C::VH_BYTES, 1024, SWZ_128B);
#pragma unroll
          for (int i = 0; i < QT; ++i) {
            if (haveV && j - 1 < nkv[i]) {  // O_i (+)= P_i(j-1) V_{j-1}, once both CTAs' softmax wrote P_i
              ok = wait_c(&bar->p_full[i], static_cast<uint32_t>(j - 1) & 1u, a.status, (0x1940u + i) | js);
              if (!ok) break;
              tc_fence_after();
              const uint32_t acc0 = j - 1 > 0 ? 1u : 0u;
#pragma unroll
              for (int kk = 0; kk < BN / 16; ++kk)
                mma_ts_pair(tbase + tO(i), tbase + tS(i) + kk * 8, desc_add(dv, kk * 2048), idO, kk > 0 ? 1u : acc0);
              if (j == nkv[i]) mma_commit_pair(&bar->o_full[i]);
            }
            if (j < nkv[i]) {  // S_i = Q_i K_j^T
              const uint64_t dq = smem_desc(smem_u32(sQ + i * C::Q_BYTES), 16, 1024, SWZ_128B);
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ss_pair(tbase + tS(i), desc_add(dq, (kk / 4) * kChunk + (kk % 4) * 32),
                            desc_add(dk, (kk / 4) * (C::KH_BYTES / 2) + (kk % 4) * 32), idS, kk > 0 ? 1u : 0u);
              mma_commit_pair(&bar->s_full[i]);
            }
          }
          if (!ok) break;
          if (haveV) mma_commit_pair(&bar->kv_empty[sV]);
          if (haveK) mma_commit_pair(&bar->kv_empty[sK]);
        }
        mma_commit_pair(&bar->mma_done);
        mbar_wait(&bar->mma_done, 0, a.status, 0x19ff);
      }
    }
  } else {
    regs_inc<C::REG_HI>();
    // ==================== softmax + correction (each CTA, its own rows) ========
    const int i = (warp - 4) / 4;          // query tile
    const uint32_t quarter = warp & 3u;
    const int row = own_row0(i) + static_cast<int>(quarter * 32 + lane);
    const int klim = key_limit(row, nq, nk, a.causal);  // keys visible to this row
    const uint32_t lane_base = tbase + ((quarter * 32u) << 16);
    const float sl2 = a.scale_log2;
    float m_used = -INFINITY;  // log2 units
    float l = 0.f;
    int n_rescale = 0, n_opp = 0;
    bool ok = true;
    for (int j = 0; j < nkv[i]; ++j) {
      ok = wait_c_warp(&bar->s_full[i], static_cast<uint32_t>(j) & 1u, a.status,
                       0x1950u + i + ((static_cast<uint32_t>(j) & 0xFFFu) << 12));
      if (!ok) break;
      tc_fence_after();
      uint32_t s[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(lane_base + tS(i) + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * c]));
      tmem_wait_ld();
      const int cnt = klim - j * BN;  // visible keys of this row inside the tile
      if (cnt < BN) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= cnt) s[c] = __float_as_uint(-INFINITY);
      }
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
      uint32_t pk[BN / 2];
      float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      const float2 sl2v = make_float2(sl2, sl2), negmu = make_float2(-mu, -mu);
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) {
        const float2 x = ffma2(make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), sl2v, negmu);
        const float2 p = make_float2(ex2_mufu(x.x), ex2_mufu(x.y));
        pk[c] = f16 ? pack_f16x2(p.x, p.y) : pack_bf16x2(p.x, p.y);
        rs[c & 1] = fadd2(rs[c & 1], p);
      }
      l += (rs[0].x + rs[0].y) + (rs[1].x + rs[1].y);
      tmem_st32(lane_base + tS(i) + 0, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st32(lane_base + tS(i) + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      if (j > 0 && __any_sync(0xffffffffu, need)) {  // rescale this CTA's O rows whose max moved
#pragma unroll
        for (int c = 0; c < kDP / 32; ++c) {
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
      if (lane == 0) mbar_arrive_cluster(&bar->p_full[i], 0);
    }
    if (a.stats != nullptr) {
      const int r = __reduce_add_sync(0xffffffffu, n_rescale), o = __reduce_add_sync(0xffffffffu, n_opp);
      if (lane == 0 && (r | o) != 0) {
        atomicAdd(&a.stats[0], static_cast<unsigned long long>(r));
        atomicAdd(&a.stats[1], static_cast<unsigned long long>(o));
      }
    }
    // ---- epilogue: O = acc / l, LSE = ln2 * (m + log2 l)
    if (ok && nkv[i] > 0) {
      ok = wait_c_warp(&bar->o_full[i], 0, a.status, 0x1960 + i);
      tc_fence_after();
    }
    const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.o) + static_cast<int64_t>(b) * a.o_sb +
                          static_cast<int64_t>(q_start + row) * a.o_sn + static_cast<int64_t>(h) * a.o_sh;
    const bool store = row < nq;
#pragma unroll
    for (int c = 0; c < kDP / 32; ++c) {
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
      if (store) {
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int t = 0; t < 4; ++t) dst[t] = make_uint4(w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
      }
    }
    if (store) {
      const float lse = (l > 0.f) ? (m_used + log2f(l)) * 0.69314718055994531f : -INFINITY;
      a.lse[static_cast<int64_t>(b) * a.lse_sb + static_cast<int64_t>(h) * a.lse_sh + q_start + row] = lse;
    }
  }

  // Neither CTA may release TMEM or leave while the other's MMAs, remote
  // arrivals or reads of its memory can still be in flight.
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tbase, 512);
}

}  // namespace fwd

cudaError_t launch_fwd_pair(const CUtensorMap& tq, const CUtensorMap& tk_h, const CUtensorMap& tv,
                            const CUtensorMap& tv16, const FwdArgs& a, cudaStream_t stream) {
  using namespace fwd;
  if (a.kv_count != nullptr || a.tiles != nullptr || a.emu_period != 0 || a.score_mod != kModNone || a.input_e4m3)
    return cudaErrorInvalidValue;
  static PerDeviceOnce once;
  cudaError_t e = once.run([]() -> cudaError_t {
    cudaError_t r = cudaFuncSetAttribute(attn_fwd_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PairCfg::SMEM);
    if (r != cudaSuccess) return r;
    cudaFuncAttributes fa{};
    r = cudaFuncGetAttributes(&fa, attn_fwd_pair_kernel);
    if (r != cudaSuccess) return r;
    // The setmaxnreg split must fit in the registers the CTA is launched with.
    return fa.numRegs * kThreads < PairCfg::REG_BUDGET ? cudaErrorInvalidConfiguration : cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  const int64_t grid = 2 * static_cast<int64_t>(a.n_mblk) * a.num_units * a.heads;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  attn_fwd_pair_kernel<<<static_cast<unsigned>(grid), kThreads, PairCfg::SMEM, stream>>>(tq, tk_h, tv, tv16, a);
  return cudaGetLastError();
}

}  // namespace gb300
