// Internal interface between the C-ABI layer (attn_api.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>

namespace gb300 {

// One-time launch configuration of a kernel (its shared-memory limit and
// checks), done once per device: cudaFuncSetAttribute applies to the current
// device, so every GPU a process launches on must see it. Devices 0..63 are
// remembered; on others the configuration simply runs again.
struct PerDeviceOnce {
  std::atomic<uint64_t> done{0};
  template <typename F>
  cudaError_t run(F&& configure) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = configure();
    if (e != cudaSuccess) return e;
    if (bit != 0) done.fetch_or(bit, std::memory_order_release);
    return cudaSuccess;
  }
};

// Makes the device that owns a pointer current for the rest of a scope and
// restores the calling thread's previous device when the scope ends (when
// that device's context exists already, so no context is created on a GPU
// the caller never used). Defined in attn_api.cu.
class DeviceScope {
 public:
  DeviceScope() = default;
  DeviceScope(const DeviceScope&) = delete;
  DeviceScope& operator=(const DeviceScope&) = delete;
  ~DeviceScope();
  // cudaErrorInvalidDevicePointer if ptr is not device (or managed) memory.
  cudaError_t bind(const void* ptr);
  int device() const { return device_; }

 private:
  int prev_ = -1;
  int device_ = -1;
  bool switched_ = false;
};

// One CTA's work in a packed variable-length launch (built by
// launch_tile_list): the sequence's row ranges, the head and the block index
// (of R rows: 256 queries forward, 128 keys dK/dV, 128 queries dQ). seq < 0:
// an empty entry past the real ones; its CTA exits.
struct TileEntry {
  int q_start, nq, k_start, nk;
  int head, blk, seq, pad;
};
static_assert(sizeof(TileEntry) == 32, "two 16-byte loads per CTA");
constexpr int kMaxListBlocks = 2047;  // longest sequence, in blocks, a list is built for

// Dispatch order of the dense launches (one CTA per (unit, head) pair and
// block; the hardware starts CTAs roughly in index order as SMs free up). The
// pairs are cut into n_groups groups of consecutive pairs (sizes differing by
// at most one); a group's CTAs come before the next group's, and inside a group
// the block rank is walked outermost, so the first-ranked blocks of all of the
// group's pairs start before any later-ranked one. n_groups = n_pairs
// gives one pair's blocks after another. With causal masking, and the kernels
// ranking their blocks heaviest first, this keeps a heavy block from being
// started last and running alone; the group is kept small enough for its K and V to stay in
// L2 (group_count below). Bijective from [0, n_pairs * n_blk).
struct GridSlot {
  int pair, rank;
};
__host__ __device__ inline GridSlot grid_slot(int x, int n_pairs, int n_blk, int n_groups) {
  if (n_groups < 1 || n_groups > n_pairs) n_groups = n_pairs;  // (unit, head)-major
  const int base = n_pairs / n_groups, extra = n_pairs - base * n_groups;
  const int big = (base + 1) * n_blk * extra;  // CTAs of the groups with base + 1 pairs
  int size, start, r;
  if (x < big) {
    const int g = x / ((base + 1) * n_blk);
    size = base + 1, start = g * (base + 1), r = x - g * (base + 1) * n_blk;
  } else {
    const int g = (x - big) / (base * n_blk);
    size = base, start = extra * (base + 1) + g * base, r = x - big - g * base * n_blk;
  }
  const int rank = r / size;
  return GridSlot{start + (r - rank * size), rank};
}
// Number of groups for n_pairs pairs that each stream bytes_per_pair of K and V
// (or Q and dO) from L2: groups of at most 32 MB, about a quarter of GB300's L2.
inline int group_count(int n_pairs, int64_t bytes_per_pair) {
  constexpr int64_t kBudget = int64_t(32) << 20;
  if (n_pairs <= 1) return 1;
  int64_t g = bytes_per_pair > 0 ? kBudget / bytes_per_pair : n_pairs;
  if (g < 1) g = 1;
  if (g > n_pairs) g = n_pairs;
  return static_cast<int>((n_pairs + g - 1) / g);
}

// Builds the list for num_seqs sequences (cu_q / cu_k offsets on the device):
// sequences with the most blocks first (by key blocks when by_keys), then
// head by head, blocks of a head in descending or ascending order. Writes
// `bound` entries (the real ones, then empty ones); seq_start is scratch of
// num_seqs int64. max_nblk bounds every sequence's block count (<= kMaxListBlocks).
cudaError_t launch_tile_list(const int* cu_q, const int* cu_k, int num_seqs, int heads, int rows_per_block,
                             bool by_keys, bool descending, int max_nblk, TileEntry* out, int64_t* seq_start,
                             int64_t bound, cudaStream_t stream);

// Forward kernel arguments (passed by value; tensor maps go separately as
// __grid_constant__ parameters).
struct FwdArgs {
  void* o;                 // bf16 output
  float* lse;              // fp32 output
  int64_t o_sb, o_sn, o_sh;  // element strides of O (batch, row, head)
  int64_t lse_sb, lse_sh;    // element strides of LSE (batch, head); row stride 1
  int batch, heads, seqlen_q, seqlen_k;
  const int* cu_q;           // varlen offsets (device) or nullptr for dense
  const int* cu_k;
  int num_units;             // batch (dense) or number of sequences (varlen)
  int n_mblk;                // 256-row query blocks per unit = ceil(max_seqlen_q / 256)
  float scale_log2;          // softmax_scale * log2(e)
  int causal;
  uint32_t* status;          // device status word
  unsigned long long* stats; // optional rescale counters
  int emu_period;            // exp2: every emu_period-th column on the FMA pipe (0 = none)
  // Block-sparse forward only (nullptr otherwise): for 256-row query block b,
  // kv_count[b] key blocks of 128 keys, listed at kv_index[b * max_kv + j].
  const int* kv_count;
  const int* kv_index;
  int max_kv;
  uint32_t spin_limit;       // diagnostic launches only: poll limit of every wait
  // Device word written by v_to_f16 before the launch: 0 = V is read from the
  // fp16 copy (map tv16) and P is packed in fp16; nonzero, or a null pointer,
  // = V and P in bf16.
  const uint32_t* v16_flag;
  // Packed variable-length only (nullptr otherwise): one entry per CTA, and
  // the number of entries (the grid).
  const TileEntry* tiles;
  int64_t n_tiles;
  // Score modification (score_mod.cuh): kind, softcap's 2 log2(e) scale / c and
  // c / scale, 1 / scale for ALiBi's per-head slopes (device float[heads]).
  int score_mod;
  float mod_k2, mod_b, inv_scale;
  const float* alibi_slopes;
  // Block-sparse: 0 = one list set shared by every (batch, head); 1 = one per
  // (batch, head), set (b * heads + h) starting at count index (b * heads + h) * n_mblk.
  int lists_per_head;
  // E4M3 inputs (maps tq, tk over bytes; V read from its fp16 copy): O is
  // multiplied by v_descale (Q's and K's descales are in scale_log2).
  int input_e4m3;
  float v_descale;
  // Dense launches (no tile list): dispatch groups of grid_slot; heads * num_units
  // gives the (unit, head)-major order.
  int n_groups;
  // Split keys (dense, kv_split > 1): kv_split ranges of kv_blocks_per_split key
  // blocks; range r writes O over its keys (fp32, normalised) to o_part and its LSE
  // to lse_part, row (b * heads + h) * seqlen_q + i of range r at r * part_rows + row.
  int kv_split, kv_blocks_per_split;
  float* o_part;
  float* lse_part;
  int64_t part_rows;
};

cudaError_t launch_fwd(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tv16, const FwdArgs& a, cudaStream_t stream);
// The forward over CTA pairs (d_qk = d_v = 128, bf16, dense or varlen without a
// tile list): a.n_mblk counts 512-row blocks; tk_h has 64-row boxes.
cudaError_t launch_fwd_pair(const CUtensorMap& tq, const CUtensorMap& tk_h, const CUtensorMap& tv,
                            const CUtensorMap& tv16, const FwdArgs& a, cudaStream_t stream);
// The forward with E4M3 Q, K, V (d_qk = d_v = 128, dense or tile list).
cudaError_t launch_fwd_e4m3(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv16, const FwdArgs& a,
                            cudaStream_t stream);
// fp16 copy of E4M3 V (exact), laid out as launch_v_to_f16's.
cudaError_t launch_v_e4m3_to_f16(const void* v, int64_t sb, int64_t sn, int64_t sh, int nb, int nrows, int heads,
                                 int dv, void* out, cudaStream_t stream);
// The forward with a score modification (a.score_mod != 0, emu_period 0):
// dense, tile list (a.tiles) or block-sparse (a.kv_count), by the arguments.
cudaError_t launch_fwd_mod(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tv16, const FwdArgs& a, cudaStream_t stream);

// fp16 copy of V (contiguous [nb, nrows, heads, dv]) for the forward's PV
// product; ORs 1 into *flag (zeroed by the caller) if a finite value is out of
// fp16's range.
cudaError_t launch_v_to_f16(const void* v, int64_t sb, int64_t sn, int64_t sh, int nb, int nrows, int heads, int dv,
                            void* out, uint32_t* flag, cudaStream_t stream);

// Block-sparse forward (dense layout, cu_q == nullptr, emu_period == 0): the
// same kernel walking a.kv_index's key blocks instead of 0 .. nkv-1.
cudaError_t launch_fwd_sparse(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tv16, const FwdArgs& a, cudaStream_t stream);

// Diagnostic: the d = 64 dense forward with no copies issued and every wait
// limited to a.spin_limit polls (attn_diag_wait_timeout).
cudaError_t launch_fwd_diag_timeout(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                    const FwdArgs& a, cudaStream_t stream);

// Fills O = 0 and LSE = -inf for rows that see no key at all (Nk == 0).
cudaError_t launch_fwd_empty(const FwdArgs& a, int d_v, cudaStream_t stream);

// Backward kernel arguments. Dense tensors are [B, N, H, d]; varlen packed
// [total, H, d] with cu_q / cu_k offsets (batch = 1 then).
struct BwdArgs {
  const void* o;             // forward output (bf16), read by the preprocess step
  const void* dout;          // incoming gradient dO (bf16)
  const float* lse;          // forward LSE (natural log), same layout as FwdArgs
  float* dsum;               // workspace: D_i = dO_i . O_i (fp32), LSE layout
  void* dq;                  // outputs (bf16)
  void* dk;
  void* dv;
  int64_t o_sb, o_sn, o_sh;
  int64_t do_sb, do_sn, do_sh;
  int64_t dq_sb, dq_sn, dq_sh;
  int64_t dk_sb, dk_sn, dk_sh;
  int64_t dv_sb, dv_sn, dv_sh;
  int64_t lse_sb, lse_sh;
  int batch, heads, seqlen_q, seqlen_k;  // varlen: seqlen_* = total rows
  const int* cu_q;
  const int* cu_k;
  int num_units;
  int n_qblk;        // q tiles per unit for the dQ kernel: ceil(max_seqlen_q / 128)
  int n_kblk;        // kv tiles per unit for the dK/dV kernel: ceil(max_seqlen_k / 128)
  float scale;       // softmax_scale
  float scale_log2;  // softmax_scale * log2(e)
  int causal;
  uint32_t* status;
  // Block-sparse backward only (nullptr otherwise). Forward lists, for the dQ
  // kernel: 256-row query block b sees key blocks kv_index[b * max_kv + j],
  // j < kv_count[b]. Transposed lists, for the dK/dV kernel: key block n is
  // seen by query blocks q_index[n * n_qb256 + j], j < q_count[n], ascending.
  const int* kv_count;
  const int* kv_index;
  int max_kv;
  const int* q_count;
  const int* q_index;
  int n_qb256;
  // Packed variable-length only (nullptr otherwise): the dK/dV kernels' list
  // (128-key blocks) and the dQ kernel's (128-query blocks), with their sizes.
  const TileEntry* tiles_kv;
  int64_t n_tiles_kv;
  const TileEntry* tiles_q;
  int64_t n_tiles_q;
  // Score modification, as in FwdArgs.
  int score_mod;
  float mod_k2, mod_b, inv_scale;
  const float* alibi_slopes;
  // Block-sparse: 1 = lists per (batch, head): forward set (b * heads + h) at
  // count index (b * heads + h) * n_qb256, transposed set at (b * heads + h) * n_kb.
  int lists_per_head;
  // Single-pass backward only (nullptr otherwise): fp32 dQ, [units][heads][seqlen_q][d]
  // (zeroed), to which the dK/dV kernel adds its dQ partials; with dq_sem set,
  // one semaphore per (unit, head, 64-row query tile), n_qt64 tiles per (unit,
  // head), orders the adds by key tile.
  float* dq_acc;
  int* dq_sem;
  int n_qt64;
  // Dense launches (no tile list): dispatch groups of grid_slot, for the dK/dV
  // and the dQ kernels; heads * num_units gives the (unit, head)-major order.
  int n_groups;
  // Split keys for the dQ kernel (dense, no block lists; dq_split <= 1 means
  // none): each 128-query tile's key blocks are cut into dq_split ranges of
  // dq_kb_per_split blocks, one CTA each (range fastest in the grid), which
  // stores its unscaled fp32 dQ over that range to
  // dq_part[(range * batch * heads + b * heads + h) * seqlen_q + row][d_qk];
  // launch_bwd_dq_merge adds the ranges in order and writes dQ.
  int dq_split;
  int dq_kb_per_split;
  float* dq_part;
};

// Single-pass backward (d_qk = d_v = 64): dK, dV and the fp32 dQ partials of
// the dK/dV kernel (a.dq_acc, ordered by a.dq_sem when set), then
// dQ = bf16(dq_acc * scale).
cudaError_t launch_bwd_single_pass(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                   const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_dq_convert(const BwdArgs& a, int d, cudaStream_t stream);
// D = rowsum(dO * O) into args.dsum.
cudaError_t launch_bwd_preprocess(int d_v, const BwdArgs& a, cudaStream_t stream);
// dK, dV (KV-stationary) and dQ (Q-stationary). Maps: q, k, v, dO. With
// a.kv_count set they walk the block-sparse lists (dense layout only).
cudaError_t launch_bwd_dkdv(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream);
// The dK/dV and dQ kernels with a score modification (a.score_mod != 0),
// dense, tile list or block-sparse by the arguments.
cudaError_t launch_bwd_dkdv_mod(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_dq_mod(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream);
// dK, dV for d_qk = d_v = 128 over CTA pairs (dense or varlen, no block
// lists): maps q and dO with 64-row boxes (_r) and 128-row boxes (_c), k, v.
cudaError_t launch_bwd_dkdv_pair(const CUtensorMap& tq_r, const CUtensorMap& tq_c, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo_r, const CUtensorMap& tdo_c,
                                 const BwdArgs& a, cudaStream_t stream);
// Builds a.q_count / a.q_index (transposed block lists) from a.kv_count / a.kv_index
// for n_kb key blocks, deterministically (ascending query blocks).
cudaError_t launch_bwd_transpose_lists(const BwdArgs& a, int n_kb, cudaStream_t stream);
cudaError_t launch_bwd_dq(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t stream);
// dQ (bf16, strided) = scale * (sum over r < a.dq_split, in order, of a.dq_part's range r).
cudaError_t launch_bwd_dq_merge(const BwdArgs& a, int d_qk, cudaStream_t stream);
// Zero-fills dQ, dK, dV rows of a problem with no keys or no queries.
cudaError_t launch_bwd_zero(const BwdArgs& a, int d_qk, int d_v, bool zero_dq, bool zero_dkdv, cudaStream_t stream);

cudaError_t launch_exp2_eval(const float* x, float* y_poly, float* y_hw, int64_t n, cudaStream_t stream);

}  // namespace gb300
