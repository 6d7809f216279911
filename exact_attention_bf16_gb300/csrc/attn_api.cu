// C-ABI entry points of libattn_gb300.so (declared in include/attn.h):
// argument validation, TMA tensor-map encoding, workspace accounting and
// kernel launches. All compute runs in the CUDA kernels (fwd_kernel.cuh and
// bwd_kernels.cuh with the translation units that instantiate them, the pair
// kernels, schedule.cu); this file holds host logic only.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "../../include/attn.h"
#include "kernels.h"

namespace gb300 {

// Process-wide device status word (one copy per device that loads the library).
__device__ uint32_t g_attn_status;

namespace {

thread_local char t_last_cuda_error[256] = "";

attn_status_t cuda_fail(cudaError_t e, const char* what) {
  std::snprintf(t_last_cuda_error, sizeof(t_last_cuda_error), "%s: %s", what, cudaGetErrorString(e));
  return ATTN_ERR_CUDA;
}

constexpr int kMaxDevices = 64;
uint32_t* g_status_ptr[kMaxDevices] = {};
std::mutex g_mu;

// Device address of g_attn_status for the current device (looked up once per device).
cudaError_t status_ptr(uint32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_status);
    if (e != cudaSuccess) return e;
    g_status_ptr[dev] = static_cast<uint32_t*>(p);
  }
  *out = g_status_ptr[dev];
  return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// TMA map over a bf16 tensor viewed as [n_b, n_rows, n_heads, d] with element
// strides (sb, sn, sh) and unit stride on d. Box: 64 columns x 1 head x
// `box_rows` rows x 1 batch, 128-byte swizzle (the UMMA K-major / MN-major
// SW128 layout). Out-of-range rows read as zero.
// elem_bytes 2: bf16 / fp16 elements, 64-column boxes; 1: E4M3 bytes, 128-column
// boxes. Either way a box row is one 128-byte swizzled chunk.
attn_status_t make_map(CUtensorMap* m, const void* base, int d, int n_heads, int64_t n_rows, int n_b, int64_t sb,
                       int64_t sn, int64_t sh, int box_rows, int elem_bytes = 2) {
  auto enc = encode_fn();
  if (!enc) return cuda_fail(cudaErrorNotSupported, "cuTensorMapEncodeTiled unavailable");
  // Size-1 dimensions may carry any stride; give them a valid one.
  if (n_heads == 1) sh = d;
  if (n_b == 1) sb = sn * (n_rows > 0 ? n_rows : 1);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n_heads),
                        static_cast<cuuint64_t>(n_rows > 0 ? n_rows : 1), static_cast<cuuint64_t>(n_b)};
  const cuuint64_t eb = static_cast<cuuint64_t>(elem_bytes);
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(sh) * eb, static_cast<cuuint64_t>(sn) * eb,
                           static_cast<cuuint64_t>(sb) * eb};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / elem_bytes), 1, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = enc(m, ty, 4, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(t_last_cuda_error, sizeof(t_last_cuda_error), "cuTensorMapEncodeTiled failed (%d)",
                  static_cast<int>(r));
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

}  // namespace

// DeviceScope (kernels.h): makes the data's device current for the launches of
// one entry point and restores the caller's current device afterwards.
// Entry points may be called from threads, such as an autograd worker, on
// which this library has not yet touched the device, and from multi-GPU
// callers whose current device must survive the call.
cudaError_t DeviceScope::bind(const void* ptr) {
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, ptr);
  if (e != cudaSuccess) return e;
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return cudaErrorInvalidDevicePointer;
  e = cudaGetDevice(&prev_);
  if (e != cudaSuccess) return e;
  device_ = attr.device;
  // Always select it: cudaSetDevice also makes the device's primary context
  // current on this thread, which a thread that never used the runtime (an
  // autograd worker) lacks even when its default device is the right one.
  e = cudaSetDevice(device_);
  if (e == cudaSuccess && prev_ != device_) switched_ = true;
  return e;
}

DeviceScope::~DeviceScope() {
  if (!switched_) return;
  // Put the caller's device back only if its primary context already exists:
  // selecting a device whose context was never created would create one (and
  // take its memory) on a GPU the caller never used.
  using GetFn = CUresult (*)(CUdevice*, int);
  using StateFn = CUresult (*)(CUdevice, unsigned int*, int*);
  static GetFn get = nullptr;
  static StateFn state = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuDeviceGet", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get = reinterpret_cast<GetFn>(f);
    if (cudaGetDriverEntryPointByVersion("cuDevicePrimaryCtxGetState", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      state = reinterpret_cast<StateFn>(f);
  });
  CUdevice dev;
  unsigned int flags = 0;
  int active = 0;
  if (get && state && get(&dev, prev_) == CUDA_SUCCESS && state(dev, &flags, &active) == CUDA_SUCCESS && active)
    cudaSetDevice(prev_);
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool stride_ok(int64_t s) { return s >= 0 && (s % 8) == 0 && s < (int64_t(1) << 38); }

bool supported_dims(int dqk, int dv) {
  return (dqk == 64 && dv == 64) || (dqk == 128 && dv == 128) || (dqk == 192 && dv == 128);
}

// Shape-level checks shared by every entry point.
attn_status_t check_common(const attn_fwd_params* p, bool varlen) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  if (!supported_dims(p->d_qk, p->d_v)) {
    if (p->d_qk <= 0 || p->d_v <= 0) return ATTN_ERR_INVALID_ARG;
    return ATTN_ERR_UNSUPPORTED;
  }
  if (p->heads < 1) return ATTN_ERR_INVALID_ARG;
  if (!(std::isfinite(p->softmax_scale) && p->softmax_scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (varlen) {
    if (!p->cu_seqlens_q || !p->cu_seqlens_k) return ATTN_ERR_INVALID_ARG;
    if (p->num_seqs < 1 || p->total_q < 0 || p->total_k < 0) return ATTN_ERR_INVALID_ARG;
    if (p->max_seqlen_q < 0 || p->max_seqlen_k < 0) return ATTN_ERR_INVALID_ARG;
    if (p->max_seqlen_q > p->total_q || p->max_seqlen_k > p->total_k) return ATTN_ERR_INVALID_ARG;
  } else {
    if (p->cu_seqlens_q || p->cu_seqlens_k) return ATTN_ERR_INVALID_ARG;
    if (p->batch < 1 || p->seqlen_q < 0 || p->seqlen_k < 0) return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

// A tensor with no rows may have a null base pointer (an empty allocation).
attn_status_t check_tensor(const void* ptr, int64_t sb, int64_t sn, int64_t sh, bool varlen, bool empty = false) {
  if ((!ptr && !empty) || !aligned16(ptr)) return ATTN_ERR_INVALID_ARG;
  if (!stride_ok(sn) || !stride_ok(sh)) return ATTN_ERR_INVALID_ARG;
  if (!varlen && !stride_ok(sb)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

#define ATTN_TRY(x)                        \
  do {                                     \
    attn_status_t _s = (x);                \
    if (_s != ATTN_OK) return _s;          \
  } while (0)

bool no_q_rows(const attn_fwd_params* p, bool varlen) { return (varlen ? p->total_q : p->seqlen_q) == 0; }
bool no_k_rows(const attn_fwd_params* p, bool varlen) { return (varlen ? p->total_k : p->seqlen_k) == 0; }

attn_status_t check_fwd(const attn_fwd_params* p, bool varlen) {
  ATTN_TRY(check_common(p, varlen));
  const bool eq = no_q_rows(p, varlen), ek = no_k_rows(p, varlen);
  ATTN_TRY(check_tensor(p->q, p->q_batch_stride, p->q_row_stride, p->q_head_stride, varlen, eq));
  ATTN_TRY(check_tensor(p->k, p->k_batch_stride, p->k_row_stride, p->k_head_stride, varlen, ek));
  ATTN_TRY(check_tensor(p->v, p->v_batch_stride, p->v_row_stride, p->v_head_stride, varlen, ek));
  ATTN_TRY(check_tensor(p->o, p->o_batch_stride, p->o_row_stride, p->o_head_stride, varlen, eq));
  if ((!p->lse && !eq) || (reinterpret_cast<uintptr_t>(p->lse) & 3u)) return ATTN_ERR_INVALID_ARG;
  switch (p->score_mod) {
    case ATTN_SCORE_NONE: break;
    case ATTN_SCORE_SOFTCAP:
      if (!(std::isfinite(p->softcap) && p->softcap > 0.f && std::isfinite(p->softcap / p->softmax_scale)))
        return ATTN_ERR_INVALID_ARG;
      break;
    case ATTN_SCORE_ALIBI:
      if (!p->alibi_slopes || (reinterpret_cast<uintptr_t>(p->alibi_slopes) & 3u)) return ATTN_ERR_INVALID_ARG;
      break;
    default: return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

// Score-modification constants for the kernels (score_mod.cuh).
template <typename Args>
void fill_score_mod(Args& a, const attn_fwd_params* p) {
  a.score_mod = p->score_mod;
  a.inv_scale = 1.f / p->softmax_scale;
  a.alibi_slopes = p->score_mod == ATTN_SCORE_ALIBI ? p->alibi_slopes : nullptr;
  if (p->score_mod == ATTN_SCORE_SOFTCAP) {
    a.mod_k2 = 2.f * 1.4426950408889634f * (p->softmax_scale / p->softcap);
    a.mod_b = p->softcap / p->softmax_scale;
  }
}

// Arrays the kernels read besides the tensors (block lists, ALiBi slopes)
// must be device memory on the same GPU as the data: one on another GPU would
// be read across devices.
attn_status_t check_lists_device(const void* data, std::initializer_list<const void*> arrays) {
  if (!data) return ATTN_OK;  // no rows: nothing is launched
  cudaPointerAttributes ad{};
  if (cudaPointerGetAttributes(&ad, data) != cudaSuccess) return ATTN_ERR_INVALID_ARG;
  for (const void* p : arrays) {
    if (!p) continue;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) return ATTN_ERR_INVALID_ARG;
    if ((at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) || at.device != ad.device)
      return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

// Block-sparse key lists (nullptr kv_count: dense or varlen attention).
struct SparseSpec {
  const int32_t* kv_count = nullptr;
  const int32_t* kv_index = nullptr;
  int32_t max_kv = 0;
  int32_t lists_per_head = 0;
};

// Tile list of a packed variable-length launch (launch_tile_list): one
// 32-byte entry per CTA of a grid bounded by heads * (total / R + sequences),
// plus 8 bytes of scratch per sequence. Not built (the grid covers the longest
// sequence for every sequence instead) when a sequence may exceed
// kMaxListBlocks blocks.
struct ListPlan {
  bool use = false;
  int rows_per_block = 0, max_nblk = 0;
  int64_t bound = 0;
  size_t list_bytes = 0;
};
size_t round256(int64_t b) { return static_cast<size_t>((b + 255) / 256 * 256); }
ListPlan list_plan(int64_t total_rows, int num_seqs, int heads, int64_t max_len, int rows_per_block) {
  ListPlan lp;
  const int64_t max_nblk = (max_len + rows_per_block - 1) / rows_per_block;
  if (total_rows <= 0 || num_seqs < 1 || heads < 1 || max_nblk > kMaxListBlocks || max_nblk < 0) return lp;
  lp.use = true;
  lp.rows_per_block = rows_per_block;
  lp.max_nblk = static_cast<int>(max_nblk);
  lp.bound = static_cast<int64_t>(heads) * (total_rows / rows_per_block + num_seqs);
  lp.list_bytes = round256(lp.bound * static_cast<int64_t>(sizeof(TileEntry)));
  return lp;
}
size_t seq_scratch_bytes(int num_seqs) { return round256(static_cast<int64_t>(num_seqs) * 8); }

// Forward workspace: a 256-byte block holding the range flag, then the fp16
// copy of V ([rows, heads, d_v], contiguous) that the PV product reads, then
// (packed variable length) the tile list and its scratch, or (split keys) the
// ranges' fp32 O and LSE.
size_t fwd_v16_bytes(const attn_fwd_params* p, bool varlen) {
  if (p->heads < 1 || p->d_v <= 0) return 0;
  const int64_t rows = varlen ? static_cast<int64_t>(p->total_k) : static_cast<int64_t>(p->batch) * p->seqlen_k;
  if (rows <= 0) return 0;
  return static_cast<size_t>((rows * p->heads * p->d_v * 2 + 255) / 256 * 256);
}
ListPlan fwd_list_plan(const attn_fwd_params* p, bool varlen) {  // the pair forward takes no list
  return varlen && !p->cta_pair ? list_plan(p->total_q, p->num_seqs, p->heads, p->max_seqlen_q, 256) : ListPlan{};
}
// Split keys (dense): when the (query block, head, batch) grid would leave most
// SMs idle and the keys are long, each 256-row block's keys are cut into
// `splits` ranges of `per` 128-key blocks (at least kSplitMinBlocks each), one
// CTA per range, and a second kernel merges the ranges (split-KV). A function of
// the parameters alone, so the workspace size and the call agree.
constexpr int64_t kSplitTargetCtas = 148;  // at most one wave (148 SMs on B200, 152 on GB300)
constexpr int kSplitMinBlocks = 8;
constexpr int kSplitMax = 32;              // one merge lane per range
struct SplitPlan {
  int splits = 1, per = 0;
};
SplitPlan fwd_split_plan(const attn_fwd_params* p, bool varlen) {
  SplitPlan sp;
  if (varlen || p->cta_pair || p->input_dtype != ATTN_INPUT_BF16 || p->score_mod != ATTN_SCORE_NONE ||
      p->exp2_emu_period != 0 || p->d_qk != p->d_v || (p->d_qk != 64 && p->d_qk != 128))
    return sp;
  if (p->batch < 1 || p->heads < 1 || p->seqlen_q < 1 || p->seqlen_k < 1) return sp;
  const int64_t ctas = static_cast<int64_t>(p->batch) * p->heads * ((p->seqlen_q + 255) / 256);
  const int nkb = (p->seqlen_k + 127) / 128;
  if (ctas * 2 > kSplitTargetCtas || nkb < 2 * kSplitMinBlocks) return sp;
  // at most kSplitTargetCtas CTAs: a range count that spills a few CTAs into a
  // second wave costs as much as a whole extra wave
  int64_t s = std::min<int64_t>(kSplitTargetCtas / ctas, nkb / kSplitMinBlocks);
  s = std::min<int64_t>(s, kSplitMax);
  if (s < 2) return sp;
  sp.per = static_cast<int>((nkb + s - 1) / s);
  sp.splits = (nkb + sp.per - 1) / sp.per;  // no empty range
  if (sp.splits < 2) sp = SplitPlan{};
  return sp;
}
size_t fwd_split_bytes(const attn_fwd_params* p, const SplitPlan& sp) {
  if (sp.splits < 2) return 0;
  const int64_t rows = static_cast<int64_t>(p->batch) * p->heads * p->seqlen_q;
  return round256(sp.splits * rows * p->d_v * 4) + round256(sp.splits * rows * 4);
}
size_t fwd_workspace_bytes(const attn_fwd_params* p, bool varlen) {
  const size_t v16 = fwd_v16_bytes(p, varlen);
  if (!v16) return 0;
  const ListPlan lp = fwd_list_plan(p, varlen);
  return 256 + v16 + (lp.use ? lp.list_bytes + seq_scratch_bytes(p->num_seqs) : 0) +
         fwd_split_bytes(p, fwd_split_plan(p, varlen));
}

// diag_limit != 0: the diagnostic launch of attn_diag_wait_timeout instead of the forward.
attn_status_t run_fwd(const attn_fwd_params* p, bool varlen, cudaStream_t stream, void* ws, size_t ws_bytes,
                      const SparseSpec& sp = {}, uint32_t diag_limit = 0) {
  ATTN_TRY(check_fwd(p, varlen));
  if (p->exp2_emu_period != 0 && p->exp2_emu_period != 4 && p->exp2_emu_period != 8) return ATTN_ERR_INVALID_ARG;
  if (p->score_mod != ATTN_SCORE_NONE && (p->exp2_emu_period != 0 || diag_limit)) return ATTN_ERR_UNSUPPORTED;
  const bool f8 = p->input_dtype == ATTN_INPUT_E4M3;
  if (f8) {
    if (p->d_qk != 128 || p->d_v != 128 || p->exp2_emu_period != 0 || p->score_mod != ATTN_SCORE_NONE ||
        sp.kv_count != nullptr || diag_limit)
      return ATTN_ERR_UNSUPPORTED;
    for (float dsc : {p->q_descale, p->k_descale, p->v_descale})
      if (!(std::isfinite(dsc) && dsc > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(p->softmax_scale * p->q_descale * p->k_descale)) return ATTN_ERR_INVALID_ARG;
    for (int64_t st : {p->q_row_stride, p->q_head_stride, p->k_row_stride, p->k_head_stride, p->v_row_stride,
                       p->v_head_stride})
      if (st % 16) return ATTN_ERR_INVALID_ARG;  // TMA strides: multiples of 16 bytes
    if (!varlen && (p->q_batch_stride % 16 || p->k_batch_stride % 16 || p->v_batch_stride % 16))
      return ATTN_ERR_INVALID_ARG;
  } else if (p->input_dtype != ATTN_INPUT_BF16) {
    return ATTN_ERR_INVALID_ARG;
  }
  if (p->cta_pair && (p->d_qk != 128 || p->d_v != 128 || f8 || p->exp2_emu_period != 0 ||
                      p->score_mod != ATTN_SCORE_NONE || sp.kv_count != nullptr || diag_limit))
    return ATTN_ERR_UNSUPPORTED;
  const int nq_rows = varlen ? p->total_q : p->seqlen_q;
  const int nk_rows = varlen ? p->total_k : p->seqlen_k;
  const int units = varlen ? p->num_seqs : p->batch;
  const int max_q = varlen ? p->max_seqlen_q : p->seqlen_q;
  if (nq_rows == 0 || max_q == 0) return ATTN_OK;
  if (nk_rows > 0 && p->score_mod == ATTN_SCORE_ALIBI) ATTN_TRY(check_lists_device(p->q, {p->alibi_slopes}));
  const size_t need_ws = diag_limit ? 0 : fwd_workspace_bytes(p, varlen);
  if (nk_rows > 0 && need_ws > 0 && (ws == nullptr || ws_bytes < need_ws || (reinterpret_cast<uintptr_t>(ws) & 255u)))
    return ATTN_ERR_WORKSPACE;
  DeviceScope scope;
  {
    cudaError_t be = scope.bind(p->q ? p->q : p->k);
    if (be != cudaSuccess) return be == cudaErrorInvalidDevicePointer ? ATTN_ERR_INVALID_ARG : cuda_fail(be, "device");
  }

  FwdArgs a{};
  a.o = p->o;
  a.lse = p->lse;
  a.o_sb = p->o_batch_stride;
  a.o_sn = p->o_row_stride;
  a.o_sh = p->o_head_stride;
  a.batch = varlen ? 1 : p->batch;
  a.heads = p->heads;
  a.seqlen_q = varlen ? p->total_q : p->seqlen_q;
  a.seqlen_k = varlen ? p->total_k : p->seqlen_k;
  a.lse_sb = varlen ? 0 : static_cast<int64_t>(p->heads) * p->seqlen_q;
  a.lse_sh = varlen ? p->total_q : p->seqlen_q;
  a.cu_q = varlen ? p->cu_seqlens_q : nullptr;
  a.cu_k = varlen ? p->cu_seqlens_k : nullptr;
  a.num_units = units;
  a.n_mblk = p->cta_pair ? (max_q + 511) / 512 : (max_q + 255) / 256;  // 512-row blocks per CTA pair
  a.scale_log2 = p->softmax_scale * 1.4426950408889634f;
  if (f8) {  // S of the codes times both descales
    a.scale_log2 = p->softmax_scale * p->q_descale * p->k_descale * 1.4426950408889634f;
    a.input_e4m3 = 1;
    a.v_descale = p->v_descale;
  }
  a.causal = p->causal ? 1 : 0;
  a.stats = p->rescale_stats;
  a.emu_period = p->exp2_emu_period;
  a.kv_count = sp.kv_count;
  a.kv_index = sp.kv_index;
  a.max_kv = sp.max_kv;
  a.lists_per_head = sp.lists_per_head;
  a.spin_limit = diag_limit;
  a.n_groups = units * p->heads;
  if (p->causal && sp.kv_count == nullptr && a.n_mblk >= 8)  // heavy blocks first across a group of heads
    a.n_groups = group_count(units * p->heads, static_cast<int64_t>(varlen ? p->max_seqlen_k : p->seqlen_k) *
                                                   (p->d_qk * (f8 ? 1 : 2) + p->d_v * 2));
  fill_score_mod(a, p);
  cudaError_t e = status_ptr(&a.status);
  if (e != cudaSuccess) return cuda_fail(e, "status word");

  if (nk_rows == 0) {
    // No keys anywhere: every row is empty. Dense and packed layouts both
    // reduce to (units x heads x rows) with the strides above.
    FwdArgs z = a;
    if (varlen) {
      z.num_units = 1;
      z.seqlen_q = p->total_q;
    }
    e = launch_fwd_empty(z, p->d_v, stream);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "fwd empty launch");
  }

  const int nb = varlen ? 1 : p->batch;
  CUtensorMap tq, tk, tv;
  const int eb = f8 ? 1 : 2;
  ATTN_TRY(make_map(&tq, p->q, p->d_qk, p->heads, nq_rows, nb, p->q_batch_stride, p->q_row_stride,
                    p->q_head_stride, 128, eb));
  ATTN_TRY(make_map(&tk, p->k, p->d_qk, p->heads, nk_rows, nb, p->k_batch_stride, p->k_row_stride,
                    p->k_head_stride, 128, eb));
  ATTN_TRY(make_map(&tv, p->v, p->d_v, p->heads, nk_rows, nb, p->v_batch_stride, p->v_row_stride,
                    p->v_head_stride, 128, eb));
  if (diag_limit) {
    e = launch_fwd_diag_timeout(tq, tk, tv, a, stream);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "fwd diag launch");
  }
  // fp16 copy of V for the PV product, and its range flag
  uint32_t* flag = static_cast<uint32_t*>(ws);
  void* v16 = static_cast<uint8_t*>(ws) + 256;
  const int64_t v16_rows = varlen ? p->total_k : p->seqlen_k;
  CUtensorMap tv16;
  ATTN_TRY(make_map(&tv16, v16, p->d_v, p->heads, nk_rows, nb, v16_rows * p->heads * p->d_v,
                    static_cast<int64_t>(p->heads) * p->d_v, p->d_v, 128));
  e = cudaMemsetAsync(flag, 0, sizeof(uint32_t), stream);
  if (e == cudaSuccess && f8)  // exact: every E4M3 value is an fp16 value, the flag stays 0
    e = launch_v_e4m3_to_f16(p->v, varlen ? 0 : p->v_batch_stride, p->v_row_stride, p->v_head_stride, nb, nk_rows,
                             p->heads, p->d_v, v16, stream);
  else if (e == cudaSuccess)
    e = launch_v_to_f16(p->v, varlen ? 0 : p->v_batch_stride, p->v_row_stride, p->v_head_stride, nb, nk_rows,
                        p->heads, p->d_v, v16, flag, stream);
  if (e != cudaSuccess) return cuda_fail(e, "fwd V conversion");
  a.v16_flag = flag;
  const ListPlan lp = fwd_list_plan(p, varlen);
  if (lp.use) {  // longest sequences first, no CTA past a sequence's end
    uint8_t* lbase = static_cast<uint8_t*>(ws) + 256 + fwd_v16_bytes(p, varlen);
    TileEntry* list = reinterpret_cast<TileEntry*>(lbase);
    int64_t* scratch = reinterpret_cast<int64_t*>(lbase + lp.list_bytes);
    e = launch_tile_list(p->cu_seqlens_q, p->cu_seqlens_k, p->num_seqs, p->heads, 256, false, true, lp.max_nblk, list,
                         scratch, lp.bound, stream);
    if (e != cudaSuccess) return cuda_fail(e, "fwd tile list");
    a.tiles = list;
    a.n_tiles = lp.bound;
  }
  const SplitPlan spl = (sp.kv_count || p->cta_pair || f8) ? SplitPlan{} : fwd_split_plan(p, varlen);
  if (spl.splits > 1) {  // fp32 O and LSE of every key range, after the fp16 copy of V
    uint8_t* pbase = static_cast<uint8_t*>(ws) + 256 + fwd_v16_bytes(p, varlen);
    a.kv_split = spl.splits;
    a.kv_blocks_per_split = spl.per;
    a.part_rows = static_cast<int64_t>(p->batch) * p->heads * p->seqlen_q;
    a.o_part = reinterpret_cast<float*>(pbase);
    a.lse_part = reinterpret_cast<float*>(pbase + round256(spl.splits * a.part_rows * p->d_v * 4));
  }
  if (p->cta_pair) {
    CUtensorMap tk_h;  // 64-key boxes: each CTA of a pair loads half of every K tile
    ATTN_TRY(make_map(&tk_h, p->k, p->d_qk, p->heads, nk_rows, nb, p->k_batch_stride, p->k_row_stride,
                      p->k_head_stride, 64));
    e = launch_fwd_pair(tq, tk_h, tv, tv16, a, stream);
  } else if (f8) {
    e = launch_fwd_e4m3(tq, tk, tv16, a, stream);
  } else if (sp.kv_count) {
    e = launch_fwd_sparse(p->d_qk, p->d_v, tq, tk, tv, tv16, a, stream);
  } else {
    e = launch_fwd(p->d_qk, p->d_v, tq, tk, tv, tv16, a, stream);
  }
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "fwd launch");
}


int bwd_dkdv_rows(int d_qk) { return d_qk == 128 ? 128 : 64; }  // query rows per step of the dK/dV kernel

// Backward workspace: D (4 bytes per query row and head), then (packed
// variable length) the dK/dV and dQ tile lists and their scratch. Invalid
// (negative) shapes need no workspace: the call itself reports them.
size_t bwd_d_bytes(const attn_bwd_params* p, bool varlen) {
  const attn_fwd_params& f = p->fwd;
  if (f.heads < 0 || (varlen ? f.total_q < 0 : (f.batch < 0 || f.seqlen_q < 0))) return 0;
  const int64_t rows = varlen ? static_cast<int64_t>(f.heads) * f.total_q
                              : static_cast<int64_t>(f.batch) * f.heads * f.seqlen_q;
  return round256(rows * 4);
}
ListPlan bwd_kv_plan(const attn_bwd_params* p, bool varlen) {
  const attn_fwd_params& f = p->fwd;
  return varlen && !p->cta_pair ? list_plan(f.total_k, f.num_seqs, f.heads, f.max_seqlen_k, 128) : ListPlan{};
}
ListPlan bwd_q_plan(const attn_bwd_params* p, bool varlen) {
  const attn_fwd_params& f = p->fwd;
  return varlen ? list_plan(f.total_q, f.num_seqs, f.heads, f.max_seqlen_q, 128) : ListPlan{};
}
// Single pass (d = 64): the fp32 dQ buffer, 4 bytes per query row, head and
// column, then (deterministic) one int32 semaphore per (unit, head, 64-row tile).
size_t bwd_dq_acc_bytes(const attn_bwd_params* p, bool varlen) {
  const attn_fwd_params& f = p->fwd;
  if (!p->single_pass || f.heads < 0 || (varlen ? f.total_q < 0 : (f.batch < 0 || f.seqlen_q < 0))) return 0;
  const int64_t rows = varlen ? static_cast<int64_t>(f.heads) * f.total_q
                              : static_cast<int64_t>(f.batch) * f.heads * f.seqlen_q;
  return round256(rows * f.d_qk * 4);
}
int64_t bwd_n_qt64(const attn_bwd_params* p, bool varlen) {
  const attn_fwd_params& f = p->fwd;
  return ((varlen ? static_cast<int64_t>(f.max_seqlen_q) : f.seqlen_q) + 63) / 64;
}
size_t bwd_sem_bytes(const attn_bwd_params* p, bool varlen) {
  const attn_fwd_params& f = p->fwd;
  if (!p->single_pass || !p->deterministic || f.heads < 0) return 0;
  const int64_t units = varlen ? f.num_seqs : f.batch;
  if (units < 0 || bwd_n_qt64(p, varlen) < 0) return 0;
  return round256(units * f.heads * bwd_n_qt64(p, varlen) * 4);
}
// Split keys for the dQ kernel (dense two-kernel backward): when the dQ grid's
// batch x heads x ceil(seqlen_q / 128) query tiles would leave most SMs idle and
// the keys are long, each tile's key blocks are cut into ranges as the forward
// does (fwd_split_plan), one CTA per range, each writing its fp32 dQ partial;
// a merge kernel adds them in range order. A function of the parameters alone.
SplitPlan bwd_dq_split_plan(const attn_bwd_params* p, bool varlen) {
  SplitPlan sp;
  const attn_fwd_params& f = p->fwd;
  if (varlen || p->single_pass || f.input_dtype != ATTN_INPUT_BF16) return sp;
  if (!((f.d_qk == 64 && f.d_v == 64) || (f.d_qk == 128 && f.d_v == 128) || (f.d_qk == 192 && f.d_v == 128)))
    return sp;
  if (f.batch < 1 || f.heads < 1 || f.seqlen_q < 1 || f.seqlen_k < 1) return sp;
  const int64_t ctas = static_cast<int64_t>(f.batch) * f.heads * ((f.seqlen_q + 127) / 128);
  const int nkb = (f.seqlen_k + 127) / 128;
  if (ctas * 2 > kSplitTargetCtas || nkb < 2 * kSplitMinBlocks) return sp;
  int64_t s = std::min<int64_t>(kSplitTargetCtas / ctas, nkb / kSplitMinBlocks);
  s = std::min<int64_t>(s, kSplitMax);
  if (s < 2) return sp;
  sp.per = static_cast<int>((nkb + s - 1) / s);
  sp.splits = (nkb + sp.per - 1) / sp.per;
  if (sp.splits < 2) sp = SplitPlan{};
  return sp;
}
size_t bwd_dq_split_bytes(const attn_bwd_params* p, const SplitPlan& sp) {
  if (sp.splits < 2) return 0;
  const attn_fwd_params& f = p->fwd;
  return round256(static_cast<int64_t>(sp.splits) * f.batch * f.heads * f.seqlen_q * f.d_qk * 4);
}
// The workspace without the split-key dQ partials (the least a call accepts).
size_t bwd_workspace_bytes(const attn_bwd_params* p, bool varlen) {
  const size_t d = bwd_d_bytes(p, varlen);
  const size_t fused = bwd_dq_acc_bytes(p, varlen) + bwd_sem_bytes(p, varlen);
  if (!varlen) return d + fused;
  const ListPlan kv = bwd_kv_plan(p, varlen), q = bwd_q_plan(p, varlen);
  const size_t lists = (kv.use ? kv.list_bytes : 0) + (q.use ? q.list_bytes : 0);
  return d + lists + (lists ? seq_scratch_bytes(p->fwd.num_seqs) : 0) + fused;
}

// Extra workspace of the block-sparse backward: the transposed lists
// (int32 q_count[sets][n_kb], then q_index[sets][n_kb][n_qb256]) after the D
// vector; sets = batch * heads for lists per (batch, head), else 1.
int64_t list_sets(const attn_fwd_params& f, int32_t lists_per_head) {
  return lists_per_head ? static_cast<int64_t>(f.batch) * f.heads : 1;
}
size_t bwd_sparse_extra_bytes(const attn_fwd_params& f, int32_t lists_per_head) {
  const int64_t n_kb = (static_cast<int64_t>(f.seqlen_k) + 127) / 128 * list_sets(f, lists_per_head);
  const int64_t n_qb = (static_cast<int64_t>(f.seqlen_q) + 255) / 256;
  return static_cast<size_t>((n_kb * 4 + 255) / 256 * 256 + (n_kb * n_qb * 4 + 255) / 256 * 256);
}

attn_status_t run_bwd(const attn_bwd_params* p, void* ws, size_t ws_bytes, bool varlen, cudaStream_t stream,
                      const SparseSpec& sp = {}) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  const attn_fwd_params& f = p->fwd;
  ATTN_TRY(check_fwd(&f, varlen));
  const bool eq = no_q_rows(&f, varlen), ek = no_k_rows(&f, varlen);
  ATTN_TRY(check_tensor(p->dout, p->do_batch_stride, p->do_row_stride, p->do_head_stride, varlen, eq));
  ATTN_TRY(check_tensor(p->dq, p->dq_batch_stride, p->dq_row_stride, p->dq_head_stride, varlen, eq));
  ATTN_TRY(check_tensor(p->dk, p->dk_batch_stride, p->dk_row_stride, p->dk_head_stride, varlen, ek));
  ATTN_TRY(check_tensor(p->dv, p->dv_batch_stride, p->dv_row_stride, p->dv_head_stride, varlen, ek));
  if (p->cta_pair && (f.d_qk != 128 || f.d_v != 128 || sp.kv_count || f.score_mod != ATTN_SCORE_NONE))
    return ATTN_ERR_UNSUPPORTED;
  if (f.input_dtype != ATTN_INPUT_BF16)  // E4M3 is a forward-only input type
    return f.input_dtype == ATTN_INPUT_E4M3 ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID_ARG;
  if (p->single_pass && (f.d_qk != 64 || f.d_v != 64 || sp.kv_count || f.score_mod != ATTN_SCORE_NONE ||
                         p->cta_pair))
    return ATTN_ERR_UNSUPPORTED;
  const int nq_rows = varlen ? f.total_q : f.seqlen_q;
  const int nk_rows = varlen ? f.total_k : f.seqlen_k;
  if (nq_rows == 0 && nk_rows == 0) return ATTN_OK;
  DeviceScope scope;
  {
    cudaError_t be = scope.bind(nq_rows ? f.q : f.k);
    if (be != cudaSuccess) return be == cudaErrorInvalidDevicePointer ? ATTN_ERR_INVALID_ARG : cuda_fail(be, "device");
  }
  const size_t need_d = bwd_workspace_bytes(p, varlen);
  const size_t need = need_d + (sp.kv_count ? bwd_sparse_extra_bytes(f, sp.lists_per_head) : 0);
  // split-key dQ (after the rest of the workspace) only when the caller's workspace holds its partials
  SplitPlan dqs = (sp.kv_count || nq_rows == 0 || nk_rows == 0) ? SplitPlan{} : bwd_dq_split_plan(p, varlen);
  if (dqs.splits > 1 && ws_bytes < need + bwd_dq_split_bytes(p, dqs)) dqs = SplitPlan{};
  if (nq_rows > 0 && nk_rows > 0 && f.score_mod == ATTN_SCORE_ALIBI) ATTN_TRY(check_lists_device(f.q, {f.alibi_slopes}));
  if (nq_rows > 0 && nk_rows > 0 && (ws == nullptr || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 15u)))
    return ATTN_ERR_WORKSPACE;

  BwdArgs a{};
  a.o = f.o;
  a.dout = p->dout;
  a.lse = f.lse;
  a.dsum = static_cast<float*>(ws);
  a.dq = p->dq;
  a.dk = p->dk;
  a.dv = p->dv;
  a.o_sb = f.o_batch_stride, a.o_sn = f.o_row_stride, a.o_sh = f.o_head_stride;
  a.do_sb = p->do_batch_stride, a.do_sn = p->do_row_stride, a.do_sh = p->do_head_stride;
  a.dq_sb = p->dq_batch_stride, a.dq_sn = p->dq_row_stride, a.dq_sh = p->dq_head_stride;
  a.dk_sb = p->dk_batch_stride, a.dk_sn = p->dk_row_stride, a.dk_sh = p->dk_head_stride;
  a.dv_sb = p->dv_batch_stride, a.dv_sn = p->dv_row_stride, a.dv_sh = p->dv_head_stride;
  if (varlen) a.o_sb = a.do_sb = a.dq_sb = a.dk_sb = a.dv_sb = 0;
  a.lse_sb = varlen ? 0 : static_cast<int64_t>(f.heads) * f.seqlen_q;
  a.lse_sh = varlen ? f.total_q : f.seqlen_q;
  a.batch = varlen ? 1 : f.batch;
  a.heads = f.heads;
  a.seqlen_q = nq_rows;
  a.seqlen_k = nk_rows;
  a.cu_q = varlen ? f.cu_seqlens_q : nullptr;
  a.cu_k = varlen ? f.cu_seqlens_k : nullptr;
  a.num_units = varlen ? f.num_seqs : f.batch;
  const int max_q = varlen ? f.max_seqlen_q : f.seqlen_q;
  const int max_k = varlen ? f.max_seqlen_k : f.seqlen_k;
  a.n_qblk = (max_q + 127) / 128;
  a.n_kblk = (max_k + 127) / 128;
  a.scale = f.softmax_scale;
  a.scale_log2 = f.softmax_scale * 1.4426950408889634f;
  a.causal = f.causal ? 1 : 0;
  a.n_groups = a.num_units * f.heads;
  // heavy blocks first across a group of heads (the deterministic single pass keeps its add order)
  if (f.causal && sp.kv_count == nullptr && !(p->single_pass && p->deterministic) && a.n_kblk >= 16)
    a.n_groups = group_count(a.num_units * f.heads,
                             static_cast<int64_t>(max_q > max_k ? max_q : max_k) * (f.d_qk + f.d_v) * 2);
  fill_score_mod(a, &f);
  const int n_kb_sparse = (f.seqlen_k + 127) / 128;
  if (sp.kv_count) {
    a.kv_count = sp.kv_count;
    a.kv_index = sp.kv_index;
    a.max_kv = sp.max_kv;
    a.n_qb256 = (f.seqlen_q + 255) / 256;
    a.lists_per_head = sp.lists_per_head;
    const int64_t n_kb_all = static_cast<int64_t>(n_kb_sparse) * list_sets(f, sp.lists_per_head);
    uint8_t* extra = static_cast<uint8_t*>(ws) + need_d;
    a.q_count = reinterpret_cast<int*>(extra);
    a.q_index = reinterpret_cast<int*>(extra + (static_cast<size_t>(n_kb_all) * 4 + 255) / 256 * 256);
  }
  cudaError_t e = status_ptr(&a.status);
  if (e != cudaSuccess) return cuda_fail(e, "status word");

  if (nq_rows > 0 && nk_rows > 0 && varlen) {  // tile lists: longest sequences first, no CTA past an end
    const ListPlan kv = bwd_kv_plan(p, varlen), qp = bwd_q_plan(p, varlen);
    uint8_t* lbase = static_cast<uint8_t*>(ws) + bwd_d_bytes(p, varlen);
    int64_t* scratch = reinterpret_cast<int64_t*>(lbase + (kv.use ? kv.list_bytes : 0) + (qp.use ? qp.list_bytes : 0));
    if (kv.use) {
      TileEntry* list = reinterpret_cast<TileEntry*>(lbase);
      // the deterministic single pass launches key tiles in descending order (its adds' order)
      const bool desc = p->single_pass && p->deterministic;
      e = launch_tile_list(f.cu_seqlens_q, f.cu_seqlens_k, f.num_seqs, f.heads, 128, true, desc, kv.max_nblk, list,
                           scratch, kv.bound, stream);
      if (e != cudaSuccess) return cuda_fail(e, "bwd tile list");
      a.tiles_kv = list;
      a.n_tiles_kv = kv.bound;
      lbase += kv.list_bytes;
    }
    if (qp.use) {
      TileEntry* list = reinterpret_cast<TileEntry*>(lbase);
      e = launch_tile_list(f.cu_seqlens_q, f.cu_seqlens_k, f.num_seqs, f.heads, 128, false, true, qp.max_nblk, list,
                           scratch, qp.bound, stream);
      if (e != cudaSuccess) return cuda_fail(e, "bwd tile list");
      a.tiles_q = list;
      a.n_tiles_q = qp.bound;
    }
  }

  if (nq_rows == 0 || nk_rows == 0) {
    // Nothing to differentiate through: no queries -> dK = dV = 0; no keys -> dQ = 0.
    e = launch_bwd_zero(a, f.d_qk, f.d_v, nk_rows == 0, nq_rows == 0, stream);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "bwd zero launch");
  }

  const int nb = varlen ? 1 : f.batch;
  const int qrows = bwd_dkdv_rows(f.d_qk);
  CUtensorMap tq, tk, tv, tdo, tq2, tdo2;
  ATTN_TRY(make_map(&tq, f.q, f.d_qk, f.heads, nq_rows, nb, f.q_batch_stride, f.q_row_stride, f.q_head_stride, 128));
  ATTN_TRY(make_map(&tk, f.k, f.d_qk, f.heads, nk_rows, nb, f.k_batch_stride, f.k_row_stride, f.k_head_stride, 128));
  ATTN_TRY(make_map(&tv, f.v, f.d_v, f.heads, nk_rows, nb, f.v_batch_stride, f.v_row_stride, f.v_head_stride, 128));
  ATTN_TRY(make_map(&tdo, p->dout, f.d_v, f.heads, nq_rows, nb, p->do_batch_stride, p->do_row_stride,
                    p->do_head_stride, 128));
  ATTN_TRY(make_map(&tq2, f.q, f.d_qk, f.heads, nq_rows, nb, f.q_batch_stride, f.q_row_stride, f.q_head_stride,
                    qrows));
  ATTN_TRY(make_map(&tdo2, p->dout, f.d_v, f.heads, nq_rows, nb, p->do_batch_stride, p->do_row_stride,
                    p->do_head_stride, qrows));
  auto mark = [&](int i) -> cudaError_t {
    return p->phase_events[i] ? cudaEventRecord(static_cast<cudaEvent_t>(p->phase_events[i]), stream) : cudaSuccess;
  };
  e = launch_bwd_preprocess(f.d_v, a, stream);
  if (e == cudaSuccess && sp.kv_count) e = launch_bwd_transpose_lists(a, n_kb_sparse, stream);
  if (e == cudaSuccess) e = mark(0);
  if (e != cudaSuccess) return cuda_fail(e, "bwd preprocess launch");
  if (p->single_pass) {  // dK, dV and the dQ partials in one kernel, then dQ * scale to bf16
    uint8_t* tail = static_cast<uint8_t*>(ws) + bwd_workspace_bytes(p, varlen) - bwd_dq_acc_bytes(p, varlen) -
                    bwd_sem_bytes(p, varlen);
    a.dq_acc = reinterpret_cast<float*>(tail);
    a.dq_sem = p->deterministic ? reinterpret_cast<int*>(tail + bwd_dq_acc_bytes(p, varlen)) : nullptr;
    a.n_qt64 = static_cast<int>(bwd_n_qt64(p, varlen));
    e = cudaMemsetAsync(tail, 0, bwd_dq_acc_bytes(p, varlen) + bwd_sem_bytes(p, varlen), stream);
    if (e == cudaSuccess) e = launch_bwd_single_pass(tq2, tk, tv, tdo2, a, stream);
    if (e == cudaSuccess) e = mark(1);
    if (e == cudaSuccess) e = launch_bwd_dq_convert(a, f.d_qk, stream);
    if (e == cudaSuccess) e = mark(2);
    return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "bwd single-pass launch");
  }
  if (p->cta_pair) {  // the two-SM kernel (d = 128, no block lists; checked before any launch)
    CUtensorMap tq_r, tdo_r;
    ATTN_TRY(make_map(&tq_r, f.q, f.d_qk, f.heads, nq_rows, nb, f.q_batch_stride, f.q_row_stride, f.q_head_stride,
                      64));
    ATTN_TRY(make_map(&tdo_r, p->dout, f.d_v, f.heads, nq_rows, nb, p->do_batch_stride, p->do_row_stride,
                      p->do_head_stride, 64));
    e = launch_bwd_dkdv_pair(tq_r, tq2, tk, tv, tdo_r, tdo2, a, stream);
  } else {
    e = launch_bwd_dkdv(f.d_qk, f.d_v, tq2, tk, tv, tdo2, a, stream);
  }
  if (e == cudaSuccess) e = mark(1);
  if (e != cudaSuccess) return cuda_fail(e, "bwd dkdv launch");
  if (dqs.splits > 1) {
    a.dq_split = dqs.splits;
    a.dq_kb_per_split = dqs.per;
    a.dq_part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + need);
  }
  e = launch_bwd_dq(f.d_qk, f.d_v, tq, tk, tv, tdo, a, stream);
  if (e == cudaSuccess && dqs.splits > 1) e = launch_bwd_dq_merge(a, f.d_qk, stream);
  if (e == cudaSuccess) e = mark(2);
  if (e != cudaSuccess) return cuda_fail(e, "bwd dq launch");
  return ATTN_OK;
}

}  // namespace

size_t bwd_workspace_min_size(const attn_bwd_params* p) {
  return bwd_workspace_bytes(p, p->fwd.cu_seqlens_q != nullptr);
}

}  // namespace gb300

using namespace gb300;

extern "C" {

size_t attn_fwd_workspace_size(const attn_fwd_params* p) {
  if (!p) return 0;
  return fwd_workspace_bytes(p, p->cu_seqlens_q != nullptr);
}

attn_status_t attn_fwd(const attn_fwd_params* p, void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  return run_fwd(p, false, static_cast<cudaStream_t>(stream), workspace, workspace_bytes);
}

attn_status_t attn_fwd_varlen(const attn_fwd_params* p, void* workspace, size_t workspace_bytes,
                              attn_stream_t stream) {
  return run_fwd(p, true, static_cast<cudaStream_t>(stream), workspace, workspace_bytes);
}

// Shared checks of the block lists; fills `sp`.
attn_status_t check_block_lists(const attn_fwd_params* p, const int32_t* kv_count, const int32_t* kv_index,
                                int32_t max_kv, int32_t lists_per_head, bool backward, SparseSpec* sp) {
  if (lists_per_head != 0 && lists_per_head != 1) return ATTN_ERR_INVALID_ARG;
  const int64_t sets = list_sets(*p, lists_per_head);
  const int64_t n_qblk = (static_cast<int64_t>(p->seqlen_q) + 255) / 256 * sets;
  const int64_t n_kblk = (static_cast<int64_t>(p->seqlen_k) + 127) / 128 * sets;
  if (max_kv < 0 || n_qblk * max_kv > 0x7fffffff) return ATTN_ERR_INVALID_ARG;
  if (backward && n_kblk * ((static_cast<int64_t>(p->seqlen_q) + 255) / 256) > 0x7fffffff) return ATTN_ERR_INVALID_ARG;
  if (n_qblk > 0) {
    if (!kv_count || (reinterpret_cast<uintptr_t>(kv_count) & 3u)) return ATTN_ERR_INVALID_ARG;
    if (max_kv > 0 && (!kv_index || (reinterpret_cast<uintptr_t>(kv_index) & 3u))) return ATTN_ERR_INVALID_ARG;
    ATTN_TRY(check_lists_device(p->q, {kv_count, max_kv > 0 ? kv_index : nullptr}));
  }
  sp->kv_count = kv_count;
  sp->kv_index = kv_index;
  sp->max_kv = max_kv;
  sp->lists_per_head = lists_per_head;
  return ATTN_OK;
}

attn_status_t attn_fwd_block_sparse(const attn_fwd_params* p, const int32_t* kv_count, const int32_t* kv_index,
                                    int32_t max_kv, int32_t lists_per_head, void* workspace, size_t workspace_bytes,
                                    attn_stream_t stream) {
  ATTN_TRY(check_fwd(p, false));
  if (p->exp2_emu_period != 0) return ATTN_ERR_INVALID_ARG;
  if (p->input_dtype != ATTN_INPUT_BF16)  // E4M3 inputs: dense and varlen forward only
    return p->input_dtype == ATTN_INPUT_E4M3 ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID_ARG;
  SparseSpec sp;
  ATTN_TRY(check_block_lists(p, kv_count, kv_index, max_kv, lists_per_head, false, &sp));
  return run_fwd(p, false, static_cast<cudaStream_t>(stream), workspace, workspace_bytes, sp);
}

size_t attn_bwd_block_sparse_workspace_size(const attn_bwd_params* p, int32_t lists_per_head) {
  if (!p || p->fwd.cu_seqlens_q != nullptr || (lists_per_head != 0 && lists_per_head != 1)) return 0;
  if (p->fwd.batch < 0 || p->fwd.heads < 0 || p->fwd.seqlen_q < 0 || p->fwd.seqlen_k < 0) return 0;
  return bwd_workspace_bytes(p, false) + bwd_sparse_extra_bytes(p->fwd, lists_per_head);
}

attn_status_t attn_bwd_block_sparse(const attn_bwd_params* p, const int32_t* kv_count, const int32_t* kv_index,
                                    int32_t max_kv, int32_t lists_per_head, void* workspace, size_t workspace_bytes,
                                    attn_stream_t stream) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  ATTN_TRY(check_fwd(&p->fwd, false));
  SparseSpec sp;
  ATTN_TRY(check_block_lists(&p->fwd, kv_count, kv_index, max_kv, lists_per_head, true, &sp));
  return run_bwd(p, workspace, workspace_bytes, false, static_cast<cudaStream_t>(stream), sp);
}

size_t attn_bwd_workspace_size(const attn_bwd_params* p) {
  if (!p) return 0;
  const bool varlen = p->fwd.cu_seqlens_q != nullptr;
  return bwd_workspace_bytes(p, varlen) + bwd_dq_split_bytes(p, bwd_dq_split_plan(p, varlen));
}

attn_status_t attn_bwd(const attn_bwd_params* p, void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  return run_bwd(p, workspace, workspace_bytes, false, static_cast<cudaStream_t>(stream));
}

attn_status_t attn_bwd_varlen(const attn_bwd_params* p, void* workspace, size_t workspace_bytes,
                              attn_stream_t stream) {
  return run_bwd(p, workspace, workspace_bytes, true, static_cast<cudaStream_t>(stream));
}

attn_status_t attn_exp2_eval(const float* x, float* y_poly, float* y_hw, int64_t n, attn_stream_t stream) {
  if (n < 0 || (n > 0 && !x) || (!y_poly && !y_hw)) return ATTN_ERR_INVALID_ARG;
  if (n == 0) return ATTN_OK;
  DeviceScope scope;
  {
    cudaError_t be = scope.bind(x);
    if (be != cudaSuccess) return be == cudaErrorInvalidDevicePointer ? ATTN_ERR_INVALID_ARG : cuda_fail(be, "device");
  }
  cudaError_t e = launch_exp2_eval(x, y_poly, y_hw, n, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e, "exp2 eval launch");
}

attn_status_t attn_diag_wait_timeout(const attn_fwd_params* p, uint32_t spin_limit, attn_stream_t stream) {
  ATTN_TRY(check_fwd(p, false));
  if (p->d_qk != 64 || p->d_v != 64 || p->exp2_emu_period != 0) return ATTN_ERR_INVALID_ARG;
  if (spin_limit < 1 || spin_limit > (1u << 20)) return ATTN_ERR_INVALID_ARG;
  if (p->seqlen_q == 0 || p->seqlen_k == 0) return ATTN_ERR_INVALID_ARG;  // the kernel must launch
  return run_fwd(p, false, static_cast<cudaStream_t>(stream), nullptr, 0, SparseSpec{}, spin_limit);
}

attn_status_t attn_get_device_status(attn_stream_t stream, uint32_t* detail) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream sync");
  uint32_t* d = nullptr;
  e = status_ptr(&d);
  if (e != cudaSuccess) return cuda_fail(e, "status word");
  uint32_t v = 0;
  e = cudaMemcpy(&v, d, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (v != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpy(d, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
  }
  if (detail) *detail = v;
  return v == 0 ? ATTN_OK : ATTN_ERR_TIMEOUT;
}

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
  }
  return "ATTN_ERR_UNKNOWN";
}

const char* attn_last_cuda_error(void) { return t_last_cuda_error; }

int32_t attn_abi_version(void) { return ATTN_ABI_VERSION; }
size_t attn_fwd_params_size(void) { return sizeof(attn_fwd_params); }
size_t attn_bwd_params_size(void) { return sizeof(attn_bwd_params); }

}  // extern "C"
