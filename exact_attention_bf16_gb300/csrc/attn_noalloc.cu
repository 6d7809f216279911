// attn_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory. It needs no counterpart in the attention method itself; it only
// changes where the backward's scratch lives.
//
// Who needs it: code that runs where allocation is not allowed or not
// possible, for example an inference or training runtime that plans all
// device memory up front and forbids cudaMalloc afterwards (a fixed memory
// budget, or a pool that owns the whole device), a plugin whose host
// framework hands it only the tensors, or a latency-sensitive loop in which a
// cudaMalloc (which may synchronise the device) is not acceptable. attn_bwd
// asks such callers for a workspace they would have to allocate; this entry
// point takes none.
//
// The scratch (D_i = dO_i . O_i, 4 bytes per (batch, head, query row)) lives
// in a file-scope __device__ array of ATTN_BWD_NOALLOC_SCRATCH_BYTES, which
// every GPU that loads this library holds until the process exits. On the
// first call on a device the array's device address is looked up with
// cudaGetSymbolAddress (with that device current) and cached; that first call
// should therefore come before any stream capture. Larger problems are
// rejected with ATTN_ERR_WORKSPACE. All calls share the one array: calls that
// can overlap on the GPU (different streams, or another thread) race on it and
// must be serialised by the caller. Nothing in the array has to start at zero:
// the D pass writes every entry that the dK/dV and dQ kernels read, so the
// previous call's contents are never used.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/attn.h"
#include "kernels.h"

namespace gb300 {
// The backward's workspace without the optional split-key dQ partials.
size_t bwd_workspace_min_size(const attn_bwd_params* p);
}  // namespace gb300

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[ATTN_BWD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_bwd_scratch on `dev`, which must be the current device.
cudaError_t scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" attn_status_t attn_bwd_noalloc(const attn_bwd_params* p, attn_stream_t stream) {
  if (!p) return ATTN_ERR_INVALID_ARG;
  const attn_fwd_params& f = p->fwd;
  const bool varlen = f.cu_seqlens_q != nullptr;
  // Shapes first: a negative size is a bad argument, not a problem too large
  // for the scratch (the workspace size is 0 for it).
  if (f.heads < 1 || (varlen ? (f.total_q < 0 || f.total_k < 0) : (f.batch < 1 || f.seqlen_q < 0 || f.seqlen_k < 0)))
    return ATTN_ERR_INVALID_ARG;
  // the workspace without the optional split-key dQ partials, which the
  // backward uses only when the scratch also holds them
  const size_t need = gb300::bwd_workspace_min_size(p);
  if (need > ATTN_BWD_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_WORKSPACE;  // problem too large for the fixed scratch
  const int nq = varlen ? f.total_q : f.seqlen_q;
  const int nk = varlen ? f.total_k : f.seqlen_k;
  void* ws = nullptr;
  if (nq > 0 && nk > 0) {
    // Set-up: with the data's device current, resolve the array's address on
    // it; the caller's current device is restored when `scope` ends.
    if (!f.q) return ATTN_ERR_INVALID_ARG;
    gb300::DeviceScope scope;
    const cudaError_t e = scope.bind(f.q);
    if (e == cudaErrorInvalidDevicePointer) return ATTN_ERR_INVALID_ARG;
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
    if (scratch_address(scope.device(), &ws) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  return varlen ? attn_bwd_varlen(p, ws, ATTN_BWD_NOALLOC_SCRATCH_BYTES, stream)
                : attn_bwd(p, ws, ATTN_BWD_NOALLOC_SCRATCH_BYTES, stream);
}
