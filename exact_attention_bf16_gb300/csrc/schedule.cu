// Work lists for packed variable-length batches (the tile scheduler for
// variable-length balance of newton wiki "FlashAttention-4", 核心技術).
//
// A variable-length launch has one CTA per (sequence, head, block of R rows).
// Without a list the grid must be sized for the longest sequence in every
// sequence, and the CTAs past a shorter sequence's end start only to exit;
// the sequences also run in their packed order, so a long sequence packed last
// leaves the GPU half idle at the end. The list built here has exactly one
// entry per real block, ordered so that the sequences with the most blocks
// come first (longest processing time first), then head by head, then the
// blocks of each head heaviest first as the kernels' own order has them, so
// that a head's CTAs still run together and share its K/V in L2. The grid is
// sized by an upper bound the host knows (heads * (total / R + sequences));
// entries past the real count are empty and their CTAs exit at once.
//
// One block builds the list: a counting sort of the sequences by block count
// (bins in shared memory), a scan over the bins from the largest count down,
// then one warp per sequence writes its entries. Sequences with the same
// block count are placed in arrival order of an atomic counter; the order
// affects only scheduling, never a result.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace gb300 {
namespace sched {

constexpr int kThreads = 1024;

__global__ void __launch_bounds__(kThreads, 1)
    tile_list_kernel(const int* cu_q, const int* cu_k, int num_seqs, int heads, int rows_per_block, int by_keys,
                     int descending, int max_nblk, TileEntry* out, int64_t* seq_start, int64_t bound) {
  __shared__ int bins[kMaxListBlocks + 1];          // sequences per block count, then cursors
  __shared__ long long bin_start[kMaxListBlocks + 1];  // first entry of each block count
  __shared__ long long chunk_sum[kThreads];
  const int tid = static_cast<int>(threadIdx.x);
  const int nb = max_nblk + 1;
  for (int b = tid; b < nb; b += kThreads) bins[b] = 0;
  __syncthreads();
  auto nblk_of = [&](int s) -> int {
    const int* cu = by_keys ? cu_k : cu_q;
    const int len = cu[s + 1] - cu[s];
    const int n = len > 0 ? (len + rows_per_block - 1) / rows_per_block : 0;
    return n < max_nblk ? n : max_nblk;  // max_nblk bounds every sequence (checked on the host)
  };
  for (int s = tid; s < num_seqs; s += kThreads) {
    const int n = nblk_of(s);
    if (n > 0) atomicAdd(&bins[n], 1);
  }
  __syncthreads();
  // bin_start[b] = entries of all block counts above b: a scan from b = nb-1 down.
  // Each thread sums a contiguous chunk of bins; thread 0 scans the chunk sums.
  const int chunk = (nb + kThreads - 1) / kThreads;
  const int b_hi = nb - 1 - tid * chunk;  // this thread's chunk, from the top
  long long acc = 0;
  for (int k = 0; k < chunk; ++k) {
    const int b = b_hi - k;
    if (b < 1) break;
    acc += static_cast<long long>(bins[b]) * b * heads;
  }
  chunk_sum[tid] = acc;
  __syncthreads();
  if (tid == 0) {
    long long run = 0;
    for (int t = 0; t < kThreads; ++t) {
      const long long v = chunk_sum[t];
      chunk_sum[t] = run;
      run += v;
    }
  }
  __syncthreads();
  acc = chunk_sum[tid];
  for (int k = 0; k < chunk; ++k) {
    const int b = b_hi - k;
    if (b < 0) break;
    bin_start[b] = acc;
    if (b >= 1) acc += static_cast<long long>(bins[b]) * b * heads;
  }
  __syncthreads();
  const long long total = bin_start[0];  // all real entries (block count 0 adds none)
  for (int b = tid; b < nb; b += kThreads) bins[b] = 0;  // now cursors
  __syncthreads();
  for (int s = tid; s < num_seqs; s += kThreads) {
    const int n = nblk_of(s);
    seq_start[s] = n > 0 ? bin_start[n] + static_cast<long long>(atomicAdd(&bins[n], 1)) * n * heads : -1;
  }
  __syncthreads();
  const int lane = tid & 31, warp = tid >> 5;
  for (int s = warp; s < num_seqs; s += kThreads / 32) {
    const long long st = seq_start[s];
    if (st < 0) continue;
    const int n = nblk_of(s);
    TileEntry e;
    e.q_start = cu_q[s];
    e.nq = cu_q[s + 1] - e.q_start;
    e.k_start = cu_k[s];
    e.nk = cu_k[s + 1] - e.k_start;
    e.seq = s;
    e.pad = 0;
    for (int i = lane; i < n * heads && st + i < bound; i += 32) {  // bound: offsets that overrun total rows
      const int h = i / n, k = i % n;
      e.head = h;
      e.blk = descending ? n - 1 - k : k;
      out[st + i] = e;
    }
  }
  for (long long i = total + tid; i < bound; i += kThreads) {
    TileEntry z{};
    z.seq = -1;
    out[i] = z;
  }
}

}  // namespace sched

cudaError_t launch_tile_list(const int* cu_q, const int* cu_k, int num_seqs, int heads, int rows_per_block,
                             bool by_keys, bool descending, int max_nblk, TileEntry* out, int64_t* seq_start,
                             int64_t bound, cudaStream_t stream) {
  if (max_nblk < 0 || max_nblk > kMaxListBlocks || num_seqs < 0 || rows_per_block <= 0) return cudaErrorInvalidValue;
  sched::tile_list_kernel<<<1, sched::kThreads, 0, stream>>>(cu_q, cu_k, num_seqs, heads, rows_per_block,
                                                           by_keys ? 1 : 0, descending ? 1 : 0, max_nblk, out,
                                                           seq_start, bound);
  return cudaGetLastError();
}

}  // namespace gb300
