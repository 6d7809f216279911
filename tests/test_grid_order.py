"""Host checks of the dense launches' dispatch order (grid_slot in the kernels'
internal header): every (pair, rank) is taken by exactly one CTA, a pair's
blocks keep their rank order (the deterministic single pass waits only on CTAs
started before it), one group per pair is the (unit, head)-major order, and the
group count keeps a group's K and V within 32 MB. The header is compiled
into a small host program; no GPU is used."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_attention_bf16_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <vector>
#include "kernels.h"
using namespace gb300;
int main() {
  int bad = 0;
  const int pairs_list[] = {1, 2, 3, 7, 16, 32, 64, 65, 128, 512};
  const int blk_list[] = {1, 2, 3, 8, 32, 128};
  for (int n_pairs : pairs_list)
    for (int n_blk : blk_list)
      for (int ng = 0; ng <= n_pairs + 1; ng += (ng < 12 ? 1 : n_pairs / 5 + 1)) {
        std::vector<int> seen(static_cast<size_t>(n_pairs) * n_blk, 0), last(n_pairs, -1);
        for (int x = 0; x < n_pairs * n_blk; ++x) {
          const GridSlot s = grid_slot(x, n_pairs, n_blk, ng);
          if (s.pair < 0 || s.pair >= n_pairs || s.rank < 0 || s.rank >= n_blk) { ++bad; continue; }
          seen[static_cast<size_t>(s.pair) * n_blk + s.rank]++;
          if (s.rank != last[s.pair] + 1) ++bad;  // ranks of a pair in increasing CTA order
          last[s.pair] = s.rank;
          if (ng == n_pairs || ng == 0 || ng > n_pairs)  // (unit, head)-major
            if (s.pair != x / n_blk || s.rank != x % n_blk) ++bad;
          if (ng == 1 && (s.rank != x / n_pairs || s.pair != x % n_pairs)) ++bad;  // rank-major
        }
        for (int c : seen) if (c != 1) ++bad;
      }
  // groups of at most 32 MB of streamed bytes, never more groups than pairs
  if (group_count(64, int64_t(4) << 20) != 8) ++bad;     // 8 pairs of 4 MB per group
  if (group_count(64, int64_t(5) << 20) != 11) ++bad;    // 6 per group -> 11 groups
  if (group_count(16, int64_t(64) << 20) != 16) ++bad;   // larger than the budget: one pair each
  if (group_count(512, int64_t(1) << 10) != 1) ++bad;    // everything in one group
  if (group_count(1, int64_t(1) << 30) != 1) ++bad;
  std::printf("%d\n", bad);
  return bad != 0;
}
"""


def test_grid_slot_is_a_bijection_that_keeps_rank_order(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    cuda_inc = "/usr/local/cuda/include"
    if not os.path.isfile(os.path.join(cuda_inc, "cuda_runtime.h")):
        pytest.skip("no CUDA headers")
    src = tmp_path / "grid_order.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "grid_order"
    r = subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, "-I", cuda_inc, str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "0", r.stdout + r.stderr
