// Host-only check of the tree-growth kernel's launch plan, built by
// tests/test_launch_plans.py with nvcc (no GPU needed): for every shape the
// interface admits (D <= 16 layers, K <= 16, chunks x K <= kGrowMaxCand), the
// staging depth is at least one row and the shared-memory plan fits the size
// the kernel opts into.
#include <cstdio>

#include "sv_grow.cuh"

int main() {
  int bad = 0, shapes = 0;
  for (int K = 1; K <= sv::kGrowMaxK; ++K)
    for (int C = 1; C * K <= sv::kGrowMaxCand; ++C)
      for (int D = 1; D <= sv::kGrowMaxD; ++D) {
        const int rows = 1 + (D - 1) * K;
        const int nnodes = 1 + K + (D - 1) * K * K;
        const int nstage = sv::grow_nstage(C, K);
        const size_t smem = sv::grow_tree_smem(C, K, rows, nnodes);
        ++shapes;
        if (nstage < 1 || smem > sv::kGrowTreeSmem || rows > sv::kGrowMaxRows ||
            nnodes > sv::kGrowMaxNodes) {
          std::printf("bad plan: K=%d chunks=%d D=%d nstage=%d smem=%zu (limit %zu)\n", K, C, D,
                      nstage, smem, sv::kGrowTreeSmem);
          bad = 1;
        }
      }
  std::printf("%d shapes checked\n", shapes);
  return bad;
}
