// sv_tree.cuh -- kernels for the draft tree around verification.
//
// Tree attention mask ("EAGLE-3 speculative decoding review", sections
// "EAGLE-2: Does Every Context Need the Same Draft Tree?" and "Must the
// Feature Be Predicted Exactly?": every tree node sees the shared prefix and
// only its own ancestors, never another branch; "The Complete EAGLE-3
// Inference Process" step 3).  The prefix part of the mask is all-visible and
// is not materialised; the kernel writes the tree block: for node v of tree b,
// a row of W = ceil(N/32) 32-bit words whose bit u % 32 of word u / 32 is set
// iff u = v or u is an ancestor of v, plus depth(v).
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr int kMaskThreads = 256;

// One thread per (tree, node, word).  The thread walks v's ancestor chain
// (parents strictly decrease, so at most v hops) and keeps the bits that fall
// in its word; a thread for word w > 0 stops once the chain drops below
// 32 w, since no later ancestor can land in its word.  The word-0 thread
// walks to the root and writes the depth (-1 and kFlagBadParent when the
// chain meets a parent outside [0, child)).
__global__ void __launch_bounds__(kMaskThreads) tree_mask_kernel(const int32_t* __restrict__ parents,
                                                                 int B, int N, int W,
                                                                 uint32_t* __restrict__ mask,
                                                                 int32_t* __restrict__ depth,
                                                                 unsigned* flags) {
  const long long t = (long long)blockIdx.x * kMaskThreads + threadIdx.x;
  const long long per_tree = (long long)N * W;
  if (t >= per_tree * B) return;
  const int b = (int)(t / per_tree);
  const int rem = (int)(t - (long long)b * per_tree);
  const int v = rem / W, w = rem - (rem / W) * W;
  const int32_t* par = parents + (size_t)b * N;
  const int lo = 32 * w;
  uint32_t word = 0;
  int cur = v, d = 0;
  bool bad = false;
  if (cur >= lo && cur < lo + 32) word |= 1u << (cur - lo);
  while (cur != 0) {
    if (w > 0 && cur < lo) break;
    const int p = __ldg(par + cur);
    if (p < 0 || p >= cur) {
      bad = true;
      break;
    }
    cur = p;
    if (cur >= lo && cur < lo + 32) word |= 1u << (cur - lo);
    ++d;
  }
  mask[t] = word;
  if (w == 0) {
    if (depth) depth[(size_t)b * N + v] = bad ? -1 : d;
    if (bad) set_flag(flags, kFlagBadParent);
  }
}

}  // namespace sv
