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
//
// KV commit of the accepted path (same page, "The Complete EAGLE-3 Inference
// Process" step 5: keep only the accepted path's cache entries and resume
// from the committed prefix).  Tree node v >= 1 holds its entries at cache
// position base + v - 1; the path 0, v_1, ..., v_d moves node v_i's entry to
// position base + i - 1 in every plane (layer, K or V), in place.
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
  // a programmatic dependent of the kernel before it in the stream: nothing
  // is read or written before that grid has finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
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

struct KvCommitParams {
  uint8_t* cache;
  long long plane_stride, seq_stride;  // bytes
  int entry_bytes, L, N, max_depth, planes;
  const int32_t* base_len;
  const int32_t* accepted_len;
  const int32_t* path_nodes;  // [B, max_depth + 1]
  int32_t* new_len;
  unsigned* flags;
  int slice_bytes;  // bytes of each moved entry staged per pass (multiple of 16)
};


constexpr int kKvMaxMoves = 64;  // path nodes staged per pass
constexpr int kKvThreads = 128;

// One CTA per (sequence, plane).  Thread 0 validates the path and lists the
// moves (entries already in place, v_i == i, are skipped).  For every column
// slice of the entries, all threads stage every moved entry in shared memory
// with 16-byte asynchronous copies, wait for all of them, and only then store
// them to their new positions, so an entry that is both moved and overwritten
// is read first.
__global__ void __launch_bounds__(kKvThreads) kv_commit_kernel(const KvCommitParams p) {
  extern __shared__ __align__(128) uint8_t kv_stage[];
  __shared__ int s_src[kKvMaxMoves], s_dst[kKvMaxMoves];
  __shared__ int s_ok, s_m;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // as in tree_mask_kernel
  asm volatile("griddepcontrol.launch_dependents;");
  const int b = blockIdx.x, plane = blockIdx.y;
  const int base = p.base_len[b], d = p.accepted_len[b];
  const int32_t* path = p.path_nodes + (size_t)b * (p.max_depth + 1);
  if (threadIdx.x == 0) {
    bool ok = base >= 1 && (long long)base + p.N - 1 <= p.L && d >= 0 && d <= p.max_depth &&
              path[0] == 0;
    for (int i = 1; ok && i <= d; ++i)
      if (path[i] < 1 || path[i] >= p.N) ok = false;
    if (plane == 0) {
      p.new_len[b] = ok ? base + d : base;
      if (!ok) set_flag(p.flags, kFlagBadPath);
    }
    s_ok = ok;
  }
  __syncthreads();
  if (!s_ok) return;
  uint8_t* row = p.cache + (long long)plane * p.plane_stride + (long long)b * p.seq_stride;
  for (int i0 = 1; i0 <= d; i0 += kKvMaxMoves) {
    const int i1 = min(d, i0 + kKvMaxMoves - 1);
    if (threadIdx.x == 0) {
      int m = 0;
      for (int i = i0; i <= i1; ++i)
        if (path[i] != i) {
          s_src[m] = base + path[i] - 1;
          s_dst[m] = base + i - 1;
          ++m;
        }
      s_m = m;
    }
    __syncthreads();
    const int m = s_m;
    for (int c0 = 0; m > 0 && c0 < p.entry_bytes; c0 += p.slice_bytes) {
      const int vps = min(p.slice_bytes, p.entry_bytes - c0) / 16;  // vectors per entry slice
      for (int idx = threadIdx.x; idx < m * vps; idx += kKvThreads) {
        const int j = idx / vps, e = idx - (idx / vps) * vps;
        const uint8_t* src = row + (long long)s_src[j] * p.entry_bytes + c0 + e * 16;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                         smem_addr(kv_stage + (size_t)j * p.slice_bytes + e * 16)),
                     "l"(src)
                     : "memory");
      }
      asm volatile("cp.async.commit_group;\ncp.async.wait_all;" ::: "memory");
      __syncthreads();  // every moved entry of this slice is staged
      for (int idx = threadIdx.x; idx < m * vps; idx += kKvThreads) {
        const int j = idx / vps, e = idx - (idx / vps) * vps;
        const uint4 v = lds128(kv_stage + (size_t)j * p.slice_bytes + e * 16);
        *reinterpret_cast<uint4*>(row + (long long)s_dst[j] * p.entry_bytes + c0 + e * 16) = v;
      }
      __syncthreads();  // the staging buffer is free again
    }
  }
}

}  // namespace sv
