// sv_grow.cuh -- EAGLE-2 dynamic draft-tree growth on synthetic draft rows.
//
// "EAGLE math", "EAGLE-2: dynamic draft trees": grow the tree greedily from
// the drafter's probabilities -- expand the nodes with the highest cumulative
// draft probability, prune low-probability paths, and re-rank which
// candidates to keep, with the number of verified nodes unchanged; "EAGLE-3
// speculative decoding review", "EAGLE-2: Does Every Context Need the Same
// Draft Tree?".
//
// Layer l expands the frontier (slot j: a node; layer 0: the root) with the
// draft row logits[b, l, j]: q = softmax(z / T); the node's children are its
// K most probable tokens (ties: lower token), valued parent + ln q(token);
// the next frontier is the layer's K best children (ties: creation order).
// After D layers the tree is the root plus the M best nodes (ties: creation
// order), in creation order with parents renumbered.
//
// A row's K best tokens and its normaliser depend on the row alone, not on
// which node the frontier put in its slot, so every row the growth reads is
// reduced in one streaming launch; only the node bookkeeping is sequential.
//
//   grow_topk_*kernel   per (draft row, 32 KB chunk), all rows of all trees:
//                       the chunk's softmax partial (integer reference,
//                       double-float sum) and its K largest logits (lowest
//                       index on ties), by a threshold filter and a ranking
//   grow_tree_kernel    one CTA per tree, all layers: merge each frontier
//                       row's chunk records, ln q of the K tokens (float64:
//                       a few values per row), create the children, choose
//                       the next frontier; then sort every node by (value
//                       desc, creation asc), keep M, renumber
// Ranking tokens by raw logit is ranking them by probability, so the token
// choices are exact; node values are float64.
#pragma once

#include "sv_kernels.cuh"

namespace sv {

constexpr int kGrowMaxK = 16;       // children per expanded node, frontier size
constexpr int kGrowMaxD = 16;       // layers
constexpr int kGrowMaxNodes = 1 + kGrowMaxK + (kGrowMaxD - 1) * kGrowMaxK * kGrowMaxK;  // 3857

struct GrowRec {  // one chunk of one draft row
  int ref;
  float hi, lo;
  int nk;                      // candidates stored
  float val[kGrowMaxK];        // raw logits, largest first
  int idx[kGrowMaxK];
};

struct GrowParams {
  const void* logits;  // [B, D, K, V]
  float scale;         // log2(e) / T
  int B, D, K, V, M, nchunks;
  int rows_per_tree;   // draft rows read per tree: 1 + (D - 1) K
  int items;           // B rows_per_tree nchunks
  GrowRec* rec;        // [B, rows_per_tree, nchunks]
  double* nval;        // [B, kGrowMaxNodes]
  int32_t* npar;
  int32_t* ntok;
  int32_t* ndep;
  int32_t* tokens;     // outputs [B, M+1]
  int32_t* parents;
  int32_t* depth;
  float* values;
  unsigned* flags;
};

// (value, index) order of candidates: larger value, then lower index.
__device__ __forceinline__ bool grow_better(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

// Order-preserving 64-bit key of a non-NaN double: a < b exactly when
// key(a) < key(b), with -0.0 folded onto +0.0.  Orders of node values are
// taken on these keys, in integer arithmetic, rather than by double compares.
__device__ __forceinline__ unsigned long long grow_key(double x) {
  unsigned long long u = (unsigned long long)__double_as_longlong(x);
  if (u == 0x8000000000000000ull) u = 0;  // -0.0
  return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

// Warp argmax over lanes of (v, i); returns the winner to every lane.
__device__ __forceinline__ void grow_warp_best(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (grow_better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

constexpr int kGrowCand = 512;  // candidates above the threshold kept per chunk

// outv/outi[r] = the r-th best of n (value, index) candidates, for r < K;
// ranks past n get (-inf, INT_MAX).  Every thread of the CTA takes part: a
// candidate's rank is the number of candidates better than it, which the
// strict order of grow_better makes unique.
__device__ __forceinline__ void grow_rank_select(const float* cv, const int* ci, int n, int K,
                                                 float* outv, int* outi) {
  for (int t = threadIdx.x; t < n; t += kThreads) {
    const float v = cv[t];
    const int i = ci[t];
    int rank = 0;
    for (int u = 0; u < n && rank < K; ++u) rank += grow_better(cv[u], ci[u], v, i);
    if (rank < K) {
      outv[rank] = v;
      outi[rank] = i;
    }
  }
  for (int r = n + (int)threadIdx.x; r < K; r += kThreads) {
    outv[r] = -INFINITY;
    outi[r] = 0x7FFFFFFF;
  }
}

// Draft row q of a tree: q = 0 is layer 0's slot 0; q = 1 + (l - 1) K + j is
// layer l's slot j.  Returns the row's element offset in logits [B, D, K, V].
__device__ __forceinline__ size_t grow_row_offset(const GrowParams& p, int rowi) {
  const int b = rowi / p.rows_per_tree, q = rowi - b * p.rows_per_tree;
  const int layer = q == 0 ? 0 : 1 + (q - 1) / p.K;
  const int slot = q == 0 ? 0 : (q - 1) - (layer - 1) * p.K;
  return (((size_t)b * p.D + layer) * p.K + slot) * (size_t)p.V;
}

struct GrowTopkSmem {
  float cv[kGrowCand];  // candidates >= theta
  int ci[kGrowCand];
  float wm[kWarps];     // warp maxima
  StatsSlot st[kWarps]; // warp softmax partials of the segment ending here
  int n;                // candidates found
  int seg_end;          // this item ends a row segment: st holds its partials
};

// Largest element of one 16-byte vector.
template <typename E>
__device__ __forceinline__ float grow_vec_max(const uint4& v);
template <>
__device__ __forceinline__ float grow_vec_max<F32>(const uint4& v) {
  return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
               fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
}
template <>
__device__ __forceinline__ float grow_vec_max<BF16>(const uint4& v) {
  const uint32_t w = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
  return fmaxf(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// The second step of an item's top-k (every thread, after the item's
// grow_topk_collect and before barrier A of the next one): ranks the
// buffer's candidates into the item's record and, if the item ends a row
// segment, merges the warps' softmax partials of the segment into it (other
// records carry an empty partial).  No CTA barrier.
__device__ __forceinline__ void grow_topk_finish(const GrowParams& p, int item,
                                                 const GrowTopkSmem& b) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  GrowRec* out = p.rec + item;  // item = row * nchunks + chunk
  grow_rank_select(b.cv, b.ci, b.n, p.K, out->val, out->idx);
  if (warp == kWarps - 1) {
    int R = kRefEmpty;
    FSum tot = FSum::zero();
    if (b.seg_end) {
      StatsSlot v = lane < kWarps ? b.st[lane] : StatsSlot{kRefEmpty, 0.0f, 0.0f, 0};
      R = warp_max_i(v.ref);
      FSum f;
      f.hi = v.hi;
      f.lo = v.lo;
      f.scale(pow2i_f(v.ref - R));
      tot = warp_sum_df(f);
    }
    if (lane == 0) {
      out->ref = R;
      out->hi = tot.hi;
      out->lo = tot.lo;
      out->nk = p.K;
    }
  }
}

// Top-k of one (draft row, 32 KB chunk) item in two steps, so that a CTA
// streaming several items overlaps the ranking of one with the
// exponentials of the next.  theta, the K-th largest of the 16 warp maxima,
// is reached by at least K elements, so the chunk's K largest are all
// >= theta: only vectors whose maximum reaches theta are searched for
// candidates (a few dozen elements per chunk).  The softmax partial runs on
// in each thread over a row's consecutive chunks (st) and is reduced over
// the CTA once per row segment.  Consecutive items alternate between two
// buffers.
//
// grow_topk_collect (every thread, the item's vectors in registers, past-
// the-end elements -inf): the partial, the warp maxima, theta and the
// candidates into sh[cur]; if ties at theta overflow the buffer, the 16
// warps' exact K best (K rounds each) replace the candidates.  Between the
// exponentials and the first CTA barrier it finishes the previous item
// (prev >= 0, held in sh[cur ^ 1]), then clears sh[cur ^ 1].n.  Two CTA
// barriers; sh[cur].n is 0 on entry.  seg_end is uniform over the CTA.
template <typename E>
__device__ __forceinline__ void grow_topk_collect(const GrowParams& p,
                                                  const uint4 (&raw)[kVecPerThread], int item,
                                                  bool seg_end, StatsState& st, int prev,
                                                  GrowTopkSmem* sh, int cur) {
  GrowTopkSmem& b = sh[cur];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = item % p.nchunks;
  const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
  const int K = p.K;
  float vm[kVecPerThread];
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) vm[q] = grow_vec_max<E>(raw[q]);
  const float tmax = fmaxf(fmaxf(vm[0], vm[1]), fmaxf(vm[2], vm[3]));
  stats_chunk<E>(raw, p.scale, st, tmax);
  const float wmax = warp_max_f(tmax);
  if (seg_end) {
    const int wref = warp_max_i(st.ref);
    FSum mine = st.acc;
    mine.scale(pow2i_f(st.ref - wref));
    const FSum wsum = warp_sum_df(mine);
    if (lane == 0) b.st[warp] = StatsSlot{wref, wsum.hi, wsum.lo, 0};
    st = StatsState();
  }
  if (lane == 0) b.wm[warp] = wmax;
  if (threadIdx.x == 0) b.seg_end = seg_end;
  if (prev >= 0) grow_topk_finish(p, prev, sh[cur ^ 1]);
  __syncthreads();  // A
  if (threadIdx.x == 0) sh[cur ^ 1].n = 0;
  // theta: the K-th largest warp maximum, by a bitonic sort of the 16
  // maxima over lanes 0..15 (largest first); every warp finds it on its own
  float theta;
  {
    float v = lane < kWarps ? b.wm[lane] : -INFINITY;
#pragma unroll
    for (int k = 2; k <= kWarps; k <<= 1)
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, j);
        v = (((lane & j) == 0) == ((lane & k) == 0)) ? fmaxf(v, o) : fminf(v, o);
      }
    theta = __shfl_sync(0xffffffffu, v, K - 1);
  }
  if (tmax >= theta) {
#pragma unroll
    for (int q = 0; q < kVecPerThread; ++q) {
      if (vm[q] < theta) continue;
#pragma unroll
      for (int e = 0; e < E::kEPV; ++e) {
        const float z = E::elem(raw[q], e);
        const int j = j0 + (q * kThreads + (int)threadIdx.x) * E::kEPV + e;
        if (z >= theta && j < j1) {
          const int at = atomicAdd(&b.n, 1);
          if (at < kGrowCand) {
            b.cv[at] = z;
            b.ci[at] = j;
          }
        }
      }
    }
  }
  __syncthreads();  // C
  if (b.n > kGrowCand) {  // uniform: every thread reads the same count
    __syncthreads();
    uint32_t used = 0;
    for (int r = 0; r < K; ++r) {
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF, bslot = -1;
#pragma unroll
      for (int q = 0; q < kVecPerThread; ++q)
#pragma unroll
        for (int e = 0; e < E::kEPV; ++e) {
          const int k = q * E::kEPV + e;
          const int j = j0 + (q * kThreads + (int)threadIdx.x) * E::kEPV + e;
          const float z = E::elem(raw[q], e);
          if (!(used >> k & 1u) && j < j1 && grow_better(z, j, bv, bi)) {
            bv = z;
            bi = j;
            bslot = k;
          }
        }
      float wv = bv;
      int wi = bi;
      grow_warp_best(wv, wi);
      if (bslot >= 0 && wi == bi) used |= 1u << bslot;
      if (lane == 0) {
        b.cv[warp * K + r] = wv;
        b.ci[warp * K + r] = wi;
      }
    }
    if (threadIdx.x == 0) b.n = kWarps * K;
    __syncthreads();
  }
}

// One CTA per item, plain loads (any row size and alignment).
template <typename E, bool kVec>
__global__ void __launch_bounds__(kThreads, 2) grow_topk_kernel(const GrowParams p) {
  using St = typename E::storage;
  __shared__ GrowTopkSmem sh[2];
  asm volatile("griddepcontrol.launch_dependents;");
  const int item = blockIdx.x;
  const int rowi = item / p.nchunks, c = item - rowi * p.nchunks;
  const St* row = reinterpret_cast<const St*>(p.logits) + grow_row_offset(p, rowi);
  const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
  uint4 raw[kVecPerThread];
  load_chunk_regs<E, kVec>(row, j0, j1, raw);  // past-the-end elements are -inf
  if (threadIdx.x == 0) sh[0].n = 0;
  StatsState st;
  grow_topk_collect<E>(p, raw, item, true, st, -1, sh, 0);
  grow_topk_finish(p, item, sh[0]);
}

// Persistent CTAs over contiguous item ranges, the chunks streamed through
// the bulk-copy ring of the verification kernels (rows of whole 16-byte
// vectors), so the copies of the next items overlap this item's ranking.
template <typename E>
__global__ void __launch_bounds__(kThreads, 2) grow_topk_stream_kernel(const GrowParams p) {
  extern __shared__ __align__(128) uint8_t stage_mem[];
  __shared__ Ring ring;
  __shared__ GrowTopkSmem sh[2];
  using St = typename E::storage;
  int i0, i1;
  item_range(p.items, i0, i1);
  // the tree kernel may begin launching; it waits for this grid
  asm volatile("griddepcontrol.launch_dependents;");
  if (i0 >= i1) return;
  const int C = p.nchunks;
  auto issue = [&](int item, int slot) {
    const int rowi = item / C, c = item - (item / C) * C;
    const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
    const unsigned bytes = (unsigned)(j1 - j0) * (unsigned)sizeof(St);
    mbar_expect_tx(&ring.full[slot], bytes);
    bulk_g2s(stage_mem + (size_t)slot * kChunkBytes,
             reinterpret_cast<const St*>(p.logits) + grow_row_offset(p, rowi) + j0, bytes,
             &ring.full[slot]);
  };
  if (threadIdx.x == 0) sh[0].n = 0;  // ring_init ends with a CTA barrier
  int issued = ring_init(ring, i0, i1, issue);
  int slot = 0;
  unsigned par = 0;
  StatsState st;  // this thread's partial over the current row segment
  for (int it = i0; it < i1; ++it) {
    const int c = it % C;
    const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
    uint4 raw[kVecPerThread];
    ring_take<E>(ring, stage_mem, slot, par, (j1 - j0) / E::kEPV, p.flags, raw);
    if (threadIdx.x == 0)
      issued = ring_refill(ring, slot, par, it + kStages, i1, issued, p.flags, issue);
    // an aborted CTA ranks -inf: its flag is set
    grow_topk_collect<E>(p, raw, it, c + 1 == C || it + 1 == i1, st, it > i0 ? it - 1 : -1, sh,
                         (it - i0) & 1);
    if (++slot == kStages) {
      slot = 0;
      par ^= 1u;
    }
  }
  grow_topk_finish(p, i1 - 1, sh[(i1 - 1 - i0) & 1]);
  if (threadIdx.x == 0) ring_drain(ring, i0, issued);
}

constexpr int kGrowMaxCand = 2048;            // chunks x K per row, checked on the host
constexpr size_t kGrowStageBudget = 128 << 10;  // staged chunk lists of the rows in flight
constexpr int kGrowMaxRows = 1 + (kGrowMaxD - 1) * kGrowMaxK;  // draft rows per tree

// Shared-memory plan of grow_tree_kernel (host and device).  Per-row results
// of the tree (ln q of the K best tokens, the tokens, the logits, the row
// normaliser and its log2) stay for the whole layer loop; behind them
// `nstage` warps stage one row's chunk lists each (values, tokens, head
// pointers).  The node sort reuses the whole space afterwards.
__host__ __device__ inline size_t grow_row_bytes(int rows, int K) {
  const size_t b = (size_t)rows * K * (sizeof(double) + sizeof(float) + sizeof(int)) +
                   (size_t)rows * (sizeof(double) + sizeof(int) + 2 * sizeof(float));
  return (b + 15) & ~(size_t)15;
}
__host__ __device__ inline size_t grow_stage_bytes(int nchunks, int K) {
  // candidates (value, token), then per chunk: head pointer, reference, sum
  // (hi, lo); then 32 gathered candidates (value, token)
  return (size_t)nchunks * K * (sizeof(float) + sizeof(int)) +
         (size_t)nchunks * (2 * sizeof(int) + 2 * sizeof(float)) + 32 * (sizeof(float) + sizeof(int));
}

__device__ __forceinline__ void grow_cp4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__host__ __device__ inline int grow_nstage(int nchunks, int K) {
  const size_t fit = kGrowStageBudget / grow_stage_bytes(nchunks, K);
  return (int)(fit < (size_t)kWarps ? fit : (size_t)kWarps);
}
__host__ __device__ inline int grow_sort_n(int nnodes) {
  int P = 1;
  while (P < nnodes - 1) P <<= 1;
  return P;
}
__host__ __device__ inline size_t grow_tree_smem(int nchunks, int K, int rows, int nnodes) {
  const size_t work = grow_row_bytes(rows, K) +
                      (size_t)grow_nstage(nchunks, K) * grow_stage_bytes(nchunks, K);
  const size_t sort = (size_t)grow_sort_n(nnodes) * (sizeof(unsigned long long) + sizeof(int)) +
                      (size_t)nnodes * sizeof(int);
  return work > sort ? work : sort;
}
constexpr size_t kGrowTreeSmem =
    ((size_t)kGrowMaxRows * kGrowMaxK * 16 + (size_t)kGrowMaxRows * 20 + 15) / 16 * 16 +
    kGrowStageBudget;

// One CTA per tree.  A draft row's K best tokens and their ln q do not
// depend on which node the frontier put in the row's slot, so every row of
// the tree is reduced first, nstage rows at a time: the CTA stages the rows'
// chunk records in shared memory, then warp w takes row q0 + w, merges the
// chunk normalisers and picks the K best tokens from the chunk lists (each
// sorted best first) by a threshold and a shuffle ranking; then
// a thread per row takes log2 of the row sum and a thread per (row, rank)
// its ln q = (z s - R - log2 S) ln 2, in float64.  The layers are then one
// warp's work: a child's value is its parent's plus the row's ln q, and the
// next frontier is the K children ranked best among the layer's children.
// Finally every non-root node is sorted by (value desc, creation asc), the
// first M are kept and renumbered in creation order.  Launched
// programmatically after the top-k grid and waits for it before reading the
// records.
__global__ void __launch_bounds__(kThreads) grow_tree_kernel(const GrowParams p) {
  extern __shared__ __align__(16) uint8_t grow_mem[];
  constexpr int kMaxKids = kGrowMaxK * kGrowMaxK;
  __shared__ double s_dval[kMaxKids];             // the layer's children: value
  __shared__ unsigned long long s_val[kMaxKids];  // ... its order key
  __shared__ int s_front[kGrowMaxK];              // frontier: node id
  __shared__ double s_fval[kGrowMaxK];            // ... and value
  __shared__ int s_wtot[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.x;
  const int K = p.K;
  const int rows = p.rows_per_tree;
  const int ncand = p.nchunks * K;
  const int nstage = grow_nstage(p.nchunks, K);
  const int nnodes = 1 + K + (p.D - 1) * K * K;
  double* nval = p.nval + (size_t)b * kGrowMaxNodes;
  int32_t* npar = p.npar + (size_t)b * kGrowMaxNodes;
  int32_t* ntok = p.ntok + (size_t)b * kGrowMaxNodes;
  int32_t* ndep = p.ndep + (size_t)b * kGrowMaxNodes;
  // per-row results: [rows K] ln q, logit, token; [rows] log2 S, R, S
  double* r_lnq = reinterpret_cast<double*>(grow_mem);
  double* r_l2 = r_lnq + (size_t)rows * K;
  float* r_z = reinterpret_cast<float*>(r_l2 + rows);
  int* r_tok = reinterpret_cast<int*>(r_z + (size_t)rows * K);
  int* r_R = r_tok + (size_t)rows * K;
  float* r_hi = reinterpret_cast<float*>(r_R + rows);
  float* r_lo = r_hi + rows;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the top-k records

  // 1. every row of the tree: normaliser and K best tokens (float
  //    arithmetic), nstage rows at a time: the CTA stages the rows' chunk
  //    records together, then warp w reduces row q0 + w
  {
    const size_t sb = grow_stage_bytes(p.nchunks, K);
    uint8_t* stage0 = grow_mem + grow_row_bytes(rows, K);
    for (int q0 = 0; q0 < rows; q0 += nstage) {
      const int nb = min(nstage, rows - q0);
      const GrowRec* rec0 = p.rec + ((size_t)b * rows + q0) * p.nchunks;
      // asynchronous 4-byte copies: every load of the batch is in flight at once
      for (int i = threadIdx.x; i < nb * ncand; i += kThreads) {
        const int w = i / ncand, k = i - w * ncand;
        const int c = k / K, r = k - c * K;
        const GrowRec& g = rec0[(size_t)w * p.nchunks + c];
        float* cv = reinterpret_cast<float*>(stage0 + (size_t)w * sb);
        grow_cp4(cv + k, &g.val[r]);
        grow_cp4(reinterpret_cast<int*>(cv + ncand) + k, &g.idx[r]);
      }
      for (int i = threadIdx.x; i < nb * p.nchunks; i += kThreads) {
        const int w = i / p.nchunks, c = i - w * p.nchunks;
        const GrowRec& g = rec0[i];
        int* hp = reinterpret_cast<int*>(stage0 + (size_t)w * sb) + 2 * (size_t)ncand;
        hp[c] = 0;
        grow_cp4(hp + p.nchunks + c, &g.ref);
        grow_cp4(hp + 2 * p.nchunks + c, &g.hi);
        grow_cp4(hp + 3 * p.nchunks + c, &g.lo);
      }
      asm volatile("cp.async.commit_group;\ncp.async.wait_all;" ::: "memory");
      __syncthreads();
      if (warp < nb) {
        const int q = q0 + warp;
        float* cv = reinterpret_cast<float*>(stage0 + (size_t)warp * sb);
        const int* ci = reinterpret_cast<const int*>(cv + ncand);
        int* hp = const_cast<int*>(ci) + ncand;  // list c's head; list c belongs to lane c mod 32
        const int* cref = hp + p.nchunks;
        const float* chi = reinterpret_cast<const float*>(cref + p.nchunks);
        const float* clo = chi + p.nchunks;
        // normaliser: (reference, double-float sum) over the chunks
        int lref = kRefEmpty;
        FSum acc = FSum::zero();
        for (int c = lane; c < p.nchunks; c += 32) {
          const int gref = cref[c];
          if (gref > lref) {
            acc.scale(pow2i_f(lref - gref));
            lref = gref;
          }
          FSum v;
          v.hi = chi[c];
          v.lo = clo[c];
          v.scale(pow2i_f(gref - lref));
          acc = df_add(acc, v);
        }
        const int R = warp_max_i(lref);
        acc.scale(pow2i_f(lref - R));
        const FSum S = df_norm(warp_sum_df(acc));
        if (lane == 0) {
          r_R[q] = R;
          r_hi[q] = S.hi;
          r_lo[q] = S.lo;
        }
        // K best over the chunk lists (each sorted best first; placeholders
        // of short chunks, index >= V, end a list).  A lane samples entry h
        // of list c (the first m = 32 / nchunks entries of every list);
        // theta = the K-th best sample: at least K entries reach it, so the
        // K best are among the entries >= theta, a prefix of each list; when
        // they fit in the 32 lanes, a lane each, they are ranked against one
        // another (broadcast shared-memory reads)
        int total = 0;  // 0: not done here
        float* gv = const_cast<float*>(clo) + p.nchunks;
        int* gx = reinterpret_cast<int*>(gv + 32);
        if (p.nchunks <= 32) {
          const int m = min(K, 32 / p.nchunks);
          const int sc = lane / m, sh = lane - sc * m;
          float hv = -INFINITY;
          int hx = 0x7FFFFFFF;
          if (sc < p.nchunks && ci[sc * K + sh] < p.V) {
            hv = cv[sc * K + sh];
            hx = ci[sc * K + sh];
          }
          gv[lane] = hv;
          gx[lane] = hx;
          __syncwarp();
          int hr = 0;
#pragma unroll 8
          for (int u = 0; u < 32; ++u) hr += grow_better(gv[u], gx[u], hv, hx) ? 1 : 0;
          const unsigned sel = __ballot_sync(0xffffffffu, hx != 0x7FFFFFFF && hr == K - 1);
          const float theta = sel ? __shfl_sync(0xffffffffu, hv, __ffs(sel) - 1) : -INFINITY;
          int cnt = 0;
          if (lane < p.nchunks)
            for (int h = 0; h < K; ++h)
              cnt += (ci[lane * K + h] < p.V && cv[lane * K + h] >= theta) ? 1 : 0;
          int incl = cnt;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          const int all = __shfl_sync(0xffffffffu, incl, 31);
          __syncwarp();  // the samples are read before the candidates replace them
          if (all <= 32) {
            total = all;
            for (int h = 0; h < cnt; ++h) {
              gv[incl - cnt + h] = cv[lane * K + h];
              gx[incl - cnt + h] = ci[lane * K + h];
            }
            __syncwarp();
            const float v = lane < total ? gv[lane] : -INFINITY;
            const int x = lane < total ? gx[lane] : 0x7FFFFFFF;
            int rank = 0;
            for (int u = 0; u < total; ++u) rank += grow_better(gv[u], gx[u], v, x) ? 1 : 0;
            if (lane < total && rank < K) {
              r_z[q * K + rank] = v;
              r_tok[q * K + rank] = x;
            }
          }
        }
        if (total == 0) {  // too many candidates: K rounds of a head merge
          // K rounds: the best head over the lists; placeholders of short
          // chunks (index >= V) end a list
          for (int r = 0; r < K; ++r) {
            float bv = -INFINITY;
            int bi = 0x7FFFFFFF, bc = -1;
            for (int c = lane; c < p.nchunks; c += 32) {
              const int h = hp[c];
              if (h < K) {
                const float v = cv[c * K + h];
                const int ix = ci[c * K + h];
                if (ix < p.V && grow_better(v, ix, bv, bi)) {
                  bv = v;
                  bi = ix;
                  bc = c;
                }
              }
            }
            float wv = bv;
            int wi = bi;
            grow_warp_best(wv, wi);
            if (bc >= 0 && wi == bi) {  // token indices are unique: one winner
              ++hp[bc];
              r_z[q * K + r] = wv;
              r_tok[q * K + r] = wi;
            }
          }
        }
      }
      __syncthreads();  // the staging area is reused by the next rows
    }
  }
  // 2. float64, a thread per row, then a thread per (row, rank)
  for (int q = threadIdx.x; q < rows; q += kThreads)
    r_l2[q] = log2((double)r_hi[q] + (double)r_lo[q]);
  __syncthreads();
  for (int t = threadIdx.x; t < rows * K; t += kThreads) {
    const int q = t / K;
    r_lnq[t] = ((double)r_z[t] * (double)p.scale - (double)r_R[q] - r_l2[q]) * 0.6931471805599453;
  }
  __syncthreads();

  // 3. the layers, one warp: children values, then the next frontier by K
  //    rounds of a head merge over the slots' child lists
  if (warp == 0) {
    if (lane == 0) {  // the root
      nval[0] = 0.0;
      npar[0] = -1;
      ntok[0] = -1;
      ndep[0] = 0;
      s_front[0] = 0;
      s_fval[0] = 0.0;
    }
    __syncwarp();
    for (int layer = 0; layer < p.D; ++layer) {
      const int nfront = layer == 0 ? 1 : K;
      const int base = layer == 0 ? 1 : 1 + K + (layer - 1) * K * K;
      const int q0 = layer == 0 ? 0 : 1 + (layer - 1) * K;  // the layer's first row
      const int nc = nfront * K;
      for (int t = lane; t < nc; t += 32) {
        const int slot = t / K;
        const double val = s_fval[slot] + r_lnq[(size_t)q0 * K + t];
        const int id = base + t;
        nval[id] = val;
        npar[id] = s_front[slot];
        ntok[id] = r_tok[(size_t)q0 * K + t];
        ndep[id] = layer + 1;
        s_dval[t] = val;
        s_val[t] = grow_key(val);
      }
      __syncwarp();
      if (layer + 1 < p.D) {
        // a child's rank = the children before it (independent loads)
        for (int t = lane; t < nc; t += 32) {
          const unsigned long long v = s_val[t];
          int rank = 0;
#pragma unroll 8
          for (int u = 0; u < nc; ++u) {
            const unsigned long long o = s_val[u];
            rank += (o > v || (o == v && u < t)) ? 1 : 0;
          }
          if (rank < K) {
            s_front[rank] = base + t;
            s_fval[rank] = s_dval[t];
          }
        }
        __syncwarp();
      }
    }
  }
  __syncthreads();

  // keep the M best non-root nodes: bitonic sort of (value key desc, id asc)
  const int n = nnodes - 1;  // non-root nodes, ids 1..nnodes-1
  const int P = grow_sort_n(nnodes);
  unsigned long long* s_key = reinterpret_cast<unsigned long long*>(grow_mem);  // [P]
  int* s_id = reinterpret_cast<int*>(s_key + P);                                // [P]
  int* s_new = s_id + P;                                                        // [nnodes]
  for (int i = threadIdx.x; i < P; i += kThreads) {
    s_key[i] = grow_key(i < n ? nval[i + 1] : -INFINITY);
    s_id[i] = i < n ? i + 1 : 0x7FFFFFFF;
  }
  for (int i = threadIdx.x; i < nnodes; i += kThreads) s_new[i] = 0;
  __syncthreads();
  if (P <= kThreads) {
    // one element per thread, in registers: partners closer than 32 are in
    // the same warp (shuffles), farther ones are exchanged through shared
    // memory.  "Before" = larger key, then smaller id; after the sort the
    // thread i < M holds the i-th best.
    const int i = threadIdx.x;
    unsigned long long key = i < P ? s_key[i] : 0ull;
    int id = i < P ? s_id[i] : 0x7FFFFFFF;
    for (int k = 2; k <= P; k <<= 1)
      for (int j = k >> 1; j > 0; j >>= 1) {
        unsigned long long okey;
        int oid;
        if (j < 32) {
          okey = __shfl_xor_sync(0xffffffffu, key, j);
          oid = __shfl_xor_sync(0xffffffffu, id, j);
        } else {
          __syncthreads();  // every read of the previous exchange is done
          if (i < P) {
            s_key[i] = key;
            s_id[i] = id;
          }
          __syncthreads();
          okey = i < P ? s_key[i ^ j] : 0ull;
          oid = i < P ? s_id[i ^ j] : 0x7FFFFFFF;
        }
        if (i < P) {
          const bool other_before = okey > key || (okey == key && oid < id);
          const bool keep_before = (i < (i ^ j)) == ((i & k) == 0);
          if (other_before == keep_before) {
            key = okey;
            id = oid;
          }
        }
      }
    __syncthreads();
    if (i < p.M) s_new[id] = 1;
  } else {
    // several elements per thread: the same network through shared memory
    for (int k = 2; k <= P; k <<= 1)
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int i = threadIdx.x; i < P; i += kThreads) {
          const int l = i ^ j;
          if (l > i) {
            const bool up = (i & k) == 0;
            const bool lbefore = s_key[l] > s_key[i] || (s_key[l] == s_key[i] && s_id[l] < s_id[i]);
            if (lbefore == up) {
              const unsigned long long tk = s_key[i];
              s_key[i] = s_key[l];
              s_key[l] = tk;
              const int ti = s_id[i];
              s_id[i] = s_id[l];
              s_id[l] = ti;
            }
          }
        }
        __syncthreads();
      }
    for (int i = threadIdx.x; i < p.M; i += kThreads) s_new[s_id[i]] = 1;
  }
  __syncthreads();
  {
    // renumber in creation order (parents come first): thread t owns the
    // contiguous ids [t per, (t + 1) per) of 1..nnodes-1; an exclusive scan
    // of the kept counts gives each range's first new id
    const int per = (n + kThreads - 1) / kThreads;
    const int v0 = 1 + (int)threadIdx.x * per, v1 = min(nnodes, v0 + per);
    int cnt = 0;
    for (int v = v0; v < v1; ++v) cnt += s_new[v];
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_wtot[warp] = incl;
    __syncthreads();
    int id = 1 + incl - cnt;
    for (int w = 0; w < warp; ++w) id += s_wtot[w];
    for (int v = v0; v < v1; ++v) s_new[v] = s_new[v] ? id++ : -1;
  }
  __syncthreads();
  const size_t ob = (size_t)b * (p.M + 1);
  if (threadIdx.x == 0) {
    p.tokens[ob] = -1;
    p.parents[ob] = -1;
    p.depth[ob] = 0;
    p.values[ob] = 0.0f;
  }
  for (int v = 1 + threadIdx.x; v < nnodes; v += kThreads) {
    const int o = s_new[v];
    if (o < 1) continue;
    const int par = npar[v];
    const int po = par == 0 ? 0 : s_new[par];
    if (po < 0) set_flag(p.flags, kFlagBadParent);  // cannot happen (closure)
    p.tokens[ob + o] = ntok[v];
    p.parents[ob + o] = po;
    p.depth[ob + o] = ndep[v];
    p.values[ob + o] = (float)nval[v];
  }
}

}  // namespace sv
