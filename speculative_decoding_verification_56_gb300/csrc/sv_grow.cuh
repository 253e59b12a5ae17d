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
//   grow_tree_kernel    two CTAs per tree (a cluster), all layers: merge each frontier
//                       row's chunk records, ln q of the K tokens (float64:
//                       a few values per row), create the children, choose
//                       the next frontier; then keep the M best nodes by
//                       (value desc, creation asc) and renumber them
// Ranking tokens by raw logit is ranking them by probability, so the token
// choices are exact; node values are float64.
#pragma once

#include <cuda_bf16.h>

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

// Draft row q of a tree: q = 0 is layer 0's slot 0; q = 1 + (l - 1) K + j is
// layer l's slot j.  Returns the row's element offset in logits [B, D, K, V].
__device__ __forceinline__ size_t grow_row_offset(const GrowParams& p, int rowi) {
  const int b = rowi / p.rows_per_tree, q = rowi - b * p.rows_per_tree;
  const int layer = q == 0 ? 0 : 1 + (q - 1) / p.K;
  const int slot = q == 0 ? 0 : (q - 1) - (layer - 1) * p.K;
  return (((size_t)b * p.D + layer) * p.K + slot) * (size_t)p.V;
}

// Streaming top-k over row segments.  A CTA walks contiguous items (row,
// 32 KB chunk); a row segment is its run of items of one row.  Each warp
// keeps the candidates of its own 1024 elements per item in a small buffer
// for the whole segment, with a running threshold thr: at least K of the
// warp's elements so far are >= thr, so no element below it can be among the
// segment's K best -- in this warp or any other, so the warps publish their
// thresholds (an atomic max in shared memory) and each uses the largest.  The
// first item of a segment takes thr = the K-th largest of the 16 warp maxima
// (one CTA barrier); a full buffer is compacted to its K best, whose K-th
// value raises thr.  Elements are tested against thr eight at a time
// (packed compares) and only vectors whose maximum reaches thr are looked at.
// At a segment end each warp leaves its sorted K best and its softmax
// partial in the segment's slot; the last warp to arrive merges them into
// the record of the segment's last item, with no CTA barrier; the segment's
// other records carry an empty list and an empty partial.
constexpr int kGrowBuf = 32;  // candidates per warp buffer
// Row segments open at once in a CTA: no warp runs more than kStages items
// ahead of the slowest (the ring), and an item opens at most one segment.
constexpr int kGrowSlots = 4;
static_assert(kStages + 1 <= kGrowSlots, "segment slots cover the ring's spread");
struct GrowSegSmem {
  uint2 buf[kWarps][kGrowBuf];        // (value bits, index) of the warp's candidates
  int n[kWarps];                      // entries appended (more than kGrowBuf: overflow)
  uint2 tmp[kWarps][kGrowMaxK];       // each warp's compaction scratch
  uint2 lists[kGrowSlots][kWarps * kGrowMaxK];  // each warp's K best at a segment end
  StatsSlot st[kGrowSlots][kWarps];   // each warp's softmax partial at a segment end
  unsigned thr_key[kGrowSlots];       // largest published threshold (grow_fkey) of the segment
  int cnt[kGrowSlots];                // warps done with the segment
  float wm[kGrowSlots][kWarps];       // warp maxima of the segment's first item
};

// Order-preserving unsigned key of a non-NaN float and back, for atomicMax.
__device__ __forceinline__ unsigned grow_fkey(float f) {
  const unsigned u = __float_as_uint(f);
  return (u >> 31) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float grow_funkey(unsigned k) {
  return __uint_as_float((k >> 31) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ void grow_seg_smem_init(GrowSegSmem& sh) {
  if (threadIdx.x < kWarps) sh.n[threadIdx.x] = 0;
  if (threadIdx.x < kGrowSlots) {
    sh.thr_key[threadIdx.x] = grow_fkey(-INFINITY);
    sh.cnt[threadIdx.x] = 0;
  }
}

__device__ __forceinline__ uint2 grow_pack(float v, int i) {
  return make_uint2(__float_as_uint(v), (unsigned)i);
}
// a before (v, i): larger value, then lower index
__device__ __forceinline__ bool grow_before(uint2 a, float v, int i) {
  return grow_better(__uint_as_float(a.x), (int)a.y, v, i);
}

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

// Bit e set iff element e of the 16-byte vector is >= thr (bf16: thr is a
// bf16 value, so the packed compare is exact).
template <typename E>
__device__ __forceinline__ unsigned grow_ge_mask(const uint4& v, float thr);
template <>
__device__ __forceinline__ unsigned grow_ge_mask<F32>(const uint4& v, float thr) {
  return (__uint_as_float(v.x) >= thr ? 1u : 0u) | (__uint_as_float(v.y) >= thr ? 2u : 0u) |
         (__uint_as_float(v.z) >= thr ? 4u : 0u) | (__uint_as_float(v.w) >= thr ? 8u : 0u);
}
template <>
__device__ __forceinline__ unsigned grow_ge_mask<BF16>(const uint4& v, float thr) {
  const __nv_bfloat16 tb = __float2bfloat16_rn(thr);
  const __nv_bfloat162 t2 = __halves2bfloat162(tb, tb);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  unsigned m = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const unsigned c = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w[k]), t2);
    m |= ((c & 1u) | ((c >> 15) & 2u)) << (2 * k);
  }
  return m;
}

// Whole warp: keep the K best of the first m (<= kGrowBuf) entries of the
// warp's buffer, best first at buf[0 ..), and return how many remain
// (min(m, K)).  Entries are distinct (distinct indices), so ranks are too.
__device__ __forceinline__ int grow_warp_compact(GrowSegSmem& sh, int m, int K) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint2* buf = sh.buf[warp];
  uint2* tmp = sh.tmp[warp];
  __syncwarp();
  if (lane < m) {
    const uint2 me = buf[lane];
    const float v = __uint_as_float(me.x);
    const int x = (int)me.y;
    int rank = 0;
    for (int u = 0; u < m; ++u) rank += grow_before(buf[u], v, x) ? 1 : 0;
    if (rank < K) tmp[rank] = me;
  }
  __syncwarp();
  const int kept = min(m, K);
  if (lane < kept) buf[lane] = tmp[lane];
  __syncwarp();
  return kept;
}

// Whole warp: append this item's elements >= thr to the warp's buffer (each
// thread walks only its vectors whose maximum reaches thr; past-the-end
// elements are -inf, so the index test matters only for thr = -inf).  If
// the buffer overflows, the item's own K best are found exactly (K rounds)
// instead and merged with the earlier entries.  Compacts a buffer that is
// more than half full.  Returns the new entry count; thr may rise.
template <typename E>
__device__ __forceinline__ int grow_warp_append(GrowSegSmem& sh, const uint4 (&raw)[kVecPerThread],
                                                const float (&vm)[kVecPerThread], int j0, int j1,
                                                int K, int nb, float& thr, unsigned* thr_key) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint2* buf = sh.buf[warp];
  thr = fmaxf(thr, grow_funkey(*(volatile unsigned*)thr_key));
  const float seen = thr;  // published already, or this warp's own segment threshold
  unsigned mx = 0;  // 1 + the highest slot this lane took
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) {
    if (!(vm[q] >= thr)) continue;
    const int jb = j0 + (q * kThreads + (int)threadIdx.x) * E::kEPV;
    unsigned em = grow_ge_mask<E>(raw[q], thr);
    if (!(thr > -INFINITY)) em &= (1u << max(0, min(E::kEPV, j1 - jb))) - 1u;  // real elements
    while (em) {
      const int e = __ffs(em) - 1;
      em &= em - 1;
      const int at = atomicAdd(&sh.n[warp], 1);
      mx = (unsigned)(at + 1);
      if (at < kGrowBuf) buf[at] = grow_pack(E::elem(raw[q], e), jb + e);
    }
  }
  int n = max(nb, (int)__reduce_max_sync(0xffffffffu, mx));  // the count after this item
  if (n <= kGrowBuf / 2) return n;  // the usual case: the count is already in place
  __syncwarp();  // every lane's entries are visible
  if (n > kGrowBuf) {
    // ties at thr: drop this item's entries, keep the earlier ones' K best,
    // and add the item's exact K best (K rounds over the warp's elements)
    n = nb > K ? grow_warp_compact(sh, nb, K) : nb;
    uint32_t used = 0;
    int added = 0;
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
      if (wi == 0x7FFFFFFF) break;  // no element left (uniform)
      if (bslot >= 0 && wi == bi) used |= 1u << bslot;
      if (lane == 0) buf[n + added] = grow_pack(wv, wi);
      ++added;
    }
    n = grow_warp_compact(sh, n + added, K);  // n + added <= 2 K <= kGrowBuf
    if (n == K) thr = fmaxf(thr, __uint_as_float(buf[K - 1].x));
  } else {
    n = grow_warp_compact(sh, n, K);  // n > 16 >= K: the K best, sorted
    thr = fmaxf(thr, __uint_as_float(buf[K - 1].x));
  }
  __syncwarp();
  if (lane == 0) {
    sh.n[warp] = n;
    if (thr > seen) atomicMax(thr_key, grow_fkey(thr));  // only a raised threshold
  }
  __syncwarp();
  return n;
}

// The merge of a closed row segment (one warp, the last to close it): K
// rounds of a head merge over the 16 sorted warp lists of its slot (token
// indices are distinct across warps, so the winner's list is the one whose
// head it is; placeholders fill short lists) and the 16 softmax partials,
// into the record of the segment's last item; then the slot is freed.
__device__ __noinline__ void grow_seg_merge(const GrowParams& p, GrowSegSmem& sh, int slot,
                                            int item) {
  const int lane = threadIdx.x & 31;
  const int K = p.K;
  GrowRec* out = p.rec + item;
  const uint2* L = sh.lists[slot];
  int h = 0;
  uint2 cur = lane < kWarps ? L[lane * kGrowMaxK] : grow_pack(-INFINITY, 0x7FFFFFFF);
  for (int r = 0; r < K; ++r) {
    float v = __uint_as_float(cur.x);
    int i = (int)cur.y;
    grow_warp_best(v, i);
    if (lane == 0) {
      out->val[r] = v;
      out->idx[r] = i;
    }
    if (lane < kWarps && i != 0x7FFFFFFF && (int)cur.y == i) {
      ++h;
      cur = h < K ? L[lane * kGrowMaxK + h] : grow_pack(-INFINITY, 0x7FFFFFFF);
    }
  }
  StatsSlot v = lane < kWarps ? sh.st[slot][lane] : StatsSlot{kRefEmpty, 0.0f, 0.0f, 0};
  const int R = warp_max_i(v.ref);
  FSum f;
  f.hi = v.hi;
  f.lo = v.lo;
  f.scale(pow2i_f(v.ref - R));
  const FSum tot = warp_sum_df(f);
  __syncwarp();
  if (lane == 0) {
    out->ref = R;
    out->hi = tot.hi;
    out->lo = tot.lo;
    out->nk = K;
    sh.thr_key[slot] = grow_fkey(-INFINITY);  // the slot is free
    sh.cnt[slot] = 0;
  }
}

// One item for the whole CTA (every thread calls it with the same flags):
// the softmax partial runs on in st; the warp appends its candidates.  A
// segment's state lives in slot seg % kGrowSlots.  first: the item opens a
// segment; thr = the K-th largest of the 16 warp maxima (at least K of the
// chunk's elements reach it), after the segment's one CTA barrier.  last:
// the item closes it; each warp leaves its K best (sorted) and its partial
// in the slot, and the last warp to arrive merges them (grow_seg_merge)
// while the other warps move on; the merge is done before its warp reaches
// the next segment's barrier, and no warp runs more than kStages items
// ahead of the slowest, so kGrowSlots slots cover every segment in use.
// Otherwise one warp writes the item's empty record.
template <typename E>
__device__ __forceinline__ void grow_seg_item(const GrowParams& p,
                                              const uint4 (&raw)[kVecPerThread], int item, int c,
                                              bool first, bool last, StatsState& st, float& thr,
                                              GrowSegSmem& sh, int& seg) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slot = seg & (kGrowSlots - 1);
  const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
  const int K = p.K;
  float vm[kVecPerThread];
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) vm[q] = grow_vec_max<E>(raw[q]);
  const float tmax = fmaxf(fmaxf(vm[0], vm[1]), fmaxf(vm[2], vm[3]));
  if (first) {
    // every warp sorts the 16 warp maxima (bitonic over lanes 0..15,
    // largest first) after the barrier
    const float wmax = warp_max_f(tmax);
    if (lane == 0) sh.wm[slot][warp] = wmax;
    __syncthreads();
    float v = lane < kWarps ? sh.wm[slot][lane] : -INFINITY;
#pragma unroll
    for (int k = 2; k <= kWarps; k <<= 1)
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, j);
        v = (((lane & j) == 0) == ((lane & k) == 0)) ? fmaxf(v, o) : fminf(v, o);
      }
    thr = __shfl_sync(0xffffffffu, v, K - 1);
  }
  const int nb = sh.n[warp];  // 0 when the segment opens
  int n = grow_warp_append<E>(sh, raw, vm, j0, j1, K, nb, thr, &sh.thr_key[slot]);
  // the softmax partial after the candidates, so that the vector maxima are
  // no longer live across its arithmetic
  stats_chunk<E>(raw, p.scale, st, tmax);
  GrowRec* out = p.rec + item;  // item = row * nchunks + chunk
  if (!last) {
    if (warp == item % kWarps) {
      if (lane < K) {
        out->val[lane] = -INFINITY;
        out->idx[lane] = 0x7FFFFFFF;
      }
      if (lane == 0) {
        out->ref = kRefEmpty;
        out->hi = 0.0f;
        out->lo = 0.0f;
        out->nk = K;
      }
    }
    return;
  }
  // segment end: this warp's K best, best first (placeholders fill a short
  // list), and its softmax partial, into the slot
  n = grow_warp_compact(sh, n, K);
  uint2* lw = sh.lists[slot] + warp * kGrowMaxK;
  for (int r = lane; r < K; r += 32) lw[r] = r < n ? sh.buf[warp][r] : grow_pack(-INFINITY, 0x7FFFFFFF);
  {
    const int wref = warp_max_i(st.ref);
    FSum mine = st.acc;
    mine.scale(pow2i_f(st.ref - wref));
    const FSum wsum = warp_sum_df(mine);
    if (lane == 0) sh.st[slot][warp] = StatsSlot{wref, wsum.hi, wsum.lo, 0};
    st = StatsState();
  }
  ++seg;
  __syncwarp();  // the warp's list and partial are written; its buffer is free
  int lastw = 0;
  if (lane == 0) {
    sh.n[warp] = 0;
    __threadfence_block();
    lastw = atomicAdd(&sh.cnt[slot], 1) == kWarps - 1;
    if (lastw) __threadfence_block();
  }
  if (__shfl_sync(0xffffffffu, lastw, 0)) grow_seg_merge(p, sh, slot, item);
}

// One CTA per item, plain loads (any row size and alignment).
template <typename E, bool kVec>
__global__ void __launch_bounds__(kThreads, 2) grow_topk_kernel(const GrowParams p) {
  using St = typename E::storage;
  __shared__ GrowSegSmem sh;
  // a programmatic dependent of the kernel before it in the stream: nothing
  // is read or written before that grid has finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int item = blockIdx.x;
  const int rowi = item / p.nchunks, c = item - rowi * p.nchunks;
  const St* row = reinterpret_cast<const St*>(p.logits) + grow_row_offset(p, rowi);
  const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
  uint4 raw[kVecPerThread];
  load_chunk_regs<E, kVec>(row, j0, j1, raw);  // past-the-end elements are -inf
  grow_seg_smem_init(sh);
  __syncthreads();
  StatsState st;
  float thr = -INFINITY;
  int seg = 0;
  grow_seg_item<E>(p, raw, item, c, true, true, st, thr, sh, seg);
}

// Persistent CTAs over contiguous item ranges, the chunks streamed through
// the bulk-copy ring of the verification kernels (rows of whole 16-byte
// vectors).  Within a row segment the loop has no CTA barrier.
template <typename E>
__global__ void __launch_bounds__(kThreads, 2) grow_topk_stream_kernel(const GrowParams p) {
  extern __shared__ __align__(128) uint8_t stage_mem[];
  __shared__ Ring ring;
  __shared__ GrowSegSmem sh;
  using St = typename E::storage;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // as in grow_topk_kernel
  int i0, i1;
  item_range(p.items, i0, i1);
  // the tree kernel may begin launching; it waits for this grid
  asm volatile("griddepcontrol.launch_dependents;");
  if (i0 >= i1) return;
  const int C = p.nchunks;
  int nrow = i0 / C, nc = i0 % C;  // the next item thread 0 issues (in order)
  auto issue = [&](int /*item: the next in order*/, int slot) {
    const int rowi = nrow, c = nc;
    if (++nc == C) {
      nc = 0;
      ++nrow;
    }
    const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
    const unsigned bytes = (unsigned)(j1 - j0) * (unsigned)sizeof(St);
    mbar_expect_tx(&ring.full[slot], bytes);
    bulk_g2s(stage_mem + (size_t)slot * kChunkBytes,
             reinterpret_cast<const St*>(p.logits) + grow_row_offset(p, rowi) + j0, bytes,
             &ring.full[slot]);
  };
  grow_seg_smem_init(sh);  // ring_init ends with a CTA barrier
  int issued = ring_init(ring, i0, i1, issue);
  int slot = 0;
  unsigned par = 0;
  StatsState st;  // this thread's partial over the current row segment
  float thr = -INFINITY;
  int seg = 0;  // row segments this CTA has closed
  int c = i0 % C;  // the item's chunk, counted along (no division per item)
  for (int it = i0; it < i1; ++it) {
    const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
    uint4 raw[kVecPerThread];
    ring_take<E>(ring, stage_mem, slot, par, (j1 - j0) / E::kEPV, p.flags, raw);
    // an aborted CTA ranks -inf: its flag is set
    grow_seg_item<E>(p, raw, it, c, it == i0 || c == 0, c + 1 == C || it + 1 == i1, st, thr,
                     sh, seg);
    // the refill after the item's work, when the other warps have usually
    // released the slot (before it, warp 0 waits for them: 0.7 us slower)
    if (threadIdx.x == 0)
      issued = ring_refill(ring, slot, par, it + kStages, i1, issued, p.flags, issue);
    if (++c == C) c = 0;
    if (++slot == kStages) {
      slot = 0;
      par ^= 1u;
    }
  }
  if (threadIdx.x == 0) ring_drain(ring, i0, issued);
}

constexpr int kGrowMaxCand = 2048;            // chunks x K per row, checked on the host
constexpr size_t kGrowStageBudget = 128 << 10;  // staged chunk lists of the rows in flight
constexpr int kGrowMaxRows = 1 + (kGrowMaxD - 1) * kGrowMaxK;  // draft rows per tree

// Shared-memory plan of grow_tree_kernel (host and device).  Per-row results
// of the tree (ln q of the K best tokens, the tokens, the logits, the row
// normaliser and its log2) stay for the whole layer loop; behind them
// `nstage` warps stage one row's chunk lists each (values, tokens, head
// pointers).  The selection of the M best nodes reuses that area afterwards.
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
// The tree kernel's block: 32 warps, so a tree's 41 draft rows (6 layers of
// 8) are staged and merged in two batches.
constexpr int kGrowTreeThreads = 1024;
constexpr int kGrowTreeWarps = kGrowTreeThreads / 32;
constexpr int kGrowLayerThreads = 128;  // warps that run the frontier layers
constexpr int kGrowTreeCluster = 2;     // CTAs per tree: each reduces half of its rows

__host__ __device__ inline int grow_nstage(int nchunks, int K) {
  const size_t fit = kGrowStageBudget / grow_stage_bytes(nchunks, K);
  return (int)(fit < (size_t)kGrowTreeWarps ? fit : (size_t)kGrowTreeWarps);
}
// The rows' results, then one area used first for staging the rows' chunk
// records and then, once every row is reduced, for the selection.
__host__ __device__ inline size_t grow_tree_smem(int nchunks, int K, int rows, int nnodes) {
  const size_t stage = (size_t)grow_nstage(nchunks, K) * grow_stage_bytes(nchunks, K);
  // the selection: every non-root node's key by id and by layer rank, its
  // rank within its layer, and the kept flags / new ids
  const size_t select = (size_t)(nnodes - 1) * (2 * sizeof(unsigned long long) + sizeof(int)) +
                        (size_t)nnodes * sizeof(int);
  return grow_row_bytes(rows, K) + (stage > select ? stage : select);
}
constexpr size_t kGrowTreeSmem =
    ((size_t)kGrowMaxRows * kGrowMaxK * 16 + (size_t)kGrowMaxRows * 20 + 15) / 16 * 16 +
    kGrowStageBudget;

// A cluster of two CTAs per tree.  A draft row's K best tokens and their
// ln q do not depend on which node the frontier put in the row's slot, so
// every row of the tree is reduced first, each CTA taking half of the rows:
// a warp per row merges the chunk normalisers and ranks the candidates of
// the row's live records (one per row segment) a lane each; rows with more
// candidates than lanes are staged in shared memory, nstage at a time, and
// warp w picks the K best from the chunk lists (each sorted best first) by
// a threshold and a shuffle ranking; then a thread per row takes log2 of the row sum and
// a thread per (row, rank) its ln q = (z s - R - log2 S) ln 2, in float64.
// The second CTA's results reach the first through distributed shared
// memory and the second CTA exits.  The layers then run on four warps of the
// first CTA: a child's value is its parent's plus the row's ln q, and the
// next frontier is the K children ranked best among the layer's children.
// Finally the M best non-root nodes by (value desc, creation asc) are kept:
// each layer's children are ranked while the layer runs, and a node's rank
// over all layers adds binary searches in the other layers' ranked keys.
// The kept nodes are renumbered in creation order.  Launched
// programmatically after the top-k grid and waits for it before reading the
// records.
__global__ void __launch_bounds__(kGrowTreeThreads, 1) grow_tree_kernel(const GrowParams p) {
  extern __shared__ __align__(16) uint8_t grow_mem[];
  constexpr int kMaxKids = kGrowMaxK * kGrowMaxK;
  __shared__ double s_dval[kMaxKids];             // the layer's children: value
  __shared__ unsigned long long s_val[kMaxKids];  // ... its order key
  __shared__ int s_front[kGrowMaxK];              // frontier: node id
  __shared__ double s_fval[kGrowMaxK];            // ... and value
  __shared__ int s_wtot[kGrowTreeWarps];
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.x / kGrowTreeCluster;
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
  // the next call's first kernel may become resident; it waits for this grid
  asm volatile("griddepcontrol.launch_dependents;");

  // 1. this CTA's half of the tree's rows, [qa, qb): normaliser and K best
  //    tokens (float arithmetic).  The streaming top-k leaves a row's
  //    result in one record per row segment (the segment's last chunk) and
  //    empty records (reference kRefEmpty, no candidates) elsewhere, so a
  //    row usually has one live record, two when it is split between CTAs.
  //    First a warp per row reads the records' headers, merges the
  //    normaliser and, when the live records hold at most 32 candidates,
  //    ranks them a lane each.  Rows with more go to the staged merge
  //    below, nstage rows at a time: the CTA stages their chunk records
  //    together, then warp w reduces the w-th of them.
  const int half = (rows + 1) / 2;
  const int qa = crank == 0 ? 0 : half, qb = crank == 0 ? half : rows;
  __shared__ int s_fb[kGrowMaxRows];  // rows left to the staged merge
  __shared__ int s_nfb;
  if (threadIdx.x == 0) s_nfb = 0;
  __syncthreads();
  for (int q = qa + warp; q < qb; q += kGrowTreeWarps) {
    const GrowRec* rec = p.rec + ((size_t)b * rows + q) * p.nchunks;
    int lref = kRefEmpty;
    FSum acc = FSum::zero();
    unsigned live = 0;
    for (int c0 = 0; c0 < p.nchunks; c0 += 32) {
      const int c = c0 + lane;
      int gref = kRefEmpty;
      FSum v = FSum::zero();
      if (c < p.nchunks) {
        gref = __ldcg(&rec[c].ref);
        v.hi = __ldcg(&rec[c].hi);
        v.lo = __ldcg(&rec[c].lo);
      }
      if (c0 == 0) live = __ballot_sync(0xffffffffu, gref != kRefEmpty);
      if (gref > lref) {
        acc.scale(pow2i_f(lref - gref));
        lref = gref;
      }
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
    const int nl = __popc(live);
    if (p.nchunks > 32 || nl * K > 32) {  // the staged merge takes this row
      if (lane == 0) s_fb[atomicAdd(&s_nfb, 1)] = q;
      continue;
    }
    // candidate e of the j-th live record, a lane each (placeholders: index
    // >= V), ranked against one another by shuffles
    const int j = lane / K, e = lane - j * K;
    float v = -INFINITY;
    int x = 0x7FFFFFFF;
    if (j < nl) {
      unsigned m = live;  // drop the j live records before this lane's
      for (int t = 0; t < j; ++t) m &= m - 1;
      const int c = __ffs(m) - 1;
      const int xi = __ldcg(&rec[c].idx[e]);
      if (xi < p.V) {
        v = __ldcg(&rec[c].val[e]);
        x = xi;
      }
    }
    int rank = 0;
#pragma unroll 8
    for (int u = 0; u < 32; ++u) {
      const float vu = __shfl_sync(0xffffffffu, v, u);
      const int xu = __shfl_sync(0xffffffffu, x, u);
      rank += (xu != 0x7FFFFFFF && grow_better(vu, xu, v, x)) ? 1 : 0;
    }
    // fewer than K candidates (a row whose finite logits are fewer than K
    // keeps -inf candidates in records marked empty): the staged merge
    if (__popc(__ballot_sync(0xffffffffu, x != 0x7FFFFFFF)) < K) {
      if (lane == 0) s_fb[atomicAdd(&s_nfb, 1)] = q;
      continue;
    }
    if (x != 0x7FFFFFFF && rank < K) {
      r_z[q * K + rank] = v;
      r_tok[q * K + rank] = x;
    }
  }
  __syncthreads();
  const int nfb = s_nfb;
  {
    const size_t sb = grow_stage_bytes(p.nchunks, K);
    uint8_t* stage0 = grow_mem + grow_row_bytes(rows, K);
    for (int q0 = 0; q0 < nfb; q0 += nstage) {
      const int nb = min(nstage, nfb - q0);
      // asynchronous 4-byte copies: every load of the batch is in flight at once
      for (int i = threadIdx.x; i < nb * ncand; i += kGrowTreeThreads) {
        const int w = i / ncand, k = i - w * ncand;
        const int c = k / K, r = k - c * K;
        const GrowRec& g = p.rec[((size_t)b * rows + s_fb[q0 + w]) * p.nchunks + c];
        float* cv = reinterpret_cast<float*>(stage0 + (size_t)w * sb);
        grow_cp4(cv + k, &g.val[r]);
        grow_cp4(reinterpret_cast<int*>(cv + ncand) + k, &g.idx[r]);
      }
      for (int i = threadIdx.x; i < nb * p.nchunks; i += kGrowTreeThreads) {
        const int w = i / p.nchunks, c = i - w * p.nchunks;
        const GrowRec& g = p.rec[((size_t)b * rows + s_fb[q0 + w]) * p.nchunks + c];
        int* hp = reinterpret_cast<int*>(stage0 + (size_t)w * sb) + 2 * (size_t)ncand;
        hp[c] = 0;
        grow_cp4(hp + p.nchunks + c, &g.ref);
        grow_cp4(hp + 2 * p.nchunks + c, &g.hi);
        grow_cp4(hp + 3 * p.nchunks + c, &g.lo);
      }
      asm volatile("cp.async.commit_group;\ncp.async.wait_all;" ::: "memory");
      __syncthreads();
      if (warp < nb) {
        const int q = s_fb[q0 + warp];
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
  for (int q = qa + (int)threadIdx.x; q < qb; q += kGrowTreeThreads)
    r_l2[q] = log2((double)r_hi[q] + (double)r_lo[q]);
  __syncthreads();
  for (int t = qa * K + (int)threadIdx.x; t < qb * K; t += kGrowTreeThreads) {
    const int q = t / K;
    r_lnq[t] = ((double)r_z[t] * (double)p.scale - (double)r_R[q] - r_l2[q]) * 0.6931471805599453;
  }
  // the second CTA's rows (ln q and tokens) into the first CTA's shared
  // memory, at the same offsets; the second CTA is done after that
  cluster.sync();
  if (crank == 0) {
    const double* peer_lnq = cluster.map_shared_rank(r_lnq, 1);
    const int* peer_tok = cluster.map_shared_rank(r_tok, 1);
    for (int t = half * K + (int)threadIdx.x; t < rows * K; t += kGrowTreeThreads) {
      r_lnq[t] = peer_lnq[t];
      r_tok[t] = peer_tok[t];
    }
  }
  cluster.sync();  // the second CTA's shared memory is no longer read
  if (crank != 0) return;

  // the selection's arrays, in the staging area (free now), written by the
  // layers: each non-root node's key by id (node id - 1), each layer's keys in
  // rank order (the layer's block of the same index range) and each node's
  // rank within its layer; the other warps clear the kept flags meanwhile
  const int n = nnodes - 1;  // non-root nodes, ids 1..nnodes-1
  unsigned long long* s_ikey =
      reinterpret_cast<unsigned long long*>(grow_mem + grow_row_bytes(rows, K));  // [n]
  unsigned long long* s_lkey = s_ikey + n;                                        // [n]
  int* s_lrank = reinterpret_cast<int*>(s_lkey + n);                              // [n]
  int* s_new = s_lrank + n;                                                       // [nnodes]

  // 3. the layers, on warps 0-3 (named barrier 2 over their 128 threads):
  //    the children's values, then the next frontier, the K children of best
  //    rank; a child's rank (the children before it) is counted by two
  //    threads over half of the layer's children each
  if (threadIdx.x < kGrowLayerThreads) {
    const int lt = threadIdx.x;
    if (lt == 0) {  // the root
      nval[0] = 0.0;
      npar[0] = -1;
      ntok[0] = -1;
      ndep[0] = 0;
      s_front[0] = 0;
      s_fval[0] = 0.0;
    }
    asm volatile("bar.sync 2, %0;" ::"n"(kGrowLayerThreads) : "memory");
    for (int layer = 0; layer < p.D; ++layer) {
      const int nfront = layer == 0 ? 1 : K;
      const int base = layer == 0 ? 1 : 1 + K + (layer - 1) * K * K;
      const int q0 = layer == 0 ? 0 : 1 + (layer - 1) * K;  // the layer's first row
      const int nc = nfront * K;
      for (int t = lt; t < nc; t += kGrowLayerThreads) {
        const int slot = t / K;
        const double val = s_fval[slot] + r_lnq[(size_t)q0 * K + t];
        const int id = base + t;
        nval[id] = val;
        npar[id] = s_front[slot];
        ntok[id] = r_tok[(size_t)q0 * K + t];
        ndep[id] = layer + 1;
        s_dval[t] = val;
        const unsigned long long key = grow_key(val);
        s_val[t] = key;
        s_ikey[id - 1] = key;
      }
      asm volatile("bar.sync 2, %0;" ::"n"(kGrowLayerThreads) : "memory");
      {  // every layer's ranks (the last layer's for the selection only)
        const int half = nc >> 1;
        const int u0 = (lt & 1) ? half : 0, u1 = (lt & 1) ? nc : half;
        // every thread runs the same trips: the pair's shuffle is warp-wide
        for (int c0 = 0; c0 < nc; c0 += kGrowLayerThreads / 2) {
          const int c = c0 + (lt >> 1);
          const bool have = c < nc;
          int rank = 0;
          if (have) {
            const unsigned long long v = s_val[c];
#pragma unroll 8
            for (int u = u0; u < u1; ++u) {
              const unsigned long long o = s_val[u];
              rank += (o > v || (o == v && u < c)) ? 1 : 0;
            }
          }
          rank += __shfl_xor_sync(0xffffffffu, rank, 1);
          if (have && (lt & 1) == 0) {
            s_lkey[base - 1 + rank] = s_val[c];
            s_lrank[base - 1 + c] = rank;
            if (rank < K && layer + 1 < p.D) {
              s_front[rank] = base + c;
              s_fval[rank] = s_dval[c];
            }
          }
        }
        asm volatile("bar.sync 2, %0;" ::"n"(kGrowLayerThreads) : "memory");
      }
    }
  } else {
    const int t = threadIdx.x - kGrowLayerThreads;
    for (int i = t; i < nnodes; i += kGrowTreeThreads - kGrowLayerThreads) s_new[i] = 0;
  }
  __syncthreads();

  // keep the M best non-root nodes by (value key desc, id asc): a node's
  // rank among all of them is its rank within its layer plus, for every other
  // layer, how many of that layer's children come before it, found by binary
  // search in the layer's keys in rank order.  On equal keys the node with
  // the smaller id comes first, and every id of an earlier layer is smaller.
  for (int i = threadIdx.x; i < n; i += kGrowTreeThreads) {
    const int L = i < K ? 0 : 1 + (i - K) / (K * K);
    const unsigned long long v = s_ikey[i];
    int g = s_lrank[i];
    for (int L2 = 0; L2 < p.D && g < p.M; ++L2) {
      if (L2 == L) continue;
      const int b0 = L2 == 0 ? 0 : K + (L2 - 1) * K * K;
      int lo = 0, hi = L2 == 0 ? K : K * K;  // the first entry not before v
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const unsigned long long e = s_lkey[b0 + mid];
        if (e > v || (e == v && L2 < L))
          lo = mid + 1;
        else
          hi = mid;
      }
      g += lo;
    }
    if (g < p.M) s_new[i + 1] = 1;
  }
  __syncthreads();
  {
    // renumber in creation order (parents come first): thread t owns the
    // contiguous ids [t per, (t + 1) per) of 1..nnodes-1; an exclusive scan
    // of the kept counts gives each range's first new id
    const int per = (n + kGrowTreeThreads - 1) / kGrowTreeThreads;
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
  for (int v = 1 + threadIdx.x; v < nnodes; v += kGrowTreeThreads) {
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
