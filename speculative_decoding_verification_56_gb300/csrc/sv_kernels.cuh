// sv_kernels.cuh -- verification kernels for sm_103a.
//
// Sampling verification ("EAGLE-3 speculative decoding review", sections
// "Speculative Decoding" step 3 and "Does Using a Small Model's Answer Reduce
// Quality?"; "EAGLE math", "Vanilla speculative decoding"):
//   sample_stats_kernel   pass 1: one streaming read of all 2k+1 rows of every
//                         sequence; per-chunk softmax partials, per-row merge,
//                         p(x_i)/q(x_i), accept test and first rejection.
//   sample_draw_kernel    pass 2: re-reads only the selected row (pair) of each
//                         sequence: residual max(0, p - q) after a rejection,
//                         else p of the bonus row; chunk sums, then the last
//                         CTA of the sequence draws the token by inverse CDF.
// Greedy and tree verification ("Does Using a Small Model's Answer Reduce
// Quality?" greedy bullets; "EAGLE-2"; "The Complete EAGLE-3 Inference
// Process" step 4):
//   argmax_verify_kernel  one streaming read of every target row; per-chunk
//                         argmax, per-row merge, then the last CTA of each
//                         sequence (tree) resolves the accepted prefix (path).
//
// Softmax arithmetic: with s = log2(e) / T, p_j = 2^(z_j s - R) / S where R
// is an integer reference >= max_j z_j s.  Integer references make every
// rescaling between threads, chunks and rows an exact power of two.
#pragma once

#include "sv_device.cuh"

namespace sv {

// ---------------------------------------------------------------------------
// Workspace records
// ---------------------------------------------------------------------------
struct SoftmaxPartial {  // one (row, chunk)
  int ref;
  int pad;
  double sum;  // sum of 2^(z s - ref) over the chunk
};
struct RowStats {  // one row after the merge
  int ref;       // integer reference R of the row
  float inv_sum; // 1 / S rounded to float
  double sum;    // S = sum_j 2^(z_j s - R)
  double prob;   // p (or q) of the row's draft token, float64
};
struct ArgPartial {
  float val;
  int idx;
};

struct SampleParams {
  const void* target;   // [B, k+1, V]
  const void* draft;    // [B, k, V]
  const int32_t* tokens;
  const float* u_accept;
  const float* u_sample;
  float scale;          // log2(e) / T
  int B, k, V, nchunks;
  int32_t* accepted_len;
  int32_t* out_tokens;
  float* p_out;
  float* q_out;
  float* resid_mass;
  // workspace
  unsigned* flags;
  unsigned* row_cnt;    // [B*(2k+1)]
  unsigned* seq_cnt;    // [B]
  unsigned* draw_cnt;   // [B]
  SoftmaxPartial* part; // [B*(2k+1)*nchunks]
  RowStats* rows;       // [B*(2k+1)]
  int32_t* sel;         // [B]
  double* csum;         // [B*nchunks]
};

// Row r of sequence b: r in [0, k] is target row r, r in [k+1, 2k] is draft
// row r-k-1.
template <typename E>
__device__ __forceinline__ const typename E::storage* seq_row_ptr(const SampleParams& p, int b,
                                                                  int r) {
  using S = typename E::storage;
  if (r <= p.k)
    return reinterpret_cast<const S*>(p.target) + ((size_t)b * (p.k + 1) + r) * (size_t)p.V;
  return reinterpret_cast<const S*>(p.draft) + ((size_t)b * p.k + (r - p.k - 1)) * (size_t)p.V;
}

// ---------------------------------------------------------------------------
// Pass 1: softmax statistics, accept test, first rejection
// ---------------------------------------------------------------------------
template <typename E, bool kVec>
__global__ void __launch_bounds__(kThreads) sample_stats_kernel(const SampleParams p) {
  __shared__ int s_ref[kWarps];
  __shared__ float s_sum[kWarps];
  __shared__ int s_flag;

  const int rows_per_seq = 2 * p.k + 1;
  const int item = blockIdx.x;
  const int row = item / p.nchunks;  // global row id b * (2k+1) + r
  const int c = item - row * p.nchunks;
  const int b = row / rows_per_seq;
  const int r = row - b * rows_per_seq;
  const int j0 = c * E::kChunk;
  const int j1 = min(p.V, j0 + E::kChunk);
  const typename E::storage* rp = seq_row_ptr<E>(p, b, r);

  float z[kVecPerThread][E::kEPV];
  load_chunk<E, kVec>(rp, j0, j1, z);

  // the dependent draw kernel may start its launch now
  asm volatile("griddepcontrol.launch_dependents;");

  float m = -INFINITY;
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q)
#pragma unroll
    for (int e = 0; e < E::kEPV; ++e) m = fmaxf(m, z[q][e]);
  const int ref = exp_ref(m, p.scale);
  const float nref = -(float)ref;
  float acc = 0.0f;
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) {
    float t[E::kEPV];
#pragma unroll
    for (int e = 0; e < E::kEPV; ++e) t[e] = ex2(__fmaf_rn(z[q][e], p.scale, nref));
    // pairwise sum of the vector
#pragma unroll
    for (int w = E::kEPV / 2; w > 0; w >>= 1)
#pragma unroll
      for (int e = 0; e < w; ++e) t[e] = __fadd_rn(t[e], t[e + w]);
    acc = __fadd_rn(acc, t[0]);
  }

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int wref = warp_max_i(ref);
  if (lane == 0) s_ref[warp] = wref;
  __syncthreads();
  int bref = s_ref[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) bref = max(bref, s_ref[w]);
  float wsum = warp_sum_f(acc * pow2i_f(ref - bref));
  if (lane == 0) s_sum[warp] = wsum;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot += (double)s_sum[w];
    SoftmaxPartial sp;
    sp.ref = bref;
    sp.pad = 0;
    sp.sum = tot;
    p.part[item] = sp;
  }

  if (!arrive_last(&p.row_cnt[row], (unsigned)p.nchunks, &s_flag)) return;

  // ---- this CTA finishes the row: merge the chunk partials (fixed order) ----
  if (warp == 0) {
    int lref = kRefEmpty;
    for (int cc = lane; cc < p.nchunks; cc += 32)
      lref = max(lref, __ldcg(&p.part[(size_t)row * p.nchunks + cc].ref));
    const int R = warp_max_i(lref);
    double lsum = 0.0;
    for (int cc = lane; cc < p.nchunks; cc += 32) {
      const SoftmaxPartial* pp = &p.part[(size_t)row * p.nchunks + cc];
      lsum += __ldcg(&pp->sum) * pow2i_d(__ldcg(&pp->ref) - R);
    }
    const double S = warp_sum_d(lsum);
    if (lane == 0) {
      double prob = 0.0;
      if (r != p.k) {  // rows with a draft token: target r < k, draft r > k
        const int i = (r < p.k) ? r : r - p.k - 1;
        const int x = p.tokens[(size_t)b * p.k + i];
        if (x >= 0 && x < p.V) {
          const float zx = E::load1(rp + x);
          const float xs = __fmaf_rn(zx, p.scale, -(float)R);
          prob = exp2((double)xs) / S;
        } else {
          set_flag(p.flags, 1u);
        }
      }
      RowStats rs;
      rs.ref = R;
      rs.inv_sum = (float)(1.0 / S);
      rs.sum = S;
      rs.prob = prob;
      p.rows[row] = rs;
    }
  }

  if (!arrive_last(&p.seq_cnt[b], (unsigned)rows_per_seq, &s_flag)) return;

  // ---- this CTA finishes the sequence: accept test left to right ----
  if (threadIdx.x == 0) {
    const size_t rb = (size_t)b * rows_per_seq;
    int n = p.k;
    for (int i = 0; i < p.k; ++i) {
      const double pi = __ldcg(&p.rows[rb + i].prob);
      const double qi = __ldcg(&p.rows[rb + p.k + 1 + i].prob);
      p.p_out[(size_t)b * p.k + i] = (float)pi;
      p.q_out[(size_t)b * p.k + i] = (float)qi;
      if (n == p.k) {
        const double u = (double)p.u_accept[(size_t)b * p.k + i];
        if (!(u * qi < pi)) n = i;
      }
    }
    p.accepted_len[b] = n;
    for (int i = 0; i <= p.k; ++i)
      p.out_tokens[(size_t)b * (p.k + 1) + i] = (i < n) ? p.tokens[(size_t)b * p.k + i] : -1;
    p.sel[b] = n;
  }
}

// ---------------------------------------------------------------------------
// Pass 2: residual / bonus draw by inverse CDF
// ---------------------------------------------------------------------------
struct DrawRows {
  const void* t;  // target row
  const void* d;  // draft row (nullptr: weights are p of the target row)
  float nref_t, inv_t, nref_d, inv_d;
};

// Weight of one element; explicit round-to-nearest intrinsics keep every
// evaluation bit-identical (no contraction differences between call sites).
__device__ __forceinline__ float draw_weight(float zt, float zd, float s, const DrawRows& w,
                                             bool resid) {
  const float pt = __fmul_rn(ex2(__fmaf_rn(zt, s, w.nref_t)), w.inv_t);
  if (!resid) return pt;
  const float pd = __fmul_rn(ex2(__fmaf_rn(zd, s, w.nref_d)), w.inv_d);
  return fmaxf(__fsub_rn(pt, pd), 0.0f);
}

// Sequential float sum of one vector's weights (the "group sum").
template <typename E, bool kVec>
__device__ __forceinline__ void chunk_group_sums(const DrawRows& w, bool resid, float s, int j0,
                                                 int j1, float (&g)[kVecPerThread]) {
  using S = typename E::storage;
  float zt[kVecPerThread][E::kEPV];
  float zd[kVecPerThread][E::kEPV];
  load_chunk<E, kVec>(reinterpret_cast<const S*>(w.t), j0, j1, zt);
  if (resid) load_chunk<E, kVec>(reinterpret_cast<const S*>(w.d), j0, j1, zd);
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) {
    float a = 0.0f;
#pragma unroll
    for (int e = 0; e < E::kEPV; ++e)
      a = __fadd_rn(a, draw_weight(zt[q][e], resid ? zd[q][e] : 0.0f, s, w, resid));
    g[q] = a;
  }
}

// Lane-level two-sum over 32 consecutive groups held in shared memory, then an
// inclusive warp scan in float64.  Lane l owns [excl_l, inc_l) with excl_l
// taken from lane l-1's inclusive value, so the lanes tile [0, inc_31).
__device__ __forceinline__ double lane_scan(const float* s_g, int lane, double* excl) {
  FSum acc;
#pragma unroll 8
  for (int g = 0; g < 32; ++g) acc.add(s_g[lane * 32 + g]);
  double inc = acc.value();
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  const double prev = __shfl_up_sync(0xffffffffu, inc, 1);
  *excl = lane == 0 ? 0.0 : prev;
  return inc;
}

template <typename E>
__device__ __forceinline__ DrawRows draw_rows(const SampleParams& p, int b, int n, bool resid) {
  using S = typename E::storage;
  const int rows_per_seq = 2 * p.k + 1;
  const size_t rb = (size_t)b * rows_per_seq;
  DrawRows w;
  const RowStats rt = p.rows[rb + n];
  w.t = reinterpret_cast<const S*>(p.target) + ((size_t)b * (p.k + 1) + n) * (size_t)p.V;
  w.nref_t = -(float)rt.ref;
  w.inv_t = rt.inv_sum;
  w.d = nullptr;
  w.nref_d = 0.0f;
  w.inv_d = 0.0f;
  if (resid) {
    const RowStats rd = p.rows[rb + p.k + 1 + n];
    w.d = reinterpret_cast<const S*>(p.draft) + ((size_t)b * p.k + n) * (size_t)p.V;
    w.nref_d = -(float)rd.ref;
    w.inv_d = rd.inv_sum;
  }
  return w;
}

// Sum of one chunk's weights, computed the same way the final scan walks them.
template <typename E, bool kVec>
__device__ double chunk_total(const DrawRows& w, bool resid, float s, int j0, int j1, float* s_g,
                              double* s_tot) {
  float g[kVecPerThread];
  chunk_group_sums<E, kVec>(w, resid, s, j0, j1, g);
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) s_g[q * kThreads + threadIdx.x] = g[q];
  __syncthreads();
  if (threadIdx.x < 32) {
    double excl;
    const double inc = lane_scan(s_g, threadIdx.x, &excl);
    if (threadIdx.x == 31) *s_tot = inc;
  }
  __syncthreads();
  const double t = *s_tot;
  __syncthreads();
  return t;
}

template <typename E, bool kVec>
__global__ void __launch_bounds__(kThreads) sample_draw_kernel(const SampleParams p) {
  __shared__ float s_g[kGroupsPerChunk];
  __shared__ double s_tot;
  __shared__ int s_flag;
  __shared__ int s_tok;

  // wait for the stats kernel's results (programmatic dependent launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int item = blockIdx.x;
  const int b = item / p.nchunks;
  const int c = item - b * p.nchunks;
  const int n = p.sel[b];
  bool resid = n < p.k;
  DrawRows w = draw_rows<E>(p, b, n, resid);

  {
    const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
    const double t = chunk_total<E, kVec>(w, resid, p.scale, j0, j1, s_g, &s_tot);
    if (threadIdx.x == 0) p.csum[item] = t;
  }

  if (!arrive_last(&p.draw_cnt[b], (unsigned)p.nchunks, &s_flag)) return;

  // ---- last CTA of sequence b: locate the chunk, then the token ----
  double* cs = p.csum + (size_t)b * p.nchunks;
  double total = 0.0;
  if (threadIdx.x == 0) {
    for (int cc = 0; cc < p.nchunks; ++cc) total += __ldcg(&cs[cc]);
    s_tot = total;
  }
  __syncthreads();
  total = s_tot;
  __syncthreads();
  bool fallback = false;
  if (resid && !(total > 0.0)) {
    // residual mass vanished in rounding: sample p of the rejected row instead
    fallback = true;
    resid = false;
    w.d = nullptr;
    total = 0.0;
    for (int cc = 0; cc < p.nchunks; ++cc) {
      const int j0 = cc * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
      const double t = chunk_total<E, kVec>(w, false, p.scale, j0, j1, s_g, &s_tot);
      if (threadIdx.x == 0) {
        cs[cc] = t;
        total += t;
      }
    }
    if (threadIdx.x == 0) {
      s_tot = total;
      set_flag(p.flags, 8u);
    }
    __syncthreads();
    total = s_tot;
    __syncthreads();
  }

  const double target = (double)p.u_sample[b] * total;
  // chunk holding the target: first chunk whose inclusive prefix exceeds it
  if (threadIdx.x == 0) {
    double cum = 0.0, base = 0.0;
    int cstar = -1, lastpos = 0;
    for (int cc = 0; cc < p.nchunks; ++cc) {
      const double v = __ldcg(&cs[cc]);
      if (v > 0.0) lastpos = cc;
      if (cstar < 0 && target < cum + v) {
        cstar = cc;
        base = cum;
      }
      cum += v;
    }
    if (cstar < 0) {  // rounding: last chunk with positive mass
      cstar = lastpos;
      base = cum - __ldcg(&cs[lastpos]);
    }
    s_flag = cstar;
    s_tot = base;
  }
  __syncthreads();
  const int cstar = s_flag;
  const double base = s_tot;
  __syncthreads();

  const int j0 = cstar * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
  float g[kVecPerThread];
  chunk_group_sums<E, kVec>(w, resid, p.scale, j0, j1, g);
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) s_g[q * kThreads + threadIdx.x] = g[q];
  if (threadIdx.x == 0) s_tok = -1;
  __syncthreads();
  if (threadIdx.x < 32) {
    using S = typename E::storage;
    const int lane = threadIdx.x;
    double excl;
    const double inc = lane_scan(s_g, lane, &excl);
    // the lane whose range [base+excl, base+inc) holds the target walks it;
    // if rounding left the target outside every range, the last lane with
    // positive mass takes its last positive element
    const bool mine = target >= base + excl && target < base + inc;
    const unsigned own = __ballot_sync(0xffffffffu, mine);
    const unsigned pos = __ballot_sync(0xffffffffu, inc > excl);
    const int owner = own ? (__ffs(own) - 1) : (pos ? (31 - __clz(pos)) : 0);
    const bool exact = own != 0;
    if (lane == owner) {
      FSum acc;
      int tok = -1, lastg = -1;
      for (int gi = 0; gi < 32; ++gi) {
        const int vi = lane * 32 + gi;
        const float gs = s_g[vi];
        if (!(gs > 0.0f)) continue;
        lastg = gi;
        FSum nxt = acc;
        nxt.add(gs);
        if (exact && target < base + excl + nxt.value()) {
          // the target lies in this vector: walk its elements in order
          const double before = base + excl + acc.value();
          const int e0 = j0 + vi * E::kEPV;
          float part = 0.0f;
          int lastpos = -1;
          for (int e = 0; e < E::kEPV && e0 + e < j1; ++e) {
            const float zt = E::load1(reinterpret_cast<const S*>(w.t) + e0 + e);
            const float zd = resid ? E::load1(reinterpret_cast<const S*>(w.d) + e0 + e) : 0.0f;
            const float we = draw_weight(zt, zd, p.scale, w, resid);
            part = __fadd_rn(part, we);
            if (we > 0.0f) lastpos = e0 + e;
            if (target < before + (double)part) {
              tok = e0 + e;
              break;
            }
          }
          if (tok < 0) tok = lastpos;  // rounding inside the vector
          break;
        }
        acc = nxt;
      }
      if (tok < 0 && lastg >= 0) {  // rounding: last positive element of the lane
        const int e0 = j0 + (lane * 32 + lastg) * E::kEPV;
        for (int e = 0; e < E::kEPV && e0 + e < j1; ++e) {
          const float zt = E::load1(reinterpret_cast<const S*>(w.t) + e0 + e);
          const float zd = resid ? E::load1(reinterpret_cast<const S*>(w.d) + e0 + e) : 0.0f;
          if (draw_weight(zt, zd, p.scale, w, resid) > 0.0f) tok = e0 + e;
        }
      }
      s_tok = tok;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int tok = s_tok;
    if (tok < 0) tok = j0;  // unreachable with finite inputs
    p.out_tokens[(size_t)b * (p.k + 1) + n] = tok;
    p.resid_mass[b] = (n < p.k && !fallback) ? (float)total : 0.0f;
  }
}

// ---------------------------------------------------------------------------
// Greedy and tree verification: argmax of every target row
// ---------------------------------------------------------------------------
struct ArgmaxParams {
  const void* target;  // [B, rows_per_seq, V]
  const int32_t* tokens;   // chain: [B, k]; tree: [B, N]
  const int32_t* parents;  // tree only: [B, N]
  int B, rows_per_seq, V, nchunks;
  int tree;       // 0 = chain greedy (rows_per_seq = k+1), 1 = tree (rows_per_seq = N)
  int max_depth;  // tree only
  int32_t* accepted_len;
  int32_t* out_tokens;  // chain: [B, k+1]; tree: [B, max_depth+1]
  int32_t* path_nodes;  // tree: [B, max_depth+1]
  unsigned* flags;
  unsigned* row_cnt;  // [B*rows_per_seq]
  unsigned* seq_cnt;  // [B]
  ArgPartial* part;   // [B*rows_per_seq*nchunks]
  int32_t* rowarg;    // [B*rows_per_seq]
};

// Chain resolve ("accept while the draft equals the target argmax").
__device__ void resolve_chain(const ArgmaxParams& p, int b) {
  if (threadIdx.x != 0) return;
  const int k = p.rows_per_seq - 1;
  const int32_t* g = p.rowarg + (size_t)b * p.rows_per_seq;
  int n = k;
  for (int i = 0; i < k; ++i) {
    const int x = p.tokens[(size_t)b * k + i];
    if (x < 0 || x >= p.V) set_flag(p.flags, 1u);
    if (x != __ldcg(&g[i])) {
      n = i;
      break;
    }
  }
  p.accepted_len[b] = n;
  for (int i = 0; i <= k; ++i) {
    int v = -1;
    if (i < n) v = p.tokens[(size_t)b * k + i];
    else if (i == n) v = __ldcg(&g[n]);
    p.out_tokens[(size_t)b * (k + 1) + i] = v;
  }
}

// Tree resolve: one thread per node walks to the root (at most max_depth + 1
// hops), then a block max over (depth, -node) picks the winner.
__device__ void resolve_tree(const ArgmaxParams& p, int b, unsigned long long* s_key) {
  const int N = p.rows_per_seq;
  const int32_t* par = p.parents + (size_t)b * N;
  const int32_t* tok = p.tokens + (size_t)b * N;
  const int32_t* g = p.rowarg + (size_t)b * N;
  const int W = p.max_depth + 1;
  unsigned long long best = 0xFFFFFFFFull;  // root: depth 0, node 0
  unsigned bad = 0;
  for (int v = 1 + threadIdx.x; v < N; v += kThreads) {
    int cur = v, d = 0;
    bool ok = true;
    while (cur != 0) {
      const int pa = par[cur];
      if (pa < 0 || pa >= cur) {
        bad |= 2u;
        ok = false;
        break;
      }
      const int tv = tok[cur];
      if (tv < 0 || tv >= p.V) bad |= 1u;
      if (tv != __ldcg(&g[pa])) ok = false;
      if (++d > p.max_depth) {
        bad |= 4u;
        ok = false;
        break;
      }
      cur = pa;
    }
    if (ok) {
      const unsigned long long key =
          ((unsigned long long)d << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)v);
      if (key > best) best = key;
    }
  }
  if (bad) set_flag(p.flags, bad);
  // block max
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
    best = y > best ? y : best;
  }
  if ((threadIdx.x & 31) == 0) s_key[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long k = s_key[0];
    for (int w = 1; w < kWarps; ++w) k = s_key[w] > k ? s_key[w] : k;
    s_key[0] = k;
  }
  __syncthreads();
  const unsigned long long key = s_key[0];
  const int depth = (int)(key >> 32);
  const int vstar = (int)(0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFull));
  for (int i = threadIdx.x; i < W; i += kThreads) {
    if (i > depth) {
      p.path_nodes[(size_t)b * W + i] = -1;
      p.out_tokens[(size_t)b * W + i] = -1;
    }
  }
  if (threadIdx.x == 0) {
    p.accepted_len[b] = depth;
    int cur = vstar;
    for (int i = depth; i >= 0; --i) {
      p.path_nodes[(size_t)b * W + i] = cur;
      if (i >= 1) p.out_tokens[(size_t)b * W + i - 1] = tok[cur];
      cur = (i >= 1) ? par[cur] : 0;
    }
    p.out_tokens[(size_t)b * W + depth] = __ldcg(&g[vstar]);
  }
}

template <typename E, bool kVec>
__global__ void __launch_bounds__(kThreads) argmax_verify_kernel(const ArgmaxParams p) {
  __shared__ float s_v[kWarps];
  __shared__ int s_i[kWarps];
  __shared__ int s_flag;
  __shared__ unsigned long long s_key[kWarps];

  const int item = blockIdx.x;
  const int row = item / p.nchunks;
  const int c = item - row * p.nchunks;
  const int b = row / p.rows_per_seq;
  const int j0 = c * E::kChunk;
  const int j1 = min(p.V, j0 + E::kChunk);
  const typename E::storage* rp =
      reinterpret_cast<const typename E::storage*>(p.target) + (size_t)row * p.V;

  float z[kVecPerThread][E::kEPV];
  load_chunk<E, kVec>(rp, j0, j1, z);
  float bv = -INFINITY;
  int bi = 0x7FFFFFFF;
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q)
#pragma unroll
    for (int e = 0; e < E::kEPV; ++e)
      if (z[q][e] > bv) {  // ascending index within the thread: strict keeps the lowest
        bv = z[q][e];
        bi = j0 + (q * kThreads + threadIdx.x) * E::kEPV + e;
      }
  warp_argmax(bv, bi);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    s_v[warp] = bv;
    s_i[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = s_v[0];
    int i = s_i[0];
    for (int w = 1; w < kWarps; ++w)
      if (better(s_v[w], s_i[w], v, i)) {
        v = s_v[w];
        i = s_i[w];
      }
    ArgPartial ap;
    ap.val = v;
    ap.idx = i;
    p.part[item] = ap;
  }

  if (!arrive_last(&p.row_cnt[row], (unsigned)p.nchunks, &s_flag)) return;

  if (warp == 0) {
    float v = -INFINITY;
    int i = 0x7FFFFFFF;
    for (int cc = lane; cc < p.nchunks; cc += 32) {
      const ArgPartial* pp = &p.part[(size_t)row * p.nchunks + cc];
      const float v2 = __ldcg(&pp->val);
      const int i2 = __ldcg(&pp->idx);
      if (better(v2, i2, v, i)) {
        v = v2;
        i = i2;
      }
    }
    warp_argmax(v, i);
    if (lane == 0) p.rowarg[row] = (i >= 0 && i < p.V) ? i : 0;
  }

  if (!arrive_last(&p.seq_cnt[b], (unsigned)p.rows_per_seq, &s_flag)) return;

  if (p.tree)
    resolve_tree(p, b, s_key);
  else
    resolve_chain(p, b);
}

}  // namespace sv
