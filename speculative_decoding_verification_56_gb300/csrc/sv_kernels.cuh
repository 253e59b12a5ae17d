// sv_kernels.cuh -- verification kernels for sm_103a.
//
// Sampling verification ("EAGLE-3 speculative decoding review", sections
// "Speculative Decoding" step 3 and "Does Using a Small Model's Answer Reduce
// Quality?"; "EAGLE math", "Vanilla speculative decoding"):
//   stats    one streaming read of all 2k+1 rows of every sequence: softmax
//            partials per row segment, per-row merge, p(x_i) and q(x_i), the
//            accept test and the first rejection (warp ballot).
//   draw     re-reads only the selected row (pair) of each sequence: residual
//            max(0, p - q) after a rejection, else p of the bonus row; chunk
//            sums, then the last CTA of the sequence draws the token by
//            inverse CDF.
// Greedy and tree verification ("Does Using a Small Model's Answer Reduce
// Quality?" greedy bullets; "EAGLE-2"; "The Complete EAGLE-3 Inference
// Process" step 4):
//   argmax   one streaming read of every target row: argmax per row segment,
//            per-row merge, then the last CTA of each sequence (tree) resolves
//            the accepted prefix (path).
//
// Two loaders feed the same per-thread arithmetic: a persistent kernel that
// streams contiguous ranges of 32 KB chunks through a ring of bulk async
// copies (rows whose bytes are a multiple of 16 at a 16-byte aligned base),
// and a one-CTA-per-chunk kernel with plain loads for any other row size.
//
// Softmax arithmetic: with s = log2(e) / T, p_j = 2^(z_j s - R) / S where R
// is an integer >= max_j z_j s.  Integer references make every rescaling
// between threads, segments and rows an exact power of two.
#pragma once

#include <cooperative_groups.h>

#include "sv_device.cuh"

namespace sv {

// ---------------------------------------------------------------------------
// Workspace records
// ---------------------------------------------------------------------------
// Segment records: a segment is a run of consecutive chunks of one row handled
// by one CTA.  The CTA writes one record in slot (row, first chunk) with nch =
// the segment's chunk count, and nch = 0 in the slots of its other chunks, so
// every slot is written on every call.  Within the CTA, each warp parks its
// partial in shared memory and the last warp to arrive combines them (no CTA
// barrier; see SegSlots).
struct SoftmaxPartial {
  int ref;
  int nch;
  float hi, lo;  // double-float sum of 2^(z s - ref) over the warp's elements
};
struct ArgPartial {
  float val;
  int idx;
  int nch;
  int pad;
};
struct RowStats {  // one row after the merge
  int ref;         // integer reference R of the row
  float inv_sum;   // 1 / S rounded to float
  float pm;        // p (or q) of the row's draft token is pm 2^pe exactly,
  int pe;          // and zero when pe < -1022 (the float64 range)
};

// What the draw needs of sequence b: the selected position n and the
// normalisers of its target (and, after a rejection, draft) row.
struct DrawDesc {
  int n;
  float nref_t, inv_t, nref_d, inv_d;
  int pad[3];
};

struct SampleParams {
  const void* target;  // [B, k+1, V]
  const void* draft;   // [B, k, V]
  const int32_t* tokens;
  const float* u_accept;
  const float* u_sample;
  float scale;  // log2(e) / T
  int B, k, V, nchunks, items;
  // rows of draft positions below keep_pos (target and draft) are streamed
  // with an L2 keep hint: the draw re-reads the rejected position's pair,
  // and early positions are the likely ones
  int keep_pos;
  int32_t* accepted_len;
  int32_t* out_tokens;
  float* p_out;
  float* q_out;
  float* resid_mass;
  // workspace
  unsigned* flags;
  SoftmaxPartial* part;  // [B*(2k+1) * nchunks]
  DrawDesc* desc;        // [B]
  // draw prefix structure per (sequence, chunk): group sums and chunk
  // totals; the _p arrays hold p-only weights of a rejected row (used when
  // its residual mass rounds to zero)
  float* gsum;     // [B*nchunks*kVecPerChunk]
  float* gsum_p;   // [B*nchunks*kVecPerChunk]
  FSum* csum;      // [B*nchunks]
  FSum* csum_p;    // [B*nchunks]
  float* zx;  // [rows] logit of each row's draft token, captured while it streams
  // limit of each wait on a bulk copy (kWaitLimitNs unless a test shortens
  // it to exercise the timeout path); drains always use kWaitLimitNs
  unsigned long long wait_ns;
  int nrec;   // statistics records per row (nchunks, or the LM head's CTAs)
  // the rows the draw re-reads, when they are not the logits inputs: fp32
  // [2B, V], row 2b the target row of sequence b's drawn position, 2b + 1 its
  // draft row (the LM head fused with sampling recomputes them); else null
  const float* drawn;
};

struct ArgmaxParams {
  const void* target;      // [B, rows_per_seq, V]
  const int32_t* tokens;   // chain: [B, k]; tree: [B, N]
  const int32_t* parents;  // tree only: [B, N]
  int B, rows_per_seq, V, nchunks, items;
  int tree;       // 0 = chain greedy (rows_per_seq = k+1), 1 = tree (rows_per_seq = N)
  int max_depth;  // tree only
  int32_t* accepted_len;
  int32_t* out_tokens;  // chain: [B, k+1]; tree: [B, max_depth+1]
  int32_t* path_nodes;  // tree: [B, max_depth+1]
  unsigned* flags;
  ArgPartial* part;   // [B*rows_per_seq * nchunks]
  int32_t* rowarg;    // [B*rows_per_seq]
  unsigned long long wait_ns;  // as SampleParams::wait_ns
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

// A 16-byte vector of elements j..j+kEPV-1 of a row; on the plain-load path
// elements at or past j1 read as -inf.
template <typename E, bool kVec>
__device__ __forceinline__ uint4 fetch_vec(const typename E::storage* row, int j, int j1) {
  if constexpr (kVec) {
    return ldg_stream(row + j);
  } else {
    uint32_t w[4];
    if constexpr (E::kEPV == 4) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = (j + e < j1) ? __float_as_uint(E::load1(row + j + e)) : 0xFF800000u;
    } else {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int j0 = j + 2 * h;
        const uint32_t lo = (j0 < j1) ? (uint32_t)reinterpret_cast<const uint16_t*>(row)[j0]
                                      : 0xFF80u;
        const uint32_t hi = (j0 + 1 < j1)
                                ? (uint32_t)reinterpret_cast<const uint16_t*>(row)[j0 + 1]
                                : 0xFF80u;
        w[h] = lo | (hi << 16);
      }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Draft token of row `row` of the sampling rows (target rows 0..k-1 and the
// draft rows carry one; the bonus row and rows past the end give -1).
__device__ __forceinline__ int row_token(const SampleParams& p, int row) {
  const int rows_per_seq = 2 * p.k + 1;
  if (row >= p.B * rows_per_seq) return -1;
  const int b = row / rows_per_seq, r = row - b * rows_per_seq;
  if (r == p.k) return -1;
  const int i = r < p.k ? r : r - p.k - 1;
  return __ldg(p.tokens + (size_t)b * p.k + i);
}

// Whether this thread holds element x of the chunk [j0, j1), and its logit.
template <typename E>
__device__ __forceinline__ bool capture_token_value(const uint4 (&raw)[kVecPerThread], int x,
                                                    int j0, int j1, float& z) {
  if (x < j0 || x >= j1) return false;
  const int off = x - j0, vi = off / E::kEPV;
  if ((vi & (kThreads - 1)) != (int)threadIdx.x) return false;
  const int q = vi / kThreads;
  const uint4 v = q == 0 ? raw[0] : q == 1 ? raw[1] : q == 2 ? raw[2] : raw[3];
  z = E::elem(v, off % E::kEPV);
  return true;
}
// The thread holding element x of the chunk [j0, j1) stores that logit, so
// that the merge needs no dependent load of it.
template <typename E>
__device__ __forceinline__ void capture_token(const SampleParams& p,
                                              const uint4 (&raw)[kVecPerThread], int x, int j0,
                                              int j1, int row) {
  float z;
  if (capture_token_value<E>(raw, x, j0, j1, z)) p.zx[row] = z;
}

// ---------------------------------------------------------------------------
// Per-thread arithmetic on one chunk (raw vectors in registers)
// ---------------------------------------------------------------------------
struct StatsState {  // running softmax partial of one thread over one segment
  int ref = kRefEmpty;
  FSum acc = FSum::zero();
};

// Element pairs of a 16-byte vector as f32x2 values: bf16 words split into
// (low, high) halves, fp32 vectors into (x, y) and (z, w).
template <typename E>
__device__ __forceinline__ void vec_pairs(const uint4& v, unsigned long long (&pr)[E::kEPV / 2]);
template <>
__device__ __forceinline__ void vec_pairs<BF16>(const uint4& v, unsigned long long (&pr)[4]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int h = 0; h < 4; ++h)
    pr[h] = f2pack(__uint_as_float(w[h] << 16), __uint_as_float(w[h] & 0xFFFF0000u));
}
template <>
__device__ __forceinline__ void vec_pairs<F32>(const uint4& v, unsigned long long (&pr)[2]) {
  pr[0] = f2pack(__uint_as_float(v.x), __uint_as_float(v.y));
  pr[1] = f2pack(__uint_as_float(v.z), __uint_as_float(v.w));
}

// Add this chunk's 2^(z s - ref) terms to the thread's running sum.  Scale and
// shift run two-wide (fma.f32x2), sums pairwise two-wide (add.f32x2), the
// exponentials on the special-function unit; one two-sum per chunk.
template <typename E>
__device__ __forceinline__ void stats_chunk(const uint4 (&raw)[kVecPerThread], float s,
                                            StatsState& st, float m) {
  // past-the-end vectors hold -inf: they raise no maximum and add 2^-inf = 0;
  // m is the maximum of the thread's elements
  const int r = exp_ref(m, s);
  if (r > st.ref) {  // exact rescale of the running sum by 2^(old - new)
    st.acc.scale(pow2i_f(st.ref - r));
    st.ref = r;
  }
  const float nref = -(float)st.ref;
  const unsigned long long s2 = f2pack(s, s), n2 = f2pack(nref, nref);
  constexpr int kP = E::kEPV / 2;
  unsigned long long vs[kVecPerThread];
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) {
    unsigned long long pr[kP];
    vec_pairs<E>(raw[q], pr);
#pragma unroll
    for (int h = 0; h < kP; ++h) {
      float x0, x1;
      f2unpack(fma2(pr[h], s2, n2), x0, x1);
      pr[h] = f2pack(ex2(x0), ex2(x1));
    }
#pragma unroll
    for (int w = kP / 2; w > 0; w >>= 1)
#pragma unroll
      for (int h = 0; h < w; ++h) pr[h] = add2(pr[h], pr[h + w]);
    vs[q] = pr[0];
  }
  float a0, a1;
  f2unpack(add2(add2(vs[0], vs[1]), add2(vs[2], vs[3])), a0, a1);
  st.acc.add(__fadd_rn(a0, a1));
}

template <typename E>
__device__ __forceinline__ void stats_chunk(const uint4 (&raw)[kVecPerThread], float s,
                                            StatsState& st) {
  stats_chunk<E>(raw, s, st, vec4_max<E>(raw));
}

struct ArgState {
  float v = -INFINITY;
  int i = 0x7FFFFFFF;
};

// The thread's running (max, lowest index) over its elements; the index is
// searched only when this chunk raises the thread's maximum.
template <typename E>
__device__ __forceinline__ void argmax_chunk(const uint4 (&raw)[kVecPerThread], int j0,
                                             ArgState& st) {
  const float m = vec4_max<E>(raw);
  if (m > st.v) {
    int idx = 0x7FFFFFFF;
#pragma unroll
    for (int q = kVecPerThread - 1; q >= 0; --q)
#pragma unroll
      for (int e = E::kEPV - 1; e >= 0; --e)
        if (E::elem(raw[q], e) == m) idx = j0 + (q * kThreads + (int)threadIdx.x) * E::kEPV + e;
    st.v = m;
    st.i = idx;
  }
}

// ---------------------------------------------------------------------------
// Segment records: per-warp partials combined by the last warp to arrive
// ---------------------------------------------------------------------------
// Four slots per CTA: in the streaming loop no warp runs more than kStages
// (= 3) items ahead of the slowest, so at most four segments are open at once.
constexpr int kSegSlots = 4;
struct StatsSlot {
  int ref;
  float hi, lo;
  int pad;
};
struct ArgSlot {
  float val;
  int idx;
};
struct SegSlots {
  int cnt[kSegSlots];
  StatsSlot st[kSegSlots][kWarps];
  ArgSlot am[kSegSlots][kWarps];
};

__device__ __forceinline__ void seg_slots_init(SegSlots& ss) {
  if (threadIdx.x < kSegSlots) ss.cnt[threadIdx.x] = 0;
}

// Park this warp's partial in `slot`; returns (to the whole warp) whether it
// arrived last, in which case the other warps' partials are visible to it.
__device__ __forceinline__ bool seg_arrive(SegSlots& ss, int slot) {
  const int lane = threadIdx.x & 31;
  int last = 0;
  if (lane == 0) {
    __threadfence_block();
    last = atomicAdd(&ss.cnt[slot], 1) == kWarps - 1;
    if (last) {
      __threadfence_block();
      ss.cnt[slot] = 0;  // no warp can reach this slot's next use yet
    }
  }
  return __shfl_sync(0xffffffffu, last, 0) != 0;
}

__device__ __forceinline__ void emit_stats_seg(const SampleParams& p, const StatsState& st,
                                               int row, int c_first, int c_last, SegSlots& ss,
                                               int& seg) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slot = seg++ & (kSegSlots - 1);
  const int wref = warp_max_i(st.ref);
  FSum mine = st.acc;
  mine.scale(pow2i_f(st.ref - wref));
  const FSum wsum = warp_sum_df(mine);
  if (lane == 0) ss.st[slot][warp] = StatsSlot{wref, wsum.hi, wsum.lo, 0};
  if (!seg_arrive(ss, slot)) return;
  StatsSlot v = lane < kWarps ? ss.st[slot][lane] : StatsSlot{kRefEmpty, 0.0f, 0.0f, 0};
  const int R = warp_max_i(v.ref);
  FSum f;
  f.hi = v.hi;
  f.lo = v.lo;
  f.scale(pow2i_f(v.ref - R));
  const FSum tot = warp_sum_df(f);
  const int n = c_last - c_first + 1;
  for (int i = lane; i < n; i += 32) {
    SoftmaxPartial sp;
    sp.ref = R;
    sp.nch = i == 0 ? n : 0;
    sp.hi = i == 0 ? tot.hi : 0.0f;
    sp.lo = i == 0 ? tot.lo : 0.0f;
    p.part[(size_t)row * p.nchunks + c_first + i] = sp;
  }
}

__device__ __forceinline__ void emit_arg_seg(const ArgmaxParams& p, const ArgState& st, int row,
                                             int c_first, int c_last, SegSlots& ss, int& seg) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slot = seg++ & (kSegSlots - 1);
  float v = st.v;
  int i = st.i;
  warp_argmax(v, i);
  if (lane == 0) ss.am[slot][warp] = ArgSlot{v, i};
  if (!seg_arrive(ss, slot)) return;
  ArgSlot a = lane < kWarps ? ss.am[slot][lane] : ArgSlot{-INFINITY, 0x7FFFFFFF};
  warp_argmax(a.val, a.idx);
  const int n = c_last - c_first + 1;
  for (int t = lane; t < n; t += 32) {
    ArgPartial ap;
    ap.val = a.val;
    ap.idx = a.idx;
    ap.nch = t == 0 ? n : 0;
    ap.pad = 0;
    p.part[(size_t)row * p.nchunks + c_first + t] = ap;
  }
}

// ---------------------------------------------------------------------------
// Row and sequence finalisation (one warp per row / sequence / tree)
// ---------------------------------------------------------------------------
// p = 2^x / S for x <= 1 and S >= 1/2, as a float mantissa 2^frac(x) / S
// and the exact power of two 2^floor(x), so probabilities far below the float
// range keep their value; zero (pe below -1022, as in float64) for x = -inf.
__device__ __forceinline__ void exp2_over(float x, float S, float* pm, int* pe) {
  const float n = floorf(x);
  *pe = n < -2000.0f ? -2000 : (int)n;
  *pm = __fdiv_rn(ex2(__fsub_rn(x, n)), S);
}

// The row's token probability rounded to float (the call's p and q outputs).
__device__ __forceinline__ float prob_float(const RowStats& r) {
  return r.pe < -1022 ? 0.0f : ldexpf(r.pm, r.pe);
}

// The accept test u q < p with p = pm 2^pe, q = qm 2^qe, decided exactly as
// float64 arithmetic decides it (u qm has at most 48 significant bits, so
// the float64 product is exact).  u qm is formed exactly as a float pair
// (product and fma remainder) and compared with pm 2^(pe - qe); uniforms
// below 2^-60 or exponent gaps beyond 60 take the float64 product.
__device__ __forceinline__ bool accept_test(float u, float pm, int pe, float qm, int qe) {
  if (pe < -1022) return false;  // u q < 0 never holds
  if (qe < -1022 || u == 0.0f) return true;
  const int e = pe - qe;
  if (u >= 0x1p-60f && e >= -60 && e <= 60) {
    const float a = __fmul_rn(u, qm);
    const float r = __fmaf_rn(u, qm, -a);
    const float t = __fmul_rn(pm, __int_as_float((e + 127) << 23));
    return a < t || (a == t && r < 0.0f);
  }
  return (double)u * ((double)qm * pow2i_d(qe)) < (double)pm * pow2i_d(pe);
}

// Merge one row's segment records (one warp).  Loads are issued four per
// lane before use, so a row of up to 128 records costs one round trip.  The
// token's logit was captured by the statistics kernel (p.zx); `tok`, when
// given, holds the sequence's draft tokens (prefetched).
template <typename E>
__device__ void finalize_stats_row(const SampleParams& p, int row, RowStats* out,
                                   const int* tok = nullptr) {
  const int lane = threadIdx.x & 31;
  const int rows_per_seq = 2 * p.k + 1;
  const int b = row / rows_per_seq, r = row - b * rows_per_seq;
  const SoftmaxPartial* pr = p.part + (size_t)row * p.nrec;
  const int nrec = p.nrec;
  float zx = 0.0f;
  int x = -1;
  if (r != p.k && lane == 0) {  // rows with a draft token: target r < k, draft r > k
    const int i = (r < p.k) ? r : r - p.k - 1;
    x = tok ? tok[i] : p.tokens[(size_t)b * p.k + i];
    zx = __ldcg(p.zx + row);
  }
  // one pass: running (reference, double-float sum), rescaled exactly when
  // a record's reference is larger
  int lref = kRefEmpty;
  FSum acc = FSum::zero();
  for (int base = lane; base < nrec; base += 128) {
    int4 rec[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      rec[u] = (base + 32 * u < nrec) ? __ldcg(reinterpret_cast<const int4*>(pr + base + 32 * u))
                                      : make_int4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (rec[u].y > 0) {
        if (rec[u].x > lref) {
          acc.scale(pow2i_f(lref - rec[u].x));
          lref = rec[u].x;
        }
        FSum v;
        v.hi = __int_as_float(rec[u].z);
        v.lo = __int_as_float(rec[u].w);
        v.scale(pow2i_f(rec[u].x - lref));
        acc = df_add(acc, v);
      }
    }
  }
  // butterfly over the lanes that hold records: the larger reference, and
  // the other partial rescaled to it exactly (powers of two), at each step
  const int width = nrec >= 32 ? 32 : (nrec <= 1 ? 1 : 1 << (32 - __clz(nrec - 1)));
  for (int o = width >> 1; o > 0; o >>= 1) {
    const int r2 = __shfl_xor_sync(0xffffffffu, lref, o);
    FSum y;
    y.hi = __shfl_xor_sync(0xffffffffu, acc.hi, o);
    y.lo = __shfl_xor_sync(0xffffffffu, acc.lo, o);
    const int m = max(lref, r2);
    acc.scale(pow2i_f(lref - m));
    y.scale(pow2i_f(r2 - m));
    acc = df_add(acc, y);
    lref = m;
  }
  const int R = lref;
  const FSum S = df_norm(acc);
  if (lane == 0) {
    RowStats rs;
    rs.ref = R;
    rs.inv_sum = __frcp_rn(S.hi);
    rs.pm = 0.0f;
    rs.pe = -2000;  // probability zero
    if (r != p.k) {
      if (x >= 0 && x < p.V)
        exp2_over(__fmaf_rn(zx, p.scale, -(float)R), S.hi, &rs.pm, &rs.pe);
      else
        set_flag(p.flags, kFlagTokenRange);
    }
    *out = rs;
  }
}

// Accept test left to right and first rejection of sequence b (one warp),
// from the sequence's merged rows `rs` (index r of rows_per_seq).  Returns the
// draw descriptor; with `write`, also stores the call's outputs for b (all
// but the drawn token) and the descriptor.  `ua` and `tok`, when given, hold
// the sequence's uniforms and draft tokens (prefetched).
template <typename RowFn>
__device__ DrawDesc resolve_sample_seq(const SampleParams& p, int b, RowFn rs, bool write,
                                       const float* ua = nullptr, const int* tok = nullptr) {
  if (!ua) ua = p.u_accept + (size_t)b * p.k;
  if (!tok) tok = p.tokens + (size_t)b * p.k;
  const int lane = threadIdx.x & 31;
  const int k = p.k;
  int n = k;
  for (int i0 = 0; i0 < k; i0 += 32) {
    const int i = i0 + lane;
    bool rej = false;
    if (i < k) {
      const RowStats ri = rs(i), rq = rs(k + 1 + i);
      if (write) {
        p.p_out[(size_t)b * k + i] = prob_float(ri);
        p.q_out[(size_t)b * k + i] = prob_float(rq);
      }
      rej = !accept_test(ua[i], ri.pm, ri.pe, rq.pm, rq.pe);
    }
    const unsigned m = __ballot_sync(0xffffffffu, rej);
    if (n == k && m) n = i0 + __ffs(m) - 1;
  }
  DrawDesc d;
  const RowStats rt = rs(n);
  d.n = n;
  d.nref_t = -(float)rt.ref;
  d.inv_t = rt.inv_sum;
  d.nref_d = 0.0f;
  d.inv_d = 0.0f;
  if (n < k) {
    const RowStats rd = rs(k + 1 + n);
    d.nref_d = -(float)rd.ref;
    d.inv_d = rd.inv_sum;
  }
  d.pad[0] = d.pad[1] = d.pad[2] = 0;
  if (write) {
    for (int i = lane; i <= k; i += 32)
      p.out_tokens[(size_t)b * (k + 1) + i] = (i < n) ? tok[i] : -1;
    if (lane == 0) {
      p.accepted_len[b] = n;
      p.desc[b] = d;
    }
  }
  return d;
}

// Merge the argmax records of rows r0, r0+stride, r0+2*stride, r0+3*stride
// of sequence b (one warp; rows past `nrows` are skipped).  All loads of a
// pass (T records per lane and row) are issued before any is used.  Returns
// the lane-uniform argmaxes.
template <int T>
__device__ void finalize_arg_rows4(const ArgmaxParams& p, int b, int r0, int stride, int nrows,
                                   int (&g)[4]) {
  const int lane = threadIdx.x & 31;
  const int nrec = p.nchunks;
  float v[4];
  int i[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    v[u] = -INFINITY;
    i[u] = 0x7FFFFFFF;
  }
  for (int base = lane; base < nrec; base += 32 * T) {
    int4 rec[4][T];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = r0 + u * stride;
      const ArgPartial* pr = p.part + ((size_t)b * p.rows_per_seq + r) * nrec;
#pragma unroll
      for (int t = 0; t < T; ++t)
        rec[u][t] = (r < nrows && base + 32 * t < nrec)
                        ? __ldcg(reinterpret_cast<const int4*>(pr + base + 32 * t))
                        : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int t = 0; t < T; ++t)
        if (rec[u][t].z > 0 && better(__int_as_float(rec[u][t].x), rec[u][t].y, v[u], i[u])) {
          v[u] = __int_as_float(rec[u][t].x);
          i[u] = rec[u][t].y;
        }
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    warp_argmax(v[u], i[u]);
    g[u] = (i[u] >= 0 && i[u] < p.V) ? i[u] : 0;
    const int r = r0 + u * stride;
    if (lane == 0 && r < nrows) p.rowarg[(size_t)b * p.rows_per_seq + r] = g[u];
  }
}

// Chain resolve: accept while the draft equals the target argmax (one warp),
// from the sequence's draft tokens `tok` [k] and row argmaxes `g` [k+1]
// (shared memory).
__device__ void resolve_chain(const ArgmaxParams& p, int b, const int32_t* tok, const int32_t* g) {
  const int lane = threadIdx.x & 31;
  const int k = p.rows_per_seq - 1;
  int n = k;
  bool bad = false;
  for (int i0 = 0; i0 < k; i0 += 32) {
    const int i = i0 + lane;
    bool miss = false;
    if (i < k) {
      const int x = tok[i];
      bad |= (x < 0 || x >= p.V);
      miss = x != g[i];
    }
    const unsigned m = __ballot_sync(0xffffffffu, miss);
    if (n == k && m) n = i0 + __ffs(m) - 1;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_flag(p.flags, kFlagTokenRange);
  for (int i = lane; i <= k; i += 32) {
    int v = -1;
    if (i < n) v = tok[i];
    else if (i == n) v = g[n];
    p.out_tokens[(size_t)b * (k + 1) + i] = v;
  }
  if (lane == 0) p.accepted_len[b] = n;
}

// Tree resolve (one warp): every node walks to the root (at most max_depth + 1
// hops); a warp max over (depth, -node) picks the deepest accepted node with
// the lowest index.
__device__ void resolve_tree(const ArgmaxParams& p, int b, const int32_t* par,
                             const int32_t* tok, const int32_t* g) {
  const int lane = threadIdx.x & 31;
  const int N = p.rows_per_seq;
  const int W = p.max_depth + 1;
  unsigned long long best = 0xFFFFFFFFull;  // the root: depth 0, node 0
  unsigned bad = 0;
  for (int v = 1 + lane; v < N; v += 32) {
    int cur = v, d = 0;
    bool ok = true;
    while (cur != 0) {
      const int pa = par[cur];
      if (pa < 0 || pa >= cur) {
        bad |= kFlagBadParent;
        ok = false;
        break;
      }
      const int tv = tok[cur];
      if (tv < 0 || tv >= p.V) bad |= kFlagTokenRange;
      if (tv != g[pa]) ok = false;
      if (++d > p.max_depth) {
        bad |= kFlagDepth;
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
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
    best = y > best ? y : best;
  }
  const int depth = (int)(best >> 32);
  const int vstar = (int)(0xFFFFFFFFu - (unsigned)(best & 0xFFFFFFFFull));
  for (int i = depth + 1 + lane; i < W; i += 32) {
    p.path_nodes[(size_t)b * W + i] = -1;
    p.out_tokens[(size_t)b * W + i] = -1;
  }
  if (lane == 0) {
    p.accepted_len[b] = depth;
    int cur = vstar;
    for (int i = depth; i >= 0; --i) {
      p.path_nodes[(size_t)b * W + i] = cur;
      if (i >= 1) p.out_tokens[(size_t)b * W + i - 1] = tok[cur];
      cur = (i >= 1) ? par[cur] : 0;
    }
    p.out_tokens[(size_t)b * W + depth] = g[vstar];
  }
}

// ---------------------------------------------------------------------------
// Resolve kernels (launched after the streaming kernel, programmatic
// dependent launch): one CTA per sequence or tree merges its rows' records,
// one warp per row, then one warp resolves the sequence.  No atomics.
// ---------------------------------------------------------------------------
// Trees up to this many nodes are walked on shared-memory copies of their
// parents, tokens and row argmaxes; larger ones read global memory.
constexpr int kTreeSmemNodes = 2048;

// Load what the resolve needs of sequence (tree) b besides the argmax kernel's
// records: the draft tokens of a chain, or the parents and tokens of a tree
// of up to kTreeSmemNodes nodes (whole CTA, before the dependency wait: the
// argmax kernel does not write them).
__device__ void resolve_prefetch(const ArgmaxParams& p, int b, int32_t* s_par, int32_t* s_tok) {
  const int N = p.rows_per_seq;
  if (!p.tree) {
    for (int i = threadIdx.x; i < N - 1; i += blockDim.x)
      s_tok[i] = p.tokens[(size_t)b * (N - 1) + i];
  } else if (N <= kTreeSmemNodes) {
    for (int v = threadIdx.x; v < N; v += blockDim.x) {
      s_par[v] = p.parents[(size_t)b * N + v];
      s_tok[v] = p.tokens[(size_t)b * N + v];
    }
  }
}

// Merge the rows of sequence (tree) b and resolve it (whole CTA; the three
// scratch arrays hold kTreeSmemNodes entries each, in shared memory, with the
// prefetched inputs).  T: records per lane and row loaded at once.
template <int T>
__device__ void resolve_sequence(const ArgmaxParams& p, int b, int32_t* s_par, int32_t* s_tok,
                                 int32_t* s_g) {
  const int N = p.rows_per_seq;
  const bool in_smem = !p.tree || N <= kTreeSmemNodes;
  for (int r0 = threadIdx.x >> 5; r0 < N; r0 += 4 * kWarps) {
    int g[4];
    finalize_arg_rows4<T>(p, b, r0, kWarps, N, g);
    if (in_smem && (threadIdx.x & 31) == 0)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (r0 + u * kWarps < N) s_g[r0 + u * kWarps] = g[u];
  }
  __threadfence_block();
  __syncthreads();
  if (threadIdx.x < 32) {
    if (!p.tree)
      resolve_chain(p, b, s_tok, s_g);
    else if (in_smem)
      resolve_tree(p, b, s_par, s_tok, s_g);
    else
      resolve_tree(p, b, p.parents + (size_t)b * N, p.tokens + (size_t)b * N,
                   p.rowarg + (size_t)b * N);
  }
}

__global__ void __launch_bounds__(kThreads) argmax_resolve_kernel(const ArgmaxParams p) {
  __shared__ int32_t s_par[kTreeSmemNodes], s_tok[kTreeSmemNodes], s_g[kTreeSmemNodes];
  resolve_prefetch(p, blockIdx.x, s_par, s_tok);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next call's streaming kernel may become resident now; it waits for
  // this grid before touching memory
  asm volatile("griddepcontrol.launch_dependents;");
  __syncthreads();  // the prefetched inputs
  resolve_sequence<4>(p, blockIdx.x, s_par, s_tok, s_g);
}

// ---------------------------------------------------------------------------
// Loader 1: persistent CTAs streaming chunk ranges through bulk async copies
// ---------------------------------------------------------------------------
// CTA g owns a contiguous range of items (item = row * nchunks + chunk; item_range).
// Thread 0 keeps kStages chunk copies in flight.  A slot is released (its
// "empty" barrier, one arrival per warp) as soon as every warp has copied it
// into registers, and thread 0 refills it with the item kStages ahead: before
// its own work on the item in the statistics kernel (heavy arithmetic), after
// it in the argmax and growth kernels.
// The loop has no CTA-wide barrier.  Every wait is bounded: a wait that runs
// out sets kFlagTimeout, the CTA keeps its control flow but stops copying and
// computing, and it drains the copies still in flight before it exits.
struct Ring {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort;
};

// CTA g's items.  CTAs start in index order (the second CTA of each SM a few
// microseconds after the first), and in a short range that start decides
// when the CTA ends: there the items left over by an even split go to the
// first CTAs.  In long ranges they are spread evenly (front-loading measured
// 2.5% slower on 67-item ranges).
constexpr int kFrontLoadItems = 48;  // ranges shorter than this: remainder first
__device__ __forceinline__ void item_range(int items, int& i0, int& i1) {
  const int G = gridDim.x, g = blockIdx.x;
  const int q = items / G, rem = items - q * G;
  if (q < kFrontLoadItems) {
    i0 = g * q + min(g, rem);
    i1 = i0 + q + (g < rem ? 1 : 0);
  } else {
    i0 = (int)((long long)items * g / G);
    i1 = (int)((long long)items * (g + 1) / G);
  }
}

// Thread 0 initialises the barriers and issues the first kStages copies
// before the CTA barrier, so the first bytes are in flight at once.
template <typename IssueFn>
__device__ __forceinline__ int ring_init(Ring& ring, int i0, int i1, IssueFn issue) {
  int issued = i0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ring.full[s], 1);
      mbar_init(&ring.empty[s], kWarps);
    }
    ring.abort = 0;
    mbar_init_fence();
    for (; issued < i1 && issued < i0 + kStages; ++issued) issue(issued, issued - i0);
  }
  __syncthreads();
  return issued;
}

// Thread 0, at the end: wait (bounded, with the default limit whatever the
// limit of the loop's waits) for the copies issued into each slot.  A slot
// is reissued only after its previous copy landed (ring_take), so only the
// last kStages issued copies can be in flight.
__device__ __noinline__ void ring_drain(Ring& ring, int i0, int issued) {
  for (int j = max(i0, issued - kStages); j < issued; ++j)
    mbar_wait_bounded(&ring.full[(j - i0) % kStages], (unsigned)(((j - i0) / kStages) & 1));
}

// Wait for the item in `slot` (phase parity `par`), copy this thread's
// vectors to registers (past-the-end vectors read as -inf) and release the
// slot.  A warp releases the slot only when its lane 0 has seen the copy
// land, so a slot is never reissued while its previous copy may still be in
// flight (a warp that gives up, or finds the CTA aborted, does not release
// it).  Returns false once the CTA has aborted.
template <typename E>
__device__ __forceinline__ bool ring_take(Ring& ring, const uint8_t* stage_mem, int slot,
                                          unsigned par, int nvec, unsigned* flags,
                                          uint4 (&raw)[kVecPerThread],
                                          uint64_t limit_ns = kWaitLimitNs) {
  bool ok = *(volatile int*)&ring.abort == 0;
  if (ok && !mbar_wait_bounded(&ring.full[slot], par, limit_ns)) {
    ok = false;
    ring.abort = 1;
    set_flag(flags, kFlagTimeout);
  }
  const uint8_t* sm = stage_mem + (size_t)slot * kChunkBytes + threadIdx.x * 16;
  const uint4 ninf = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) {
    const int vi = q * kThreads + (int)threadIdx.x;
    raw[q] = (ok && vi < nvec) ? lds128(sm + q * kThreads * 16) : ninf;
  }
  __syncwarp();
  if ((threadIdx.x & 31) == 0 && ok) mbar_arrive(&ring.empty[slot]);
  return ok;
}

// Thread 0: once every warp has released `slot` (phase parity `par`), reuse
// it for item `nxt` (if any).  Returns the new count of issued items.  Every
// release follows the landing of the slot's previous copy (ring_take), so a
// completed wait makes the reissue safe even if the CTA has aborted since;
// after an abort the missing releases let the wait run out instead.
template <typename IssueFn>
__device__ __forceinline__ int ring_refill(Ring& ring, int slot, unsigned par, int nxt, int i1,
                                           int issued, unsigned* flags, IssueFn issue,
                                           uint64_t limit_ns = kWaitLimitNs) {
  if (nxt >= i1 || *(volatile int*)&ring.abort) return issued;
  if (!mbar_wait_bounded(&ring.empty[slot], par, limit_ns)) {
    ring.abort = 1;
    set_flag(flags, kFlagTimeout);
    return issued;
  }
  issue(nxt, slot);
  return nxt + 1;
}

// kEarly (chosen by the host for short per-CTA ranges): the kernel reads
// only its inputs (logits, draft tokens) before its first write and waits
// for the preceding grid there (a segment record, or a captured logit kept
// in a register until then), so its copies start while the call before it
// is finishing.  The inputs must therefore not be written by the call
// before it on the stream (no call of this library writes a caller's
// inputs; a caller's kernel never triggers early).  In long ranges the
// early copies only compete with the previous call's finish for bandwidth
// (B=256, k=7: 243.8 -> 248.9 us), and the kernel waits before anything, as
// every first kernel of a call otherwise does.
template <typename E, bool kEarly>
__global__ void __launch_bounds__(kThreads, 2) stream_stats_kernel(const SampleParams p) {
  extern __shared__ __align__(128) uint8_t stage_mem[];
  __shared__ Ring ring;
  __shared__ SegSlots ss;
  using S = typename E::storage;

  // launched as a programmatic dependent of whatever kernel precedes it in
  // the stream (see kEarly above for when it waits for that grid)
  if constexpr (!kEarly) asm volatile("griddepcontrol.wait;" ::: "memory");
  int i0, i1;
  item_range(p.items, i0, i1);
  // the dependent draw kernel may begin launching; it waits for this grid
  asm volatile("griddepcontrol.launch_dependents;");
  if (i0 >= i1) {
    if constexpr (kEarly) asm volatile("griddepcontrol.wait;" ::: "memory");
    return;
  }
  const int C = p.nchunks;
  const int rows_per_seq = 2 * p.k + 1;
  bool waited = false;  // kEarly: the preceding grid has finished
  int pend_row = -1;    // kEarly: a captured token logit not yet stored
  float pend_z = 0.0f;
  auto wait_prior = [&]() {  // kEarly, before this grid's first write
    if (waited) return;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    waited = true;
    if (pend_row >= 0) p.zx[pend_row] = pend_z;
    pend_row = -1;
  };

  const uint64_t pol_keep = l2_policy_keep(), pol_stream = l2_policy_stream();
  // thread 0 issues the range's items in order (ring_init, then one refill
  // per item), so the next one's sequence, row and chunk are counted along
  int nb = (i0 / C) / rows_per_seq, nr = i0 / C - nb * rows_per_seq, nc = i0 % C;
  auto issue = [&](int /*item: the next in order*/, int slot) {
    const int b = nb, r = nr, c = nc;
    if (++nc == C) {
      nc = 0;
      if (++nr == rows_per_seq) {
        nr = 0;
        ++nb;
      }
    }
    const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
    const unsigned bytes = (unsigned)(j1 - j0) * (unsigned)sizeof(S);
    const int pos = r <= p.k ? r : r - p.k - 1;  // draft position of the row
    mbar_expect_tx(&ring.full[slot], bytes);
    bulk_g2s_hint(stage_mem + (size_t)slot * kChunkBytes, seq_row_ptr<E>(p, b, r) + j0, bytes,
                  &ring.full[slot], pos < p.keep_pos ? pol_keep : pol_stream);
  };

  seg_slots_init(ss);
  int issued = ring_init(ring, i0, i1, issue);

  StatsState st;
  int seg = 0;
  int row = i0 / C, c = i0 - row * C, c_first = c;
  int slot = 0;
  unsigned par = 0;
  // draft tokens of the current row and the next (loaded one row ahead)
  int tok = row_token(p, row), tok_next = row_token(p, row + 1);
  for (int it = i0; it < i1; ++it) {
    const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
    uint4 raw[kVecPerThread];
    const bool ok =
        ring_take<E>(ring, stage_mem, slot, par, (j1 - j0) / E::kEPV, p.flags, raw, p.wait_ns);
    // the refill before this thread's (heavy) work on the item, so the copy
    // three items ahead goes out at once (after the work: 0.5-6 us slower)
    if (threadIdx.x == 0)
      issued = ring_refill(ring, slot, par, it + kStages, i1, issued, p.flags, issue, p.wait_ns);
    if (ok) {
      stats_chunk<E>(raw, p.scale, st);
      if constexpr (kEarly) {
        float z;
        if (capture_token_value<E>(raw, tok, j0, j1, z)) {
          if (!waited && pend_row >= 0) wait_prior();  // a second capture: store the first
          if (waited) {
            p.zx[row] = z;
          } else {
            pend_row = row;
            pend_z = z;
          }
        }
      } else {
        capture_token<E>(p, raw, tok, j0, j1, row);
      }
    }
    const bool row_end = (c + 1 == C);
    if (row_end || it + 1 == i1) {
      if constexpr (kEarly) wait_prior();
      emit_stats_seg(p, st, row, c_first, c, ss, seg);
      st = StatsState();
      c_first = 0;
    }
    if (row_end) {
      c = 0;
      ++row;
      tok = tok_next;
      tok_next = row_token(p, row + 1);
    } else {
      ++c;
    }
    if (++slot == kStages) {
      slot = 0;
      par ^= 1u;
    }
  }
  if (threadIdx.x == 0) ring_drain(ring, i0, issued);
}

template <typename E>
__global__ void __launch_bounds__(kThreads, 2) stream_argmax_kernel(const ArgmaxParams p) {
  extern __shared__ __align__(128) uint8_t stage_mem[];
  __shared__ Ring ring;
  __shared__ SegSlots ss;
  using S = typename E::storage;

  // launched as a programmatic dependent of whatever kernel precedes it in
  // the stream.  It reads only the logits before its first write (a segment
  // record), and waits for that grid only there: so its copies start while
  // the call before it is finishing.  The logits must therefore not be
  // written by the call before it on the stream (no call of this library
  // writes a caller's logits; a caller's kernel never triggers early, so it
  // has finished before this one starts).
  int i0, i1;
  item_range(p.items, i0, i1);
  asm volatile("griddepcontrol.launch_dependents;");
  if (i0 >= i1) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    return;
  }
  const int C = p.nchunks;
  bool waited = false;

  // (the item's row and chunk by division: counting them along, as the
  // statistics kernel does, measured 0.2-0.6 us slower here)
  auto issue = [&](int item, int slot) {
    const int row = item / C, c = item - (item / C) * C;
    const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
    const unsigned bytes = (unsigned)(j1 - j0) * (unsigned)sizeof(S);
    mbar_expect_tx(&ring.full[slot], bytes);
    bulk_g2s(stage_mem + (size_t)slot * kChunkBytes,
             reinterpret_cast<const S*>(p.target) + (size_t)row * p.V + j0, bytes,
             &ring.full[slot]);
  };

  seg_slots_init(ss);
  int issued = ring_init(ring, i0, i1, issue);

  ArgState st;
  int seg = 0;
  int row = i0 / C, c = i0 - row * C, c_first = c;
  int slot = 0;
  unsigned par = 0;
  for (int it = i0; it < i1; ++it) {
    const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
    uint4 raw[kVecPerThread];
    const bool ok =
        ring_take<E>(ring, stage_mem, slot, par, (j1 - j0) / E::kEPV, p.flags, raw, p.wait_ns);
    if (ok) argmax_chunk<E>(raw, j0, st);
    // the refill after this thread's own (light) work on the item: by then
    // the other warps have usually released the slot, so warp 0 is not held
    // (before the work, as in the statistics kernel, measured 0.2-2 us slower)
    if (threadIdx.x == 0)
      issued = ring_refill(ring, slot, par, it + kStages, i1, issued, p.flags, issue, p.wait_ns);
    const bool row_end = (c + 1 == C);
    if (row_end || it + 1 == i1) {
      if (!waited) {  // the first write of this grid: the grid before it has finished
        asm volatile("griddepcontrol.wait;" ::: "memory");
        waited = true;
      }
      emit_arg_seg(p, st, row, c_first, c, ss, seg);
      st = ArgState();
      c_first = 0;
    }
    if (row_end) {
      c = 0;
      ++row;
    } else {
      ++c;
    }
    if (++slot == kStages) {
      slot = 0;
      par ^= 1u;
    }
  }
  if (threadIdx.x == 0) ring_drain(ring, i0, issued);
}

// ---------------------------------------------------------------------------
// Loader 2: one CTA per chunk with plain loads (any row size)
// ---------------------------------------------------------------------------
template <typename E, bool kVec>
__device__ __forceinline__ void load_chunk_regs(const typename E::storage* row, int j0, int j1,
                                                uint4 (&raw)[kVecPerThread]) {
  const int nvec = (j1 - j0 + E::kEPV - 1) / E::kEPV;
  const uint4 ninf = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) {
    const int vi = q * kThreads + (int)threadIdx.x;
    raw[q] = vi < nvec ? fetch_vec<E, kVec>(row, j0 + vi * E::kEPV, j1) : ninf;
  }
}

template <typename E, bool kVec>
__global__ void __launch_bounds__(kThreads) chunk_stats_kernel(const SampleParams p) {
  __shared__ SegSlots ss;
  seg_slots_init(ss);
  __syncthreads();
  int seg = 0;
  const int rows_per_seq = 2 * p.k + 1;
  const int item = blockIdx.x;
  const int row = item / p.nchunks, c = item - row * p.nchunks;
  const int b = row / rows_per_seq, r = row - b * rows_per_seq;
  const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
  uint4 raw[kVecPerThread];
  load_chunk_regs<E, kVec>(seq_row_ptr<E>(p, b, r), j0, j1, raw);
  const int tok = row_token(p, row);
  asm volatile("griddepcontrol.launch_dependents;");
  StatsState st;
  stats_chunk<E>(raw, p.scale, st);
  capture_token<E>(p, raw, tok, j0, j1, row);
  emit_stats_seg(p, st, row, c, c, ss, seg);
}

template <typename E, bool kVec>
__global__ void __launch_bounds__(kThreads) chunk_argmax_kernel(const ArgmaxParams p) {
  __shared__ SegSlots ss;
  seg_slots_init(ss);
  __syncthreads();
  int seg = 0;
  asm volatile("griddepcontrol.launch_dependents;");
  const int item = blockIdx.x;
  const int row = item / p.nchunks, c = item - row * p.nchunks;
  const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
  uint4 raw[kVecPerThread];
  load_chunk_regs<E, kVec>(
      reinterpret_cast<const typename E::storage*>(p.target) + (size_t)row * p.V, j0, j1, raw);
  ArgState st;
  argmax_chunk<E>(raw, j0, st);
  emit_arg_seg(p, st, row, c, c, ss, seg);
}

// ---------------------------------------------------------------------------
// Draw: residual / bonus inverse CDF
// ---------------------------------------------------------------------------
// Prefix structure of one chunk of draw weights, in vector (element) order:
//   group  g[vi]  sequential float sum of vector vi's weights (2048 groups)
//   quad   Q      double-float sum of groups 4Q..4Q+3 added to zero in order;
//                 quad Q belongs to thread Q of a 512-thread CTA
//   warp   w      inclusive double-float warp scan of quads 32w..32w+31
//   chunk         the 16 warp totals added in order
// draw_kernel builds it per chunk (group sums and chunk totals kept in the
// workspace); draw_resolve_kernel rebuilds the quad and warp levels of the
// chosen chunk with the same arithmetic and walks down to the token.
struct DrawRows {
  const void* t;  // target row
  const void* d;  // draft row (residual only)
  float nref_t, inv_t, nref_d, inv_d;
};

template <typename E>
__device__ __forceinline__ DrawRows draw_rows(const SampleParams& p, int b, const DrawDesc& d) {
  using S = typename E::storage;
  DrawRows w;
  if (p.drawn) {  // recomputed rows (fp32)
    w.t = p.drawn + (size_t)(2 * b) * p.V;
    w.d = d.n < p.k ? p.drawn + (size_t)(2 * b + 1) * p.V : nullptr;
  } else {
    w.t = reinterpret_cast<const S*>(p.target) + ((size_t)b * (p.k + 1) + d.n) * (size_t)p.V;
    w.d = d.n < p.k
              ? reinterpret_cast<const S*>(p.draft) + ((size_t)b * p.k + d.n) * (size_t)p.V
              : nullptr;
  }
  w.nref_t = d.nref_t;
  w.inv_t = d.inv_t;
  w.nref_d = d.nref_d;
  w.inv_d = d.inv_d;
  return w;
}

// p of one target element, and the residual max(0, p - q) with the draft
// element.  Element e of a vector takes 2^x on the FMA pipe when e <
// kDrawPoly, else on the special-function unit (this pass is bound by the
// latter); explicit round-to-nearest intrinsics keep every evaluation of an
// element bit-identical wherever it is computed.
constexpr int kDrawPoly = 2;
__device__ __forceinline__ float draw_exp2(float x, int e) {
  return e < kDrawPoly ? exp2_fma(x) : ex2(x);
}
__device__ __forceinline__ float draw_p(float zt, float s, const DrawRows& w, int e) {
  return __fmul_rn(draw_exp2(__fmaf_rn(zt, s, w.nref_t), e), w.inv_t);
}
__device__ __forceinline__ float draw_r(float pt, float zd, float s, const DrawRows& w, int e) {
  const float pd = __fmul_rn(draw_exp2(__fmaf_rn(zd, s, w.nref_d), e), w.inv_d);
  return fmaxf(__fsub_rn(pt, pd), 0.0f);
}
// Weight of element e: the residual after a rejection, else p.
__device__ __forceinline__ float draw_weight(float zt, float zd, float s, const DrawRows& w,
                                             bool resid, int e) {
  const float pt = draw_p(zt, s, w, e);
  return resid ? draw_r(pt, zd, s, w, e) : pt;
}

__device__ __forceinline__ FSum quad_sum(const float4& v) {
  FSum a = FSum::zero();
  a.add(v.x);
  a.add(v.y);
  a.add(v.z);
  a.add(v.w);
  return a;
}

// Quad scan of one chunk's group array held in shared memory (512 threads):
// every thread gets its quad's inclusive scan within its warp; warp totals go
// to s_w; thread 0 returns the chunk total (the warp totals added in order).
__device__ __forceinline__ FSum chunk_scan_cta(const float* s_g, FSum* s_w, FSum* my_inc,
                                               FSum* my_quad) {
  const FSum q = quad_sum(*reinterpret_cast<const float4*>(s_g + 4 * threadIdx.x));
  const FSum inc = warp_scan_df(q);
  if ((threadIdx.x & 31) == 31) s_w[threadIdx.x >> 5] = inc;
  *my_inc = inc;
  *my_quad = q;
  __syncthreads();
  FSum t = s_w[0];
  if (threadIdx.x == 0)
    for (int i = 1; i < kWarps; ++i) t = df_add(t, s_w[i]);
  return t;
}

// The sequences's rows are merged by every draw CTA of the sequence (one warp
// per row), into shared memory, followed by the accept test: the CTA of chunk
// 0 writes the outputs.  Limits: 2k+1 <= kMaxSeqRows.
constexpr int kMaxDraft = 256;  // draft positions per sequence (the C interface's limit)
constexpr int kMaxSeqRows = 2 * kMaxDraft + 1;

template <typename E, bool kVec>
__global__ void __launch_bounds__(kThreads) draw_kernel(const SampleParams p) {
  using St = typename E::storage;
  __shared__ __align__(16) float s_g[kVecPerChunk];
  __shared__ __align__(16) float s_gp[kVecPerChunk];
  __shared__ RowStats s_rows[kMaxSeqRows];
  __shared__ DrawDesc s_desc;
  __shared__ FSum s_w[kWarps];

  // wait for the statistics kernel's records (programmatic dependent launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  const int item = blockIdx.x;
  const int b = item / p.nchunks;
  const int c = item - b * p.nchunks;
  const int rows_per_seq = 2 * p.k + 1;
  for (int r = threadIdx.x >> 5; r < rows_per_seq; r += kWarps)
    finalize_stats_row<E>(p, b * rows_per_seq + r, &s_rows[r]);
  __syncthreads();
  if (threadIdx.x < 32) {
    const DrawDesc dd =
        resolve_sample_seq(p, b, [&](int r) { return s_rows[r]; }, c == 0);
    if (threadIdx.x == 0) s_desc = dd;
  }
  __syncthreads();
  const DrawDesc d = s_desc;
  const bool resid = d.n < p.k;
  const DrawRows w = draw_rows<E>(p, b, d);
  const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
  const int nvec = (j1 - j0 + E::kEPV - 1) / E::kEPV;
  const size_t gofs = (size_t)item * kVecPerChunk;

  uint4 vt[kVecPerThread], vd[kVecPerThread];
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) {
    const int vi = q * kThreads + (int)threadIdx.x;
    const int j = j0 + vi * E::kEPV;
    vt[q] = vi < nvec ? fetch_vec<E, kVec>(reinterpret_cast<const St*>(w.t), j, j1)
                      : make_uint4(0, 0, 0, 0);
    vd[q] = (resid && vi < nvec) ? fetch_vec<E, kVec>(reinterpret_cast<const St*>(w.d), j, j1)
                                 : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) {
    const int vi = q * kThreads + (int)threadIdx.x;
    float g = 0.0f, gp = 0.0f;
    if (vi < nvec) {
#pragma unroll
      for (int e = 0; e < E::kEPV; ++e) {
        const float pt = draw_p(E::elem(vt[q], e), p.scale, w, e);
        gp = __fadd_rn(gp, pt);
        g = __fadd_rn(g, resid ? draw_r(pt, E::elem(vd[q], e), p.scale, w, e) : pt);
      }
    }
    s_g[vi] = g;
    p.gsum[gofs + vi] = g;
    if (resid) {
      s_gp[vi] = gp;
      p.gsum_p[gofs + vi] = gp;
    }
  }
  __syncthreads();
  {
    FSum inc, q;
    const FSum t = chunk_scan_cta(s_g, s_w, &inc, &q);
    if (threadIdx.x == 0) p.csum[item] = t;
  }
  if (resid) {
    __syncthreads();
    FSum inc, q;
    const FSum t = chunk_scan_cta(s_gp, s_w, &inc, &q);
    if (threadIdx.x == 0) p.csum_p[item] = t;
  }
}

// Inclusive double-float scan of the chunk totals by one warp; with a target,
// also finds the first chunk whose inclusive prefix exceeds it (else the last
// chunk with positive mass) and that chunk's exclusive prefix.  Returns the
// (normalised) total.
__device__ __forceinline__ FSum chunk_prefix(const FSum* cs, int C, const FSum* target,
                                             int* cstar, FSum* base) {
  const int lane = threadIdx.x & 31;
  FSum carry = FSum::zero();
  int found = -1, lastpos = -1;
  FSum fbase = FSum::zero(), lbase = FSum::zero();
  for (int c0 = 0; c0 < C; c0 += 32) {
    const int c = c0 + lane;
    FSum v = FSum::zero();
    if (c < C) {
      const float2 t = __ldcg(reinterpret_cast<const float2*>(cs + c));
      v.hi = t.x;
      v.lo = t.y;
    }
    const FSum inc = df_norm(df_add(carry, warp_scan_df(v)));
    FSum excl;
    excl.hi = __shfl_up_sync(0xffffffffu, inc.hi, 1);
    excl.lo = __shfl_up_sync(0xffffffffu, inc.lo, 1);
    if (lane == 0) excl = carry;
    if (target) {
      const unsigned hit = __ballot_sync(0xffffffffu, c < C && df_less(*target, inc));
      if (found < 0 && hit) {
        const int L = __ffs(hit) - 1;
        found = c0 + L;
        fbase.hi = __shfl_sync(0xffffffffu, excl.hi, L);
        fbase.lo = __shfl_sync(0xffffffffu, excl.lo, L);
      }
      const unsigned pos = __ballot_sync(0xffffffffu, c < C && v.hi > 0.0f);
      if (pos) {
        const int L = 31 - __clz(pos);
        lastpos = c0 + L;
        lbase.hi = __shfl_sync(0xffffffffu, excl.hi, L);
        lbase.lo = __shfl_sync(0xffffffffu, excl.lo, L);
      }
    }
    carry.hi = __shfl_sync(0xffffffffu, inc.hi, 31);
    carry.lo = __shfl_sync(0xffffffffu, inc.lo, 31);
  }
  if (target) {
    if (found < 0) {
      found = lastpos < 0 ? 0 : lastpos;
      fbase = lastpos < 0 ? FSum::zero() : lbase;
    }
    *cstar = found;
    *base = fbase;
  }
  return carry;
}

// Walk one chunk's prefix structure down to the token (whole CTA; the chunk's
// group sums are in shared memory `s_g`, the target and the chunk's exclusive
// prefix `base` are known): warp block (16 warp totals), quad (lane of that
// warp), vector, element.  Where rounding leaves the target just past a
// level's end, the last position with positive weight is taken (such a target
// lies within ~1e-15 of a boundary).  Returns the token to every thread.
struct WalkScratch {
  FSum w[kWarps];
  int wb, exact, tok;
};

template <typename E, bool kVec>
__device__ int walk_chunk(const SampleParams& p, const DrawRows& w, bool resid, const float* s_g,
                          int cstar, const FSum& target, const FSum& base, WalkScratch& ws) {
  using St = typename E::storage;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  FSum inc, quad;
  chunk_scan_cta(s_g, ws.w, &inc, &quad);
  if (warp == 0) {
    const FSum wv = lane < kWarps ? ws.w[lane] : FSum::zero();
    const FSum winc = df_norm(df_add(base, warp_scan_df(wv)));
    const unsigned hit = __ballot_sync(0xffffffffu, lane < kWarps && df_less(target, winc));
    const unsigned pos = __ballot_sync(0xffffffffu, lane < kWarps && wv.hi > 0.0f);
    if (lane == 0) {
      ws.wb = hit ? (__ffs(hit) - 1) : (pos ? (31 - __clz(pos)) : 0);
      ws.exact = hit != 0;
      ws.tok = -1;
    }
  }
  __syncthreads();
  const int wb = ws.wb;
  const bool exact = ws.exact != 0;
  const int j0 = cstar * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
  if (warp == wb) {
    // exclusive prefix of this warp block: base + warp totals before it
    FSum wbase = base;
    for (int i = 0; i < wb; ++i) wbase = df_add(wbase, ws.w[i]);
    FSum exc;
    exc.hi = __shfl_up_sync(0xffffffffu, inc.hi, 1);
    exc.lo = __shfl_up_sync(0xffffffffu, inc.lo, 1);
    if (lane == 0) exc = FSum::zero();
    const unsigned hit =
        __ballot_sync(0xffffffffu, exact && df_less(target, df_norm(df_add(wbase, inc))));
    const unsigned pos = __ballot_sync(0xffffffffu, quad.hi > 0.0f);
    const int L = hit ? (__ffs(hit) - 1) : (pos ? (31 - __clz(pos)) : 0);
    if (lane == L) {
      const float4 g4 = *reinterpret_cast<const float4*>(s_g + 4 * threadIdx.x);
      const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
      FSum run = df_add(wbase, exc);
      int tok = -1, lastv = -1;
      for (int i = 0; i < 4 && tok < 0; ++i) {
        if (!(gv[i] > 0.0f)) continue;
        const int vi = 4 * threadIdx.x + i;  // vector index within the chunk
        lastv = vi;
        const FSum nxt = df_add(run, df_from(gv[i]));
        if (hit && df_less(target, df_norm(nxt))) {
          const int j = j0 + vi * E::kEPV;
          const uint4 vt = fetch_vec<E, kVec>(reinterpret_cast<const St*>(w.t), j, j1);
          const uint4 vd = resid ? fetch_vec<E, kVec>(reinterpret_cast<const St*>(w.d), j, j1)
                                 : make_uint4(0, 0, 0, 0);
          float part = 0.0f;
          int lastpos = -1;
#pragma unroll
          for (int e = 0; e < E::kEPV; ++e) {
            const float we = draw_weight(E::elem(vt, e), resid ? E::elem(vd, e) : 0.0f, p.scale,
                                         w, resid, e);
            part = __fadd_rn(part, we);
            if (we > 0.0f && j + e < j1) lastpos = j + e;
            if (tok < 0 && we > 0.0f && df_less(target, df_norm(df_add(run, df_from(part)))))
              tok = j + e;
          }
          if (tok < 0) tok = lastpos;  // rounding inside the vector
        }
        run = nxt;
      }
      if (tok < 0 && lastv >= 0) {  // rounding: last positive element of the quad
        const int j = j0 + lastv * E::kEPV;
        const uint4 vt = fetch_vec<E, kVec>(reinterpret_cast<const St*>(w.t), j, j1);
        const uint4 vd = resid ? fetch_vec<E, kVec>(reinterpret_cast<const St*>(w.d), j, j1)
                               : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int e = 0; e < E::kEPV; ++e)
          if (j + e < j1 && draw_weight(E::elem(vt, e), resid ? E::elem(vd, e) : 0.0f, p.scale,
                                        w, resid, e) > 0.0f)
            tok = j + e;
      }
      ws.tok = tok;
    }
  }
  __syncthreads();
  int tok = ws.tok;
  if (tok < 0 || tok >= p.V) tok = min(j0, p.V - 1);  // unreachable with finite inputs
  return tok;
}

// Two-kernel path (rows of more than kClusterMaxChunks chunks): one CTA per
// sequence picks the chunk from the stored chunk totals and walks it.
template <typename E, bool kVec>
__global__ void __launch_bounds__(kThreads) draw_resolve_kernel(const SampleParams p) {
  __shared__ __align__(16) float s_g[kVecPerChunk];
  __shared__ WalkScratch ws;
  __shared__ FSum s_target, s_base;
  __shared__ int s_c, s_fallback;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");  // see argmax_resolve_kernel
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.x;
  const int C = p.nchunks;
  const DrawDesc d = p.desc[b];
  const DrawRows w = draw_rows<E>(p, b, d);
  FSum total = FSum::zero();
  if (warp == 0) {
    int cstar = 0;
    FSum base = FSum::zero();
    const FSum* cs = p.csum + (size_t)b * C;
    total = chunk_prefix(cs, C, nullptr, &cstar, &base);
    int fb = 0;
    if (d.n < p.k && !(total.hi > 0.0f)) {
      // the residual mass vanished in rounding: sample p of the rejected row
      fb = 1;
      cs = p.csum_p + (size_t)b * C;
      total = chunk_prefix(cs, C, nullptr, &cstar, &base);
      if (lane == 0) set_flag(p.flags, kFlagResidualFallback);
    }
    const FSum target = df_mul_f(p.u_sample[b], total);
    chunk_prefix(cs, C, &target, &cstar, &base);
    if (lane == 0) {
      s_c = cstar;
      s_base = base;
      s_target = target;
      s_fallback = fb;
    }
  }
  __syncthreads();
  const bool fallback = s_fallback != 0;
  const bool resid = d.n < p.k && !fallback;
  const int cstar = s_c;
  const float* gs = (fallback ? p.gsum_p : p.gsum) + ((size_t)b * C + cstar) * kVecPerChunk;
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q)
    s_g[q * kThreads + threadIdx.x] = __ldcg(gs + q * kThreads + threadIdx.x);
  __syncthreads();
  const int tok = walk_chunk<E, kVec>(p, w, resid, s_g, cstar, s_target, s_base, ws);
  if (threadIdx.x == 0) {
    p.out_tokens[(size_t)b * (p.k + 1) + d.n] = tok;
    p.resid_mass[b] = (d.n < p.k && !fallback) ? __fadd_rn(total.hi, total.lo) : 0.0f;
  }
}

// ---------------------------------------------------------------------------
// Cluster path: merge, accept test, draw prefix sums and walk in one kernel
// ---------------------------------------------------------------------------
// One cluster of kClusterCTAs CTAs per sequence (rows of up to
// kClusterMaxChunks chunks).  Before waiting for the statistics kernel, each
// CTA loads the sequence's draft tokens and uniforms (inputs the statistics
// kernel does not write).  Every CTA merges all of the sequence's rows (one
// warp per row; the records are few and in L2) and runs the accept test
// itself (rank 0 writes the outputs).  CTA `rank` then builds the prefix
// structure of chunks c = rank (mod kClusterCTAs) in its shared memory: its
// first chunk through registers while a bulk async copy brings the second
// (target and draft) into a staging buffer, and so on alternately.  Each CTA
// writes its chunk totals into every CTA's shared memory (distributed shared
// memory); after one cluster barrier every CTA picks the chunk from its own
// copy, the others leave, and the chunk's owner walks it.
constexpr int kClusterCTAs = 4;
constexpr int kLocalChunks = 4;
constexpr int kClusterMaxChunks = kClusterCTAs * kLocalChunks;
constexpr size_t kFinishGroupBytes = (size_t)kLocalChunks * kVecPerChunk * sizeof(float);
constexpr size_t kFinishSmem = kFinishGroupBytes + 2 * (size_t)kChunkBytes;

// Quad sums of one chunk's group array (thread t: vectors 4t..4t+3) and
// their inclusive scan within each warp; lane 31 leaves the warp's total in
// wt[warp].  Every evaluation over the same group array gives the same
// values, so the walk can repeat it for one warp.
__device__ __forceinline__ FSum quad_scan(const float* s_g, FSum* wt, FSum* my_quad) {
  const FSum q = quad_sum(*reinterpret_cast<const float4*>(s_g + 4 * threadIdx.x));
  const FSum inc = warp_scan_df(q);
  if (wt && (threadIdx.x & 31) == 31) wt[threadIdx.x >> 5] = inc;
  *my_quad = q;
  return inc;
}

// Prefixes of the warp totals of up to two local chunks at once (one warp,
// a 16-lane scan per chunk): wp[lc][i] = wt[lc][0] + ... + wt[lc][i], and
// ctot[lc] = wp[lc][kWarps - 1], the chunk total.  The walk compares the
// target against these same prefixes to pick the warp block.
static_assert(kWarps == 16, "two chunks of warp totals per warp scan");
__device__ __forceinline__ void warp_prefixes(const FSum (*wt)[kWarps], FSum (*wp)[kWarps],
                                              FSum* ctot, int nl) {
  const int lane = threadIdx.x & 31;
  for (int lc0 = 0; lc0 < nl; lc0 += 2) {
    const int lc = lc0 + (lane >> 4), i = lane & 15;
    FSum v = lc < nl ? wt[lc][i] : FSum::zero();
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      FSum y;
      y.hi = __shfl_up_sync(0xffffffffu, v.hi, o);
      y.lo = __shfl_up_sync(0xffffffffu, v.lo, o);
      if (i >= o) v = df_add(y, v);
    }
    if (lc < nl) {
      wp[lc][i] = v;
      if (i == 15) ctot[lc] = v;
    }
  }
}

// Chunk choice of the draw (one warp, n <= 32 chunk totals v in lane order):
// the normalised inclusive scan gives the total; the target is u * total;
// the chosen chunk is the first whose inclusive prefix exceeds the target
// (else the last with positive mass), with its exclusive prefix.
struct ChunkChoice {
  FSum total, target, base;
  int c;
};
__device__ __forceinline__ ChunkChoice choose_chunk(const FSum& v, int n, float u) {
  const int lane = threadIdx.x & 31;
  const FSum inc = df_norm(warp_scan_df(v));
  ChunkChoice ch;
  ch.total.hi = __shfl_sync(0xffffffffu, inc.hi, 31);
  ch.total.lo = __shfl_sync(0xffffffffu, inc.lo, 31);
  ch.target = df_mul_f(u, ch.total);
  const unsigned hit = __ballot_sync(0xffffffffu, lane < n && df_less(ch.target, inc));
  const unsigned pos = __ballot_sync(0xffffffffu, lane < n && v.hi > 0.0f);
  ch.c = hit ? (__ffs(hit) - 1) : (pos ? (31 - __clz(pos)) : 0);
  FSum excl;
  excl.hi = __shfl_up_sync(0xffffffffu, inc.hi, 1);
  excl.lo = __shfl_up_sync(0xffffffffu, inc.lo, 1);
  if (lane == 0) excl = FSum::zero();
  ch.base.hi = __shfl_sync(0xffffffffu, excl.hi, ch.c);
  ch.base.lo = __shfl_sync(0xffffffffu, excl.lo, ch.c);
  return ch;
}

// Group sums of one chunk's draw weights from 16-byte vectors already in
// registers (vt: target, vd: draft) into g[vi]; with `gp`, the p-only sums
// too.
template <typename E>
__device__ __forceinline__ void draw_groups_from(const SampleParams& p, const DrawRows& w,
                                                 bool resid, int nvec, const uint4 (&vt)[kVecPerThread],
                                                 const uint4 (&vd)[kVecPerThread], float* g) {
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) {
    const int vi = q * kThreads + (int)threadIdx.x;
    float a = 0.0f;
    if (vi < nvec) {
#pragma unroll
      for (int e = 0; e < E::kEPV; ++e) {
        const float pt = draw_p(E::elem(vt[q], e), p.scale, w, e);
        a = __fadd_rn(a, resid ? draw_r(pt, E::elem(vd[q], e), p.scale, w, e) : pt);
      }
    }
    g[vi] = a;
  }
}

// Walk of the chosen chunk by its owner CTA, from what the chunk pass left:
// the group sums (s_g), the warp totals (wt) and their sequential prefixes
// (wp).
// Warp 0 picks the warp block from the prefixes; that block's warp scans its
// quads, loads its block's vectors (coalesced, while it scans), and finds
// the vector and element all at once: lane l takes element l % E of the
// quad's vector l / E, recomputes that vector's weights and adds them in the
// order of the group sums, so each lane holds exactly the running sum a
// sequential walk reaches at its element.  Rounding that leaves the target
// just past a level's end takes the last position with positive weight, as
// in walk_chunk.
struct QuadWalk {
  FSum wbase;
  int wb, exact, tok;
};

template <typename E, bool kVec>
__device__ int walk_chunk_quads(const SampleParams& p, const DrawRows& w, bool resid,
                                const float* s_g, const FSum* wt, const FSum* wp, int cstar,
                                const FSum& target, const FSum& base, QuadWalk& qw) {
  using St = typename E::storage;
  constexpr int kE = E::kEPV;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int j0 = cstar * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
  const int nvec = (j1 - j0 + kE - 1) / kE;
  if (warp == 0) {
    const FSum pre = lane < kWarps ? df_add(base, wp[lane]) : FSum::zero();
    const float wv = lane < kWarps ? wt[lane].hi : 0.0f;
    const unsigned hit = __ballot_sync(0xffffffffu, lane < kWarps && df_less(target, df_norm(pre)));
    const unsigned pos = __ballot_sync(0xffffffffu, lane < kWarps && wv > 0.0f);
    const int wb = hit ? (__ffs(hit) - 1) : (pos ? (31 - __clz(pos)) : 0);
    FSum prev;
    prev.hi = __shfl_sync(0xffffffffu, pre.hi, wb > 0 ? wb - 1 : 0);
    prev.lo = __shfl_sync(0xffffffffu, pre.lo, wb > 0 ? wb - 1 : 0);
    if (lane == 0) {
      qw.wb = wb;
      qw.exact = hit != 0;
      qw.wbase = wb > 0 ? prev : base;
      qw.tok = -1;
    }
  }
  __syncthreads();
  if (warp == qw.wb) {
    // this warp block's vectors, coalesced: lane l holds vectors 32 i + l
    const uint4 ninf = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
    uint4 xt[4], xd[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int vi = 128 * warp + 32 * i + lane;
      const int j = j0 + vi * kE;
      xt[i] = vi < nvec ? fetch_vec<E, kVec>(reinterpret_cast<const St*>(w.t), j, j1) : ninf;
      xd[i] = (resid && vi < nvec)
                  ? fetch_vec<E, kVec>(reinterpret_cast<const St*>(w.d), j, j1)
                  : ninf;
    }
    FSum q;
    const FSum inc = quad_scan(s_g, nullptr, &q);
    FSum exc;
    exc.hi = __shfl_up_sync(0xffffffffu, inc.hi, 1);
    exc.lo = __shfl_up_sync(0xffffffffu, inc.lo, 1);
    if (lane == 0) exc = FSum::zero();
    const FSum wbase = qw.wbase;
    const unsigned qhit =
        __ballot_sync(0xffffffffu, qw.exact && df_less(target, df_norm(df_add(wbase, inc))));
    const unsigned qpos = __ballot_sync(0xffffffffu, q.hi > 0.0f);
    const int L = qhit ? (__ffs(qhit) - 1) : (qpos ? (31 - __clz(qpos)) : 0);
    FSum run;
    run.hi = __shfl_sync(0xffffffffu, exc.hi, L);
    run.lo = __shfl_sync(0xffffffffu, exc.lo, L);
    run = df_add(wbase, run);
    const bool act = lane < 4 * kE;
    const int v = act ? lane / kE : 3, e = lane % kE;
    // vector v of quad L is vector 4L + v of the block: lane (4L + v) % 32,
    // register L / 8 (the same for every lane)
    const int r = L >> 3, srcl = (4 * L + v) & 31;
    const uint4 st = r == 0 ? xt[0] : r == 1 ? xt[1] : r == 2 ? xt[2] : xt[3];
    const uint4 sd = r == 0 ? xd[0] : r == 1 ? xd[1] : r == 2 ? xd[2] : xd[3];
    uint4 at, ad;
    at.x = __shfl_sync(0xffffffffu, st.x, srcl);
    at.y = __shfl_sync(0xffffffffu, st.y, srcl);
    at.z = __shfl_sync(0xffffffffu, st.z, srcl);
    at.w = __shfl_sync(0xffffffffu, st.w, srcl);
    ad.x = __shfl_sync(0xffffffffu, sd.x, srcl);
    ad.y = __shfl_sync(0xffffffffu, sd.y, srcl);
    ad.z = __shfl_sync(0xffffffffu, sd.z, srcl);
    ad.w = __shfl_sync(0xffffffffu, sd.w, srcl);
    const int quad = warp * 32 + L;
    const float4 g4 = *reinterpret_cast<const float4*>(s_g + 4 * quad);
    const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
    // running sum before vector v, as a walk over the quad's vectors adds it
#pragma unroll
    for (int i = 0; i < 3; ++i)
      if (i < v && gv[i] > 0.0f) run = df_add(run, df_from(gv[i]));
    const float gme = v == 0 ? gv[0] : v == 1 ? gv[1] : v == 2 ? gv[2] : gv[3];
    const bool vhit =
        act && qhit != 0 && gme > 0.0f && df_less(target, df_norm(df_add(run, df_from(gme))));
    float part = 0.0f, we = 0.0f;
#pragma unroll
    for (int i = 0; i < kE; ++i) {
      const float wi =
          draw_weight(E::elem(at, i), resid ? E::elem(ad, i) : 0.0f, p.scale, w, resid, i);
      if (i <= e) part = __fadd_rn(part, wi);
      if (i == e) we = wi;
    }
    const int jj = j0 + (4 * quad + v) * kE + e;
    const unsigned vh = __ballot_sync(0xffffffffu, vhit && e == 0);
    const unsigned vp = __ballot_sync(0xffffffffu, act && e == 0 && gme > 0.0f);
    // the first vector whose end passes the target, else the last positive one
    const int vsel = vh ? (__ffs(vh) - 1) / kE : (vp ? (31 - __clz(vp)) / kE : -1);
    const bool mine = act && v == vsel;
    const unsigned eh = __ballot_sync(
        0xffffffffu,
        vh != 0 && mine && we > 0.0f && df_less(target, df_norm(df_add(run, df_from(part)))));
    const unsigned lp = __ballot_sync(0xffffffffu, mine && we > 0.0f && jj < j1);
    const int src = eh ? (__ffs(eh) - 1) : (lp ? (31 - __clz(lp)) : 0);
    const int tj = __shfl_sync(0xffffffffu, jj, src);
    if (lane == 0) qw.tok = (eh | lp) ? tj : -1;
  }
  __syncthreads();
  int tok = qw.tok;
  if (tok < 0 || tok >= p.V) tok = min(j0, p.V - 1);  // unreachable with finite inputs
  return tok;
}

template <typename E, bool kVec>
__global__ void __launch_bounds__(kThreads, 2) sample_finish_kernel(const SampleParams p) {
  using St = typename E::storage;
  namespace cg = cooperative_groups;
  extern __shared__ __align__(128) uint8_t fin_mem[];
  float* s_g = reinterpret_cast<float*>(fin_mem);  // [kLocalChunks][kVecPerChunk]
  uint8_t* s_stage = fin_mem + kFinishGroupBytes;  // target chunk | draft chunk
  __shared__ RowStats s_rows[kMaxSeqRows];
  __shared__ int s_tok[kMaxDraft];
  __shared__ float s_ua[kMaxDraft];
  __shared__ FSum s_ctot[kLocalChunks], s_call[kClusterMaxChunks];
  __shared__ FSum s_wt[kLocalChunks][kWarps], s_wp[kLocalChunks][kWarps];
  __shared__ QuadWalk s_walk;
  __shared__ DrawDesc s_desc;
  __shared__ FSum s_target, s_base, s_total;
  __shared__ uint64_t s_bar;
  __shared__ int s_c, s_fallback;

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / kClusterCTAs;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int C = p.nchunks;
  const int rows_per_seq = 2 * p.k + 1;

  // 0. inputs the statistics kernel does not write, before waiting for it
  for (int i = threadIdx.x; i < p.k; i += kThreads) {
    s_tok[i] = p.tokens[(size_t)b * p.k + i];
    s_ua[i] = p.u_accept[(size_t)b * p.k + i];
  }
  const float u_sample = p.u_sample[b];
  if (kVec && threadIdx.x == 0) {
    mbar_init(&s_bar, 1);
    mbar_init_fence();
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");  // see argmax_resolve_kernel
  __syncthreads();

  // 1. merge every row of the sequence
  for (int r = warp; r < rows_per_seq; r += kWarps)
    finalize_stats_row<E>(p, b * rows_per_seq + r, &s_rows[r], s_tok);
  __syncthreads();

  // 2. accept test over the whole sequence
  if (warp == 0) {
    const DrawDesc dd =
        resolve_sample_seq(p, b, [&](int r) { return s_rows[r]; }, rank == 0, s_ua, s_tok);
    if (lane == 0) s_desc = dd;
  }
  __syncthreads();
  const DrawDesc d = s_desc;
  const bool resid = d.n < p.k;
  const DrawRows w = draw_rows<E>(p, b, d);

  // 3. prefix structure of this CTA's chunks: even local chunks through
  // registers, odd ones through the staging buffer (bulk async copies);
  // each chunk leaves its group sums (s_g) and its warp totals (s_wt)
  // thread 0 keeps at most one staging copy (pair) in flight; stage_pending
  // is the barrier parity of the one it has not yet seen land (-1: none)
  int stage_pending = -1;
  auto stage_issue = [&](int lc) {  // thread 0
    const int c = rank + kClusterCTAs * lc;
    stage_pending = (lc >> 1) & 1;
    const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
    const unsigned bytes = (unsigned)(j1 - j0) * (unsigned)sizeof(St);
    mbar_expect_tx(&s_bar, resid ? 2 * bytes : bytes);
    bulk_g2s(s_stage, reinterpret_cast<const St*>(w.t) + j0, bytes, &s_bar);
    if (resid) bulk_g2s(s_stage + kChunkBytes, reinterpret_cast<const St*>(w.d) + j0, bytes, &s_bar);
  };
  if (kVec && threadIdx.x == 0 && rank + kClusterCTAs < C) stage_issue(1);
  bool stage_ok = true;
  for (int lc = 0; lc < kLocalChunks; ++lc) {
    const int c = rank + kClusterCTAs * lc;
    if (c >= C) break;
    float* g = s_g + lc * kVecPerChunk;
    const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
    const int nvec = (j1 - j0 + E::kEPV - 1) / E::kEPV;
    uint4 vt[kVecPerThread], vd[kVecPerThread];
    if (kVec && (lc & 1)) {
      if (!mbar_wait_bounded(&s_bar, (unsigned)(lc >> 1) & 1u, p.wait_ns)) {
        stage_ok = false;
        if (threadIdx.x == 0) set_flag(p.flags, kFlagTimeout);
      } else if (threadIdx.x == 0) {
        stage_pending = -1;
      }
#pragma unroll
      for (int q = 0; q < kVecPerThread; ++q) {
        const int vi = q * kThreads + (int)threadIdx.x;
        const bool in = stage_ok && vi < nvec;
        vt[q] = in ? lds128(s_stage + (size_t)vi * 16) : make_uint4(0, 0, 0, 0);
        vd[q] = in && resid ? lds128(s_stage + kChunkBytes + (size_t)vi * 16)
                            : make_uint4(0, 0, 0, 0);
      }
      __syncthreads();  // staging buffer free
      if (threadIdx.x == 0 && stage_ok && c + 2 * kClusterCTAs < C) stage_issue(lc + 2);
    } else {
#pragma unroll
      for (int q = 0; q < kVecPerThread; ++q) {
        const int vi = q * kThreads + (int)threadIdx.x;
        const int j = j0 + vi * E::kEPV;
        vt[q] = vi < nvec ? fetch_vec<E, kVec>(reinterpret_cast<const St*>(w.t), j, j1)
                          : make_uint4(0, 0, 0, 0);
        vd[q] = (resid && vi < nvec) ? fetch_vec<E, kVec>(reinterpret_cast<const St*>(w.d), j, j1)
                                     : make_uint4(0, 0, 0, 0);
      }
    }
    draw_groups_from<E>(p, w, resid, nvec, vt, vd, g);
    __syncthreads();  // the chunk's group sums are complete
    FSum q;
    quad_scan(g, s_wt[lc], &q);
  }
  const int nl = (C - rank + kClusterCTAs - 1) / kClusterCTAs;  // local chunks
  // warp 0: this CTA's chunk totals, written into every CTA's s_call
  // (distributed shared memory), so that after the cluster barrier each CTA
  // reads only its own shared memory and may leave without a second barrier
  auto totals_to_cluster = [&]() {
    warp_prefixes(s_wt, s_wp, s_ctot, nl);
    __syncwarp();
    const int lc = lane / kClusterCTAs, peer = lane % kClusterCTAs;
    if (lc < nl) *cluster.map_shared_rank(&s_call[rank + kClusterCTAs * lc], peer) = s_ctot[lc];
  };
  __syncthreads();  // warp totals of every local chunk
  if (warp == 0) totals_to_cluster();
  cluster.sync();

  // 4. the chunk choice; every CTA computes the same total, so the rare
  // fallback below is taken by the whole cluster or by none of it
  if (warp == 0) {
    const FSum v = lane < C ? s_call[lane] : FSum::zero();
    const ChunkChoice ch = choose_chunk(v, C, u_sample);
    if (lane == 0) {
      s_fallback = resid && !(ch.total.hi > 0.0f);
      s_c = ch.c;
      s_base = ch.base;
      s_target = ch.target;
      s_total = ch.total;
    }
  }
  __syncthreads();
  const bool fallback = s_fallback != 0;
  if (fallback) {
    // the residual mass vanished in rounding: sample p of the rejected row;
    // its group sums and chunk totals replace the residual ones
    cluster.sync();  // every CTA has read the residual totals from its s_call
    for (int lc = 0; lc < kLocalChunks; ++lc) {
      const int c = rank + kClusterCTAs * lc;
      if (c >= C) break;
      float* g = s_g + lc * kVecPerChunk;
      const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
      const int nvec = (j1 - j0 + E::kEPV - 1) / E::kEPV;
      uint4 vt[kVecPerThread], vd[kVecPerThread];
#pragma unroll
      for (int q = 0; q < kVecPerThread; ++q) {
        const int vi = q * kThreads + (int)threadIdx.x;
        vt[q] = vi < nvec ? fetch_vec<E, kVec>(reinterpret_cast<const St*>(w.t),
                                                j0 + vi * E::kEPV, j1)
                          : make_uint4(0, 0, 0, 0);
        vd[q] = make_uint4(0, 0, 0, 0);
      }
      draw_groups_from<E>(p, w, false, nvec, vt, vd, g);
      __syncthreads();
      FSum q;
      quad_scan(g, s_wt[lc], &q);
    }
    __syncthreads();
    if (warp == 0) totals_to_cluster();
    cluster.sync();
    if (warp == 0) {
      const FSum v = lane < C ? s_call[lane] : FSum::zero();
      const ChunkChoice ch = choose_chunk(v, C, u_sample);
      if (lane == 0) {
        s_c = ch.c;
        s_base = ch.base;
        s_target = ch.target;
        s_total = ch.total;
      }
    }
    if (rank == 0 && threadIdx.x == 0) set_flag(p.flags, kFlagResidualFallback);
    __syncthreads();
  }
  // no CTA touches a peer's shared memory after this point

  // a staging copy whose wait ran out may still be in flight: wait for it
  // again (bounded, with the default limit) before leaving
  if (kVec && threadIdx.x == 0 && stage_pending >= 0)
    mbar_wait_bounded(&s_bar, (unsigned)stage_pending);

  // 5. the owner of the chosen chunk walks it
  const int cstar = s_c;
  if (cstar % kClusterCTAs != rank) return;
  const int lcs = cstar / kClusterCTAs;
  const int tok = walk_chunk_quads<E, kVec>(p, w, resid && !fallback, s_g + lcs * kVecPerChunk,
                                            s_wt[lcs], s_wp[lcs], cstar, s_target, s_base,
                                            s_walk);
  if (threadIdx.x == 0) {
    p.out_tokens[(size_t)b * (p.k + 1) + d.n] = tok;
    p.resid_mass[b] = (d.n < p.k && !fallback) ? __fadd_rn(s_total.hi, s_total.lo) : 0.0f;
  }
}

__global__ void selftest_exp2_kernel(const float* x, float* y_fma, float* y_sfu, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    y_fma[i] = exp2_fma(x[i]);
    y_sfu[i] = ex2(x[i]);
  }
}

}  // namespace sv
