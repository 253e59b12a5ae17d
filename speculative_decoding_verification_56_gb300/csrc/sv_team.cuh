// sv_team.cuh -- sampling verification in one kernel: teams of CTAs (thread-
// block clusters) that stream a sequence's rows and finish it while they
// stream the next one.
//
// "EAGLE-3 speculative decoding review", "Speculative Decoding" step 3 and
// "Does Using a Small Model's Answer Reduce Quality?" (eqs. A(x),
// p_residual); "EAGLE math", "Vanilla speculative decoding": per sequence,
// the softmax statistics of the 2k+1 target and draft rows, the accept test
// and first rejection, then the residual (or bonus) draw by inverse CDF.
//
// A team is a cluster of CS CTAs, one CTA per SM.  The team owns a contiguous
// range of sequences and handles them one after another.  Each CTA has three
// warp roles:
//   consumers (warps 0-15)  the first pass: a sequence's items (row, 32 KB
//       chunk) are split into CS contiguous ranges, one per CTA, streamed
//       through a ring of bulk async copies; each row segment's softmax
//       partial and the captured draft-token logit go to a per-sequence table
//       in this CTA's shared memory (two tables, alternating by sequence).
//   finishers (warps 16-23) finish a sequence while the consumers stream the
//       next: once every CTA of the team has filled its table, they merge the
//       rows (reading the peers' tables through distributed shared memory),
//       run the accept test, build the prefix sums of their share of the
//       drawn row's chunks (the re-read rows were streamed a moment earlier
//       and are usually still in L2), exchange chunk totals, and the CTA that
//       owns the chosen chunk walks it down to the token.
//   producer (warp 24, one thread) issues the ring's copies, in the order
//       the consumers take them.
// CTAs of a team meet only through mbarriers in each other's shared memory
// (remote arrivals, cluster-scope acquire), which the cluster's co-scheduling
// makes safe; no CTA waits on a CTA outside its cluster.  Every wait is
// bounded.  Shared-memory tables are reused every second sequence, after
// every peer has signalled that it finished reading them.
#pragma once

#include <cooperative_groups.h>

#include "sv_kernels.cuh"

namespace sv {

constexpr int kTmConsumers = kThreads;      // 512 consumer threads: the chunk layout
constexpr int kTmFinWarps = 8;
constexpr int kTmFinThreads = kTmFinWarps * 32;
constexpr int kTmProducerWarp = kWarps + kTmFinWarps;     // warp 24
constexpr int kTmThreads = (kTmProducerWarp + 1) * 32;     // 800
constexpr int kTmMaxStages = 6;
constexpr int kTmLocalChunks = 4;           // second-pass chunks per CTA
constexpr int kTmOctet = 8;                 // groups (vectors) per finisher thread
static_assert(kTmFinThreads * kTmOctet == kVecPerChunk, "one octet of groups per finisher");
// Segments open at once in a CTA: a consumer warp runs at most kTmMaxStages
// items ahead of the slowest (the producer refills a slot only once every
// warp has released it), so at most kTmMaxStages segments are open.
constexpr int kTmSegSlots = 8;
static_assert(kTmSegSlots >= kTmMaxStages && (kTmSegSlots & (kTmSegSlots - 1)) == 0,
              "segment slots: a power of two covering the ring");

struct TeamSegSlots {
  int cnt[kTmSegSlots];
  StatsSlot st[kTmSegSlots][kWarps];
};

// One row segment's partial in a CTA's per-sequence table, and the draft
// token's logit when this CTA streamed that element.
struct TeamRow {
  int ref;
  float hi, lo;
  float zx;
};

struct TeamParams {
  SampleParams p;
  int nstages;      // ring depth (bulk copies of 32 KB in flight per CTA)
  int seq_per_team; // sequences per team (contiguous)
};

// Shared memory of a team CTA (dynamic part; the ring comes first): nloc =
// second-pass chunks of this CTA, ceil(chunks per row / CS).
struct TeamLayout {
  int ring, rows, srows, g, bytes;
  __host__ __device__ static TeamLayout make(int nstages, int rows_per_seq, int nloc) {
    TeamLayout L;
    L.ring = 0;
    L.rows = nstages * kChunkBytes;                                   // TeamRow [2][rows]
    L.srows = L.rows + 2 * rows_per_seq * (int)sizeof(TeamRow);       // RowStats [rows]
    L.srows = (L.srows + 15) & ~15;
    L.g = L.srows + rows_per_seq * (int)sizeof(RowStats);             // float [lc][2048]
    L.g = (L.g + 15) & ~15;
    L.bytes = L.g + nloc * kVecPerChunk * (int)sizeof(float);
    return L;
  }
};

struct TeamShared {
  uint64_t full[kTmMaxStages], empty[kTmMaxStages];
  uint64_t seq_done[2];   // consumers -> finishers, this CTA (16 warp arrivals)
  uint64_t team_done[2];  // every CTA's table of the sequence is complete (CS arrivals)
  uint64_t team_tot[2];   // every CTA's chunk totals are complete (CS arrivals)
  uint64_t team_free[2];  // every CTA has read this CTA's buffers of the sequence
  uint64_t team_fb;       // every CTA's p-only totals are complete (residual fallback)
  int abort;
  TeamSegSlots ss;
  FSum ctot[2][kTmLocalChunks];    // chunk totals of the drawn row (read by peers)
  FSum ctot_p[2][kTmLocalChunks];  // p-only totals (fallback), read by peers
  FSum wtot[kTmLocalChunks][kTmFinWarps];  // warp totals of each local chunk
  int tok[kMaxDraft];
  float ua[kMaxDraft];
  DrawDesc desc;
  FSum target, base, total;
  int cstar, fallback;
};

// --- cluster helpers ---------------------------------------------------------

__device__ __forceinline__ uint32_t tm_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t tm_cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

// Arrive (release, cluster scope) on the barrier at the same offset in CTA
// `rank` of this cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint64_t* bar, uint32_t rank) {
  asm volatile(
      "{\n .reg .b32 ra;\n mapa.shared::cluster.u32 ra, %0, %1;\n"
      " mbarrier.arrive.release.cluster.shared::cluster.b64 _, [ra];\n}\n" ::"r"(smem_addr(bar)),
      "r"(rank)
      : "memory");
}

// Test a barrier phase with cluster-scope acquire (peers released into it).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, unsigned parity,
                                                      uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, "
      "%3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, unsigned parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t hint = limit_ns < kSuspendHintNs ? (uint32_t)limit_ns : kSuspendHintNs;
  if (mbar_try_wait_cluster(bar, parity, hint)) return true;
  if (limit_ns <= 1) return false;
  const uint64_t t0 = global_ns();
  for (unsigned it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait_cluster(bar, parity, hint)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
  return false;
}

__device__ __forceinline__ void fin_sync() {  // the finisher warps only
  asm volatile("bar.sync 1, %0;" ::"n"(kTmFinThreads) : "memory");
}

// Every finisher thread waits (bounded) for a team barrier phase.
__device__ __forceinline__ void fin_wait_team(uint64_t* bar, unsigned parity, unsigned* flags) {
  if (!mbar_wait_cluster(bar, parity)) set_flag(flags, kFlagTimeout);
}

// One finisher thread arrives on the barrier at this offset in every CTA of
// the team.
template <int CS>
__device__ __forceinline__ void team_arrive_all(uint64_t* bar) {
#pragma unroll
  for (int q = 0; q < CS; ++q) mbar_arrive_remote(bar, (uint32_t)q);
}

// CTA of the team that streams sequence-local item i (of I items split in CS
// contiguous ranges [I r / CS, I (r+1) / CS)).
template <int CS>
__device__ __forceinline__ int team_owner(int i, int I) {
  return (int)((((long long)i + 1) * CS - 1) / I);
}

// Sum of one finisher thread's octet of groups, added to zero in order (the
// same arithmetic wherever an octet's sum is needed).
__device__ __forceinline__ FSum octet_sum(const float* g) {
  const float4 a = *reinterpret_cast<const float4*>(g);
  const float4 b = *reinterpret_cast<const float4*>(g + 4);
  FSum s = FSum::zero();
  s.add(a.x);
  s.add(a.y);
  s.add(a.z);
  s.add(a.w);
  s.add(b.x);
  s.add(b.y);
  s.add(b.z);
  s.add(b.w);
  return s;
}

// Group sums of local chunk `c` of the drawn row(s) into g[vi] (finisher
// threads; coalesced 16-byte loads of the rows, usually from L2), then the
// octet sums, the warp scans and the chunk total.  Returns the total to
// finisher thread 0; warp totals go to wt[8].
template <typename E>
__device__ FSum team_chunk_groups(const SampleParams& p, const DrawRows& w, bool resid, int c,
                                  float* g, FSum* wt) {
  using St = typename E::storage;
  const int ft = threadIdx.x - kTmConsumers, fw = ft >> 5, lane = ft & 31;
  const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
  const int nvec = (j1 - j0) / E::kEPV;  // whole vectors (bulk-copy path)
  const St* rt = reinterpret_cast<const St*>(w.t) + j0;
  const St* rd = resid ? reinterpret_cast<const St*>(w.d) + j0 : nullptr;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint4 vt[4], vd[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int vi = (half * 4 + jj) * kTmFinThreads + ft;
      vt[jj] = vi < nvec ? __ldg(reinterpret_cast<const uint4*>(rt) + vi) : make_uint4(0, 0, 0, 0);
      vd[jj] = (resid && vi < nvec) ? __ldg(reinterpret_cast<const uint4*>(rd) + vi)
                                    : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int vi = (half * 4 + jj) * kTmFinThreads + ft;
      float a = 0.0f;
      if (vi < nvec) {
#pragma unroll
        for (int e = 0; e < E::kEPV; ++e) {
          const float pt = draw_p(E::elem(vt[jj], e), p.scale, w, e);
          a = __fadd_rn(a, resid ? draw_r(pt, E::elem(vd[jj], e), p.scale, w, e) : pt);
        }
      }
      g[vi] = a;
    }
  }
  fin_sync();
  const FSum inc = warp_scan_df(octet_sum(g + kTmOctet * ft));
  if (lane == 31) wt[fw] = inc;
  fin_sync();
  FSum t = wt[0];
  if (ft == 0)
    for (int i = 1; i < kTmFinWarps; ++i) t = df_add(t, wt[i]);
  return t;
}

// Walk local chunk `c` (group sums g, warp totals wt) down to the token, from
// the chunk's exclusive prefix `base` and the draw target (finisher warp 0).
// Where rounding leaves the target just past a level's end, the last
// position with positive weight is taken.
template <typename E>
__device__ int team_walk(const SampleParams& p, const DrawRows& w, bool resid, int c,
                         const float* g, const FSum* wt, const FSum& target, const FSum& base) {
  using St = typename E::storage;
  const int lane = threadIdx.x & 31;
  const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
  // warp block
  const FSum wv = lane < kTmFinWarps ? wt[lane] : FSum::zero();
  const FSum winc = df_norm(df_add(base, warp_scan_df(wv)));
  unsigned hit = __ballot_sync(0xffffffffu, lane < kTmFinWarps && df_less(target, winc));
  unsigned pos = __ballot_sync(0xffffffffu, lane < kTmFinWarps && wv.hi > 0.0f);
  const int wb = hit ? (__ffs(hit) - 1) : (pos ? (31 - __clz(pos)) : 0);
  bool exact = hit != 0;
  FSum wbase = base;
  for (int i = 0; i < wb; ++i) wbase = df_add(wbase, wt[i]);
  // lane (octet) within the block
  const int oct = wb * 32 + lane;
  const FSum ov = octet_sum(g + kTmOctet * oct);
  const FSum oinc = warp_scan_df(ov);
  FSum oexc;
  oexc.hi = __shfl_up_sync(0xffffffffu, oinc.hi, 1);
  oexc.lo = __shfl_up_sync(0xffffffffu, oinc.lo, 1);
  if (lane == 0) oexc = FSum::zero();
  hit = __ballot_sync(0xffffffffu, exact && df_less(target, df_norm(df_add(wbase, oinc))));
  pos = __ballot_sync(0xffffffffu, ov.hi > 0.0f);
  const int L = hit ? (__ffs(hit) - 1) : (pos ? (31 - __clz(pos)) : 0);
  exact = exact && hit != 0;
  int tok = -1;
  if (lane == L) {
    const float* gv = g + kTmOctet * oct;
    FSum run = df_add(wbase, oexc);
    int lastv = -1;
    for (int i = 0; i < kTmOctet && tok < 0; ++i) {
      if (!(gv[i] > 0.0f)) continue;
      const int vi = kTmOctet * oct + i;  // vector index within the chunk
      lastv = vi;
      const FSum nxt = df_add(run, df_from(gv[i]));
      if (exact && df_less(target, df_norm(nxt))) {
        const int j = j0 + vi * E::kEPV;
        const uint4 vt = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const St*>(w.t) + j));
        const uint4 vd = resid ? __ldg(reinterpret_cast<const uint4*>(
                                     reinterpret_cast<const St*>(w.d) + j))
                               : make_uint4(0, 0, 0, 0);
        float part = 0.0f;
        int lastpos = -1;
#pragma unroll
        for (int e = 0; e < E::kEPV; ++e) {
          const float we =
              draw_weight(E::elem(vt, e), resid ? E::elem(vd, e) : 0.0f, p.scale, w, resid, e);
          part = __fadd_rn(part, we);
          if (we > 0.0f && j + e < j1) lastpos = j + e;
          if (tok < 0 && we > 0.0f && df_less(target, df_norm(df_add(run, df_from(part)))))
            tok = j + e;
        }
        if (tok < 0) tok = lastpos;  // rounding inside the vector
      }
      run = nxt;
    }
    if (tok < 0 && lastv >= 0) {  // rounding: last positive element of the octet
      const int j = j0 + lastv * E::kEPV;
      const uint4 vt = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const St*>(w.t) + j));
      const uint4 vd = resid ? __ldg(reinterpret_cast<const uint4*>(
                                   reinterpret_cast<const St*>(w.d) + j))
                             : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int e = 0; e < E::kEPV; ++e)
        if (j + e < j1 &&
            draw_weight(E::elem(vt, e), resid ? E::elem(vd, e) : 0.0f, p.scale, w, resid, e) > 0.0f)
          tok = j + e;
    }
  }
  tok = __shfl_sync(0xffffffffu, tok, L);
  if (tok < 0 || tok >= p.V) tok = min(j0, p.V - 1);  // unreachable with finite inputs
  return tok;
}

// Wait for the copy in ring slot `slot` (phase parity `par`), move this
// consumer thread's vectors to registers (past-the-end vectors read as -inf)
// and release the slot.  A consumer that gives up sets sh.abort before it
// releases the slot, so the producer issues nothing more.
template <typename E>
__device__ __forceinline__ bool team_take(TeamShared& sh, const uint8_t* ring, int slot,
                                          unsigned par, int nvec, unsigned* flags,
                                          uint4 (&raw)[kVecPerThread], uint64_t limit_ns) {
  bool ok = *(volatile int*)&sh.abort == 0;
  if (ok && !mbar_wait_bounded(&sh.full[slot], par, limit_ns)) {
    ok = false;
    sh.abort = 1;
    set_flag(flags, kFlagTimeout);
  }
  const uint8_t* sm = ring + (size_t)slot * kChunkBytes + threadIdx.x * 16;
  const uint4 ninf = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) {
    const int vi = q * kThreads + (int)threadIdx.x;
    raw[q] = (ok && vi < nvec) ? lds128(sm + q * kThreads * 16) : ninf;
  }
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.empty[slot]);
  return ok;
}

// Emit a row segment's softmax partial into this CTA's table (consumers; the
// last warp to arrive combines the 16 warp partials).
__device__ __forceinline__ void team_emit_stats(const StatsState& st, TeamRow* row,
                                                TeamSegSlots& ss, int& seg) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slot = seg++ & (kTmSegSlots - 1);
  const int wref = warp_max_i(st.ref);
  FSum mine = st.acc;
  mine.scale(pow2i_f(st.ref - wref));
  const FSum wsum = warp_sum_df(mine);
  if (lane == 0) ss.st[slot][warp] = StatsSlot{wref, wsum.hi, wsum.lo, 0};
  // the last warp to arrive combines (the others' partials are visible to it)
  int last = 0;
  if (lane == 0) {
    __threadfence_block();
    last = atomicAdd(&ss.cnt[slot], 1) == kWarps - 1;
    if (last) {
      __threadfence_block();
      ss.cnt[slot] = 0;  // no warp can reach this slot's next use yet
    }
  }
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  StatsSlot v = lane < kWarps ? ss.st[slot][lane] : StatsSlot{kRefEmpty, 0.0f, 0.0f, 0};
  const int R = warp_max_i(v.ref);
  FSum f;
  f.hi = v.hi;
  f.lo = v.lo;
  f.scale(pow2i_f(v.ref - R));
  const FSum tot = warp_sum_df(f);
  if (lane == 0) {
    row->ref = R;
    row->hi = tot.hi;
    row->lo = tot.lo;
  }
}

template <typename E, int CS>
__global__ void __launch_bounds__(kTmThreads, 1) team_sample_kernel(const TeamParams tp) {
  namespace cg = cooperative_groups;
  extern __shared__ __align__(1024) uint8_t tm_mem[];
  __shared__ TeamShared sh;
  using St = typename E::storage;
  const SampleParams& p = tp.p;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)tm_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = tp.nstages;
  const int C = p.nchunks;
  const int rows_per_seq = 2 * p.k + 1;
  const int I = rows_per_seq * C;          // items of one sequence
  const int lo = (int)((long long)I * rank / CS), hi = (int)((long long)I * (rank + 1) / CS);
  const int b0 = (int)tm_cluster_id() * tp.seq_per_team;
  const int b1 = min(p.B, b0 + tp.seq_per_team);
  const TeamLayout L = TeamLayout::make(S, rows_per_seq, (C + CS - 1) / CS);
  TeamRow* rows = reinterpret_cast<TeamRow*>(tm_mem + L.rows);        // [2][rows_per_seq]
  RowStats* srows = reinterpret_cast<RowStats*>(tm_mem + L.srows);    // [rows_per_seq]
  float* sg = reinterpret_cast<float*>(tm_mem + L.g);                 // [lc][2048]

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kWarps);
    }
    for (int u = 0; u < 2; ++u) {
      mbar_init(&sh.seq_done[u], kWarps);
      mbar_init(&sh.team_done[u], CS);
      mbar_init(&sh.team_tot[u], CS);
      mbar_init(&sh.team_free[u], CS);
    }
    mbar_init(&sh.team_fb, CS);
    sh.abort = 0;
    mbar_init_fence();
  }
  if (threadIdx.x < kTmSegSlots) sh.ss.cnt[threadIdx.x] = 0;
  __syncthreads();
  cluster.sync();  // every peer's barriers are initialised before any remote arrival
  // a programmatic dependent of the kernel before it in the stream: nothing is
  // read or written before that grid has finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");

  if (warp < kWarps) {
    // ------------------------------ consumers ------------------------------
    StatsState st;
    int seg = 0, slot = 0;
    unsigned par = 0;
    for (int b = b0; b < b1; ++b) {
      const int ls = b - b0, buf = ls & 1, use = ls >> 1;
      TeamRow* tbl = rows + buf * rows_per_seq;
      // the peers have read this table's previous contents
      if (use > 0 && !mbar_wait_cluster(&sh.team_free[buf], (unsigned)(use - 1) & 1u))
        set_flag(p.flags, kFlagTimeout);
      int row = lo / C, c = lo - row * C;
      int tok = row_token(p, b * rows_per_seq + row);
      for (int it = lo; it < hi; ++it) {
        const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
        uint4 raw[kVecPerThread];
        const bool ok = team_take<E>(sh, tm_mem, slot, par, (j1 - j0) / E::kEPV, p.flags, raw,
                                     p.wait_ns);
        if (ok) {
          stats_chunk<E>(raw, p.scale, st);
          if (tok >= j0 && tok < j1) {
            const int off = tok - j0, vi = off / E::kEPV;
            if ((vi & (kThreads - 1)) == (int)threadIdx.x) {
              const int q = vi / kThreads;
              const uint4 v = q == 0 ? raw[0] : q == 1 ? raw[1] : q == 2 ? raw[2] : raw[3];
              tbl[row].zx = E::elem(v, off % E::kEPV);
            }
          }
        }
        if (c + 1 == C || it + 1 == hi) {
          team_emit_stats(st, &tbl[row], sh.ss, seg);
          st = StatsState();
        }
        if (c + 1 == C) {
          c = 0;
          ++row;
          tok = row_token(p, b * rows_per_seq + row);
        } else {
          ++c;
        }
        if (++slot == S) {
          slot = 0;
          par ^= 1u;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.seq_done[buf]);
    }
  } else if (warp == kTmProducerWarp) {
    // ------------------------------ producer -------------------------------
    if (lane == 0) {
      int n = 0;  // items issued
      bool stop = false;
      for (int b = b0; b < b1 && !stop; ++b) {
        for (int it = lo; it < hi; ++it, ++n) {
          const int slot = n % S;
          if (n >= S) {
            if (!mbar_wait_bounded(&sh.empty[slot], (unsigned)((n / S - 1) & 1), p.wait_ns)) {
              sh.abort = 1;
              set_flag(p.flags, kFlagTimeout);
            }
          }
          // a consumer that gave up on a copy sets abort before it releases
          // the slot: no copy lands on a slot whose previous copy may still
          // be in flight
          if (*(volatile int*)&sh.abort) {
            stop = true;
            break;
          }
          const int row = it / C, c = it - (it / C) * C;
          const int j0 = c * E::kChunk, j1 = min(p.V, j0 + E::kChunk);
          const unsigned bytes = (unsigned)(j1 - j0) * (unsigned)sizeof(St);
          mbar_expect_tx(&sh.full[slot], bytes);
          bulk_g2s(tm_mem + (size_t)slot * kChunkBytes, seq_row_ptr<E>(p, b, row) + j0, bytes,
                   &sh.full[slot]);
        }
      }
      // every copy issued has landed before the CTA can leave
      for (int j = max(0, n - S); j < n; ++j)
        mbar_wait_bounded(&sh.full[j % S], (unsigned)((j / S) & 1));
    }
    __syncwarp();
  } else {
    // ------------------------------ finishers ------------------------------
    const int ft = threadIdx.x - kTmConsumers, fw = ft >> 5;
    int nfb = 0;  // residual fallbacks so far (the team_fb barrier's phase)
    for (int b = b0; b < b1; ++b) {
      const int ls = b - b0, buf = ls & 1, use = ls >> 1;
      const unsigned ph = (unsigned)use & 1u;
      for (int i = ft; i < p.k; i += kTmFinThreads) {
        sh.tok[i] = p.tokens[(size_t)b * p.k + i];
        sh.ua[i] = p.u_accept[(size_t)b * p.k + i];
      }
      const float u_sample = p.u_sample[b];
      // this CTA's table is complete: tell the team, then wait for the team
      if (!mbar_wait_bounded(&sh.seq_done[buf], ph)) set_flag(p.flags, kFlagTimeout);
      if (ft == 0) team_arrive_all<CS>(&sh.team_done[buf]);
      fin_wait_team(&sh.team_done[buf], ph, p.flags);
      fin_sync();  // sh.tok, sh.ua

      // 1. merge every row of the sequence from the team's tables
      for (int x = fw; x < rows_per_seq; x += kTmFinWarps) {
        const int r0 = team_owner<CS>(x * C, I), r1 = team_owner<CS>(x * C + C - 1, I);
        int ref = kRefEmpty;
        FSum f = FSum::zero();
        const int rr = r0 + lane;  // a CTA whose range is empty wrote nothing
        if (rr <= r1 && (long long)I * rr / CS < (long long)I * (rr + 1) / CS) {
          const TeamRow* pr = cluster.map_shared_rank(rows + buf * rows_per_seq + x, rr);
          ref = pr->ref;
          f.hi = pr->hi;
          f.lo = pr->lo;
        }
        const int R = warp_max_i(ref);
        f.scale(pow2i_f(ref - R));
        const FSum Ssum = df_norm(warp_sum_df(f));
        if (lane == 0) {
          double prob = 0.0;
          if (x != p.k) {
            const int i = x < p.k ? x : x - p.k - 1;
            const int t = sh.tok[i];
            if (t >= 0 && t < p.V) {
              const int owner = team_owner<CS>(x * C + t / E::kChunk, I);
              const float zx = cluster.map_shared_rank(rows + buf * rows_per_seq + x, owner)->zx;
              prob = exp2_over(__fmaf_rn(zx, p.scale, -(float)R), Ssum.hi);
            } else {
              set_flag(p.flags, kFlagTokenRange);
            }
          }
          RowStats rs;
          rs.ref = R;
          rs.inv_sum = __frcp_rn(Ssum.hi);
          rs.prob = prob;
          srows[x] = rs;
        }
      }
      fin_sync();

      // 2. accept test (rank 0 writes the outputs but the drawn token)
      if (fw == 0) {
        const DrawDesc dd =
            resolve_sample_seq(p, b, [&](int r) { return srows[r]; }, rank == 0, sh.ua);
        if (lane == 0) sh.desc = dd;
      }
      fin_sync();
      const DrawDesc d = sh.desc;
      const bool resid = d.n < p.k;
      const DrawRows w = draw_rows<E>(p, b, d);

      // 3. prefix structure of this CTA's chunks c = rank + CS * lc
      if (use > 0) fin_wait_team(&sh.team_free[buf], ph ^ 1u, p.flags);
      for (int lc = 0; lc < kTmLocalChunks; ++lc) {
        const int c = rank + CS * lc;
        if (c >= C) break;
        const FSum t = team_chunk_groups<E>(p, w, resid, c, sg + lc * kVecPerChunk, sh.wtot[lc]);
        if (ft == 0) sh.ctot[buf][lc] = t;
      }
      fin_sync();
      if (ft == 0) team_arrive_all<CS>(&sh.team_tot[buf]);
      fin_wait_team(&sh.team_tot[buf], ph, p.flags);

      // 4. every CTA reads the chunk totals and takes the same decisions
      if (fw == 0) {
        FSum v = FSum::zero();
        if (lane < C) v = *cluster.map_shared_rank(&sh.ctot[buf][lane / CS], lane % CS);
        int sel = 0;
        FSum excl;
        const FSum total = lane_prefix_select(v, C, nullptr, &sel, &excl);
        if (lane == 0) {
          sh.fallback = resid && !(total.hi > 0.0f);
          sh.total = total;
        }
      }
      fin_sync();
      const bool fallback = sh.fallback != 0;
      if (fallback) {
        // the residual mass vanished in rounding: sample p of the rejected
        // row; its group sums replace the residual ones
        for (int lc = 0; lc < kTmLocalChunks; ++lc) {
          const int c = rank + CS * lc;
          if (c >= C) break;
          const FSum t =
              team_chunk_groups<E>(p, w, false, c, sg + lc * kVecPerChunk, sh.wtot[lc]);
          if (ft == 0) sh.ctot_p[buf][lc] = t;
        }
        fin_sync();
        if (ft == 0) team_arrive_all<CS>(&sh.team_fb);
        fin_wait_team(&sh.team_fb, (unsigned)nfb & 1u, p.flags);
        ++nfb;
        if (rank == 0 && ft == 0) set_flag(p.flags, kFlagResidualFallback);
      }
      if (fw == 0) {
        FSum v = FSum::zero();
        if (lane < C)
          v = *cluster.map_shared_rank(fallback ? &sh.ctot_p[buf][lane / CS] : &sh.ctot[buf][lane / CS],
                                       lane % CS);
        int sel = 0;
        FSum excl;
        const FSum total = lane_prefix_select(v, C, nullptr, &sel, &excl);
        const FSum target = df_mul_f(u_sample, total);
        lane_prefix_select(v, C, &target, &sel, &excl);
        if (lane == 0) {
          sh.cstar = sel;
          sh.base = excl;
          sh.target = target;
          sh.total = total;
        }
      }
      fin_sync();
      // every read of the peers' buffers for this sequence is done
      if (ft == 0) team_arrive_all<CS>(&sh.team_free[buf]);

      // 5. the owner of the chosen chunk walks it
      const int cstar = sh.cstar;
      if (cstar % CS == rank && fw == 0) {
        const int lc = cstar / CS;
        const int tok = team_walk<E>(p, w, resid && !fallback, cstar, sg + lc * kVecPerChunk,
                                     sh.wtot[lc], sh.target, sh.base);
        if (lane == 0) {
          p.out_tokens[(size_t)b * (p.k + 1) + d.n] = tok;
          p.resid_mass[b] = (resid && !fallback) ? __fadd_rn(sh.total.hi, sh.total.lo) : 0.0f;
        }
      }
      fin_sync();  // the group sums are reused by the next sequence
    }
  }
  // no CTA leaves while a peer may still read its shared memory or arrive on
  // its barriers
  __syncwarp();
  cluster.sync();
}

}  // namespace sv
