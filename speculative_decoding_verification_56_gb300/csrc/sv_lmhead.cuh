// sv_lmhead.cuh -- the target's LM head fused with greedy verification, on
// the 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// "EAGLE math", "Why feature drafting lands a higher acceptance rate": the
// target's logits are its LM head applied to the hidden state, z = W_LM h.
// Greedy verification ("EAGLE-3 speculative decoding review", "Does Using a
// Small Model's Answer Reduce Quality?" greedy bullets) needs only each
// target row's argmax, so the GEMM's epilogue keeps a running (max, lowest
// index) per row and the [rows, V] logits are never written.
//
//   Z tile^T = W_LM[v0 : v0+256, :] x H[rows, :]^T   (both K-major, bf16)
//
// The vocabulary is the MMA's M and the rows are its N (up to 384 columns,
// one or two MMAs of N <= 256), so rows are padded only to a multiple of 64.
// Two CTAs of a cluster, on two SMs, share each tile through the two-CTA
// form of the MMA (cta_group::2, M = 256): each CTA loads its own 128
// vocabulary rows of W and half of each MMA's rows of H into its shared
// memory, and each holds the 128 x rows accumulator of its vocabulary rows
// (fp32) in its own tensor memory.  Per SM and K step this moves 16 KB of W
// and half of H, against all of H for a CTA that computes 128 x rows alone.
// Each pair walks a contiguous range of 256-entry vocabulary tiles for a
// group of rows.  Warp roles (320 threads per CTA):
//   warp 0     TMA producer (both CTAs): per 64-wide K step, the CTA's W
//              slice and H halves (128-byte swizzled) into a ring of up to
//              eight stages; both CTAs' bytes complete on the leader's
//              `full` barrier of the stage
//   warp 1     allocates tensor memory (both CTAs); in the leader (cluster
//              rank 0) lane 0 issues tcgen05.mma (M=256, N=rows/2 or rows,
//              K=16) and commits stage releases and tile completion to the
//              barriers of both CTAs
//   warps 2-9  epilogue (both CTAs), two warps per 32-lane quadrant of
//              tensor memory taking alternate 32-column blocks: tcgen05.ld,
//              a butterfly reduction across lanes per column (row), a merge
//              of the four quadrants in shared memory and a running argmax
//              per row (lowest index wins ties)
// Tensor memory holds two to four accumulator slots (three of 160 columns
// for 320 rows), used in rotation: the next tile's MMAs start in the free
// slot while the epilogue still reads the previous tile, and each slot is
// released to the leader as soon as both CTAs' epilogues have read it.
// Each CTA writes one argmax record per row for its vocabulary lanes, in the
// layout the greedy resolve kernel merges.  Every wait is bounded, and both
// CTAs meet at cluster barriers after set-up and before tensor memory is
// freed, so no CTA leaves while its peer can still touch its memory.
#pragma once

#include <cuda.h>

#include "sv_kernels.cuh"

namespace sv {

constexpr int kLmBV = 128;           // vocabulary rows per CTA and tile (tensor-memory lanes)
constexpr int kLmPairBV = 2 * kLmBV;  // vocabulary per tile of a CTA pair (UMMA M)
constexpr int kLmMaxRows = 384;       // rows per row group (UMMA N total, tensor-memory columns)
constexpr int kLmMaxN = 256;          // N of one MMA instruction
constexpr int kLmBK = 64;             // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kLmMaxStages = 8;
constexpr int kLmRingBytes = 192 * 1024;  // operand ring per CTA (dynamic shared memory)
constexpr int kLmThreads = 320;
constexpr int kLmEpiThreads = kLmThreads - 64;  // warps 2-9
constexpr int kLmABytes = kLmBV * kLmBK * 2;  // 16 KB: the CTA's W slice
constexpr int kLmHBox = 64;                   // row groups are multiples of this
constexpr int kLmTmemCols = 512;
constexpr int kLmMaxSlots = 4;  // accumulator slots of nper columns in tensor memory

// MMAs per K step of 16 for a row group of R rows (a multiple of kLmHBox),
// the rows of each MMA that one CTA of the pair holds, a CTA's bytes per
// stage, and the ring depth that fits kLmRingBytes.
__host__ __device__ constexpr int lm_nmma(int R) { return (R + kLmMaxN - 1) / kLmMaxN; }
__host__ __device__ constexpr int lm_half_rows(int R) { return R / lm_nmma(R) / 2; }
__host__ __device__ constexpr int lm_stage_bytes(int R) { return kLmABytes + R * 64; }
__host__ __device__ constexpr int lm_stages(int stage_bytes) {
  return kLmRingBytes / stage_bytes < kLmMaxStages ? kLmRingBytes / stage_bytes : kLmMaxStages;
}

// What the epilogue makes of each accumulator tile.
enum LmMode : int {
  kLmArgmax = 0,  // running (max, lowest index) per row: greedy verification
  kLmStats = 1,   // running softmax partial per row and the draft token's logit: sampling
  kLmLogits = 2,  // the logits themselves, fp32 (the rows a sampling draw re-reads)
};

struct LmHeadParams {
  int rows, d, V;       // rows of the first matrix (argmax: B * (k+1))
  int ntiles;           // ceil(V / kLmPairBV): tiles of a CTA pair
  int grp_rows;         // rows per row group of the first matrix (multiple of kLmHBox)
  int stage_bytes;      // ring stride: lm_stage_bytes of the larger row group
  int nstages;          // lm_stages(stage_bytes)
  ArgPartial* part;     // argmax: [rows, gridDim.x] one record per CTA segment
  unsigned* flags;
  // sampling (kLmStats): the first matrix holds the target rows [B(k+1), d],
  // the second the drafted features [Bk, d]; records use the sampling row
  // numbering b(2k+1) + r (r <= k target, r > k draft)
  int ngroups0;         // row groups of the first matrix (blockIdx.y below it)
  int rows1, grp_rows1; // rows and rows per group of the second matrix
  int k;
  float scale;          // log2(e) / T
  const int32_t* tokens;    // [B, k]
  SoftmaxPartial* spart;    // [B(2k+1), gridDim.x]
  float* zx;                // [B(2k+1)]: the draft token's logit
  float* logits;            // kLmLogits: [rows, V] fp32
};

// --- tcgen05 / TMA helpers (inline PTX) ------------------------------------

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled operand:
// start address >> 4 (bits 0-13), leading-byte offset 0 (unused for swizzled
// K-major), stride-byte offset 1024 >> 4 between 8-row groups (bits 32-45),
// descriptor version 1 (bits 46-47), layout "128-byte swizzle" = 2 (bits
// 61-63).  The operand tile starts on a 1024-byte boundary; a K step of 16
// elements inside the 128-byte row advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_byte_addr) {
  return (uint64_t)((smem_byte_addr & 0x3FFFFu) >> 4) | ((uint64_t)(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3
// (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t umma_idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// This CTA's rank in its cluster, and the shared::cluster address of a
// shared-memory variable in the cluster's CTA `rank`.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(rank));
  return a;
}

// Every thread of both CTAs; memory before it is visible to the cluster after.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier of either CTA of the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

// mbar_wait_bounded for a barrier that the peer CTA also arrives on: the
// phase test acquires at cluster scope.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, unsigned parity) {
  const uint64_t t0 = global_ns();
  for (unsigned it = 0; it < (1u << 30); ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, "
        "%3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    if (done) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
  return false;
}

// 2-D tile load into this CTA's shared memory whose bytes complete on an
// mbarrier of either CTA of the pair (bar_cluster: shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

// One MMA of the CTA pair (issued by the leader): A's 256 rows are the two
// CTAs' 128-row operands at the same shared-memory address, B's N rows the
// two CTAs' N/2-row operands (the leader's first), and each CTA's tensor
// memory receives the accumulator rows of its own A rows.
__device__ __forceinline__ void umma_bf16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the barrier at `bar`'s offset in both CTAs of the pair when
// every tcgen05 operation this thread issued completes.
__device__ __forceinline__ void umma_commit_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_addr(bar)),
      "h"((unsigned short)3)
      : "memory");
}

// The same, on this CTA's barrier only.
__device__ __forceinline__ void umma_commit_own(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of the warp's 32 lanes: thread t gets lane
// (quadrant base + t), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// The same load without its wait, and the wait: tmem_wait_ld ties the
// registers of one earlier load, so that nothing reads them before the
// loads have completed (the first wait covers every load issued before it).
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// ---------------------------------------------------------------------------

// (value, index) comparison: larger value, then lower index.
__device__ __forceinline__ bool lm_better(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

// Sampling row number (b(2k+1) + r) of local row `lr` of the CTA's matrix.
__device__ __forceinline__ int lm_sample_row(const LmHeadParams& p, bool draft, int lr) {
  if (!draft) {
    const int b = lr / (p.k + 1), i = lr - b * (p.k + 1);
    return b * (2 * p.k + 1) + i;
  }
  const int b = lr / p.k, i = lr - b * p.k;
  return b * (2 * p.k + 1) + p.k + 1 + i;
}

// Butterfly over the 32 lanes of a warp for 32 columns at once: afterwards
// lane c holds the reduction of column c over all lanes in v[0].
template <typename Op>
__device__ __forceinline__ void lane_butterfly(float (&v)[32], Op op) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int j = 0; j < off; ++j) {
      const float send = upper ? v[j] : v[j + off];
      const float keep = upper ? v[j + off] : v[j];
      v[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, off));
    }
  }
}

template <int Mode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kLmThreads, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap map_h,
                  const __grid_constant__ CUtensorMap map_h1,
                  const __grid_constant__ CUtensorMap map_w, const LmHeadParams p) {
  extern __shared__ uint8_t lm_raw[];
  __shared__ uint64_t full[kLmMaxStages], empty[kLmMaxStages];
  __shared__ uint64_t acc_full[2], slot_empty[kLmMaxSlots], drain;
  __shared__ uint32_t tmem_base_holder;
  __shared__ int s_abort;
  __shared__ float red_v[4][kLmMaxRows];  // per-quadrant column results of one tile
  __shared__ int red_i[4][kLmMaxRows];
  __shared__ int s_tok[kLmMaxRows];       // kLmStats: the draft token of each column (row)

  // 1024-byte aligned operand ring (128-byte swizzle atoms)
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(lm_raw) + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: the pair's leader, which issues the MMAs
  const bool leader = rank == 0;
  // the pair's row group: of the first matrix, or (sampling) of the second
  const bool second = (int)blockIdx.y >= p.ngroups0;
  const int R = second ? p.grp_rows1 : p.grp_rows;  // columns used (rows past the end read as 0)
  const int row0 = second ? ((int)blockIdx.y - p.ngroups0) * p.grp_rows1 : blockIdx.y * p.grp_rows;
  const int nrows = second ? p.rows1 : p.rows;
  const CUtensorMap* hmap = second ? &map_h1 : &map_h;
  const int nmma = lm_nmma(R);          // MMAs per K step of 16
  const int half = lm_half_rows(R);     // rows of each MMA held by one CTA
  const int nper = 2 * half;            // N of each MMA (a multiple of 32)
  // Tensor memory holds nslots accumulator slots of nper columns; tile j's
  // MMA m accumulates in slot (j * nmma + m) mod nslots.  With three slots of
  // 160 columns (320 rows) the next tile's first MMA writes the free slot
  // and its second the slot the epilogue reads first; with one MMA per tile
  // the two slots alternate.  nslots <= 2 * nmma keeps the MMAs at most one
  // tile ahead of the epilogue (a slot is reused by the tile after next at
  // the latest), which the two alternating acc_full barriers rely on.
  const int nslots = min(kLmTmemCols / nper, 2 * nmma);
  const int S = p.nstages;
  // the pair owns the vocabulary tiles [T0, T1)
  int T0, T1;
  {
    const long long G = gridDim.x / 2, g = blockIdx.x / 2;
    T0 = (int)((long long)p.ntiles * g / G);
    T1 = (int)((long long)p.ntiles * (g + 1) / G);
  }
  const int nsteps = T1 - T0;
  const int nk = (p.d + kLmBK - 1) / kLmBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);   // the leader's producer; both CTAs' bytes (leader only)
      mbar_init(&empty[s], 1);  // released by the MMAs that read the stage
    }
    mbar_init(&acc_full[0], 1);
    mbar_init(&acc_full[1], 1);
    // the eight epilogue warps of both CTAs read every slot (leader only)
    for (int s = 0; s < kLmMaxSlots; ++s) mbar_init(&slot_empty[s], 16);
    mbar_init(&drain, 1);
    s_abort = 0;
    mbar_init_fence();
  }
  if (warp == 1) {  // tensor memory for the accumulators (a warp of each CTA, together)
    asm volatile(
        "tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
            smem_addr(&tmem_base_holder)),
        "r"(kLmTmemCols)
        : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  // both CTAs' barriers and tensor memory exist before either CTA's copies,
  // MMAs or commits can reach them
  tmem_fence_before();
  cluster_sync_all();
  tmem_fence_after();
  const uint32_t tmem_base = tmem_base_holder;
  // a programmatic dependent of the kernel before it in the stream: the set-up
  // above overlaps that kernel's end; no global memory is touched before it
  // has finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if constexpr (Mode == kLmStats) {
    // the draft token of each row of the group (-1: the bonus row, padding)
    for (int c = threadIdx.x; c < R; c += kLmThreads) {
      const int lr = row0 + c;
      int t = -1;
      if (lr < nrows) {
        if (!second) {
          const int b = lr / (p.k + 1), i = lr - b * (p.k + 1);
          if (i < p.k) t = p.tokens[(size_t)b * p.k + i];
        } else {
          t = p.tokens[lr];  // draft row b*k + i carries token [b, i]
        }
      }
      s_tok[c] = t;
    }
    __syncthreads();
  }

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    const uint32_t full0 = cluster_addr(&full[0], 0);  // the leader's barriers
    const unsigned pair_bytes = 2u * (unsigned)lm_stage_bytes(R);
    int stage = 0, issued = 0;
    unsigned phase = 0;
    for (int j = 0; j < nsteps && !*(volatile int*)&s_abort; ++j) {
      const int t = T0 + j;
      for (int kb = 0; kb < nk; ++kb) {
        // the MMAs that read this stage's previous contents have completed
        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u)) {
          s_abort = 1;
          set_flag(p.flags, kFlagTimeout);
          break;
        }
        ++issued;
        uint8_t* st = ring + (size_t)stage * p.stage_bytes;
        const uint32_t fb = full0 + 8u * (uint32_t)stage;
        if (leader) mbar_expect_tx(&full[stage], pair_bytes);
        tma_load_2d_pair(st, &map_w, kb * kLmBK, t * kLmPairBV + (int)rank * kLmBV, fb);
        for (int m = 0; m < nmma; ++m)
          tma_load_2d_pair(st + kLmABytes + m * half * 128, hmap, kb * kLmBK,
                           row0 + m * nper + (int)rank * half, fb);
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // every copy this thread issued has landed before the CTA can leave: the
    // leader sees its stages fill; the follower's copies complete on the
    // leader's barriers, so it waits for the MMAs that read them to release
    // the stages
    for (int j = max(0, issued - S); j < issued; ++j) {
      const unsigned par = (unsigned)((j / S) & 1);
      if (leader)
        mbar_wait_bounded(&full[j % S], par);
      else
        mbar_wait_bounded(&empty[j % S], par);
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ---------------- MMA issuer (the leader) ----------------
    const uint32_t idesc = umma_idesc_bf16_f32(kLmPairBV, nper);
    // The issue loop is what paces the tensor cores here (one thread issues
    // every MMA of the pair), so descriptors are built once: the start
    // address field (16-byte units, bits 0-13) advances by 2 per K step of
    // 16 and by stage_bytes / 16 per stage.  Shared-memory offsets stay below
    // 2^18 bytes, so the additions never carry out of the field.
    const uint64_t adesc0 = umma_desc_sw128(smem_addr(ring));
    const uint64_t sstep = (uint64_t)(p.stage_bytes >> 4);
    const uint64_t bofs = (uint64_t)(kLmABytes >> 4);
    const uint64_t mofs = (uint64_t)((half * 128) >> 4);
    const bool two = nmma > 1;
    int stage = 0, sbase = 0;
    unsigned phase = 0, spar = 0;  // spar: bit s = uses of slot s so far, mod 2
    for (int j = 0; j < nsteps && !*(volatile int*)&s_abort; ++j) {
      // both CTAs' epilogues have read the slots this tile accumulates in
      const int sl0 = sbase, sl1 = sbase + 1 < nslots ? sbase + 1 : 0;
      bool ok = mbar_wait_cluster_bounded(&slot_empty[sl0], ((spar >> sl0) & 1u) ^ 1u);
      spar ^= 1u << sl0;
      if (ok && two) {
        ok = mbar_wait_cluster_bounded(&slot_empty[sl1], ((spar >> sl1) & 1u) ^ 1u);
        spar ^= 1u << sl1;
      }
      if (!ok) {
        s_abort = 1;
        set_flag(p.flags, kFlagTimeout);
        break;
      }
      tmem_fence_after();
      const uint32_t tm0 = tmem_base + (uint32_t)(sl0 * nper);
      const uint32_t tm1 = tmem_base + (uint32_t)(sl1 * nper);
      sbase = (sbase + nmma) % nslots;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_bounded(&full[stage], phase)) {
          s_abort = 1;
          set_flag(p.flags, kFlagTimeout);
          break;
        }
        tmem_fence_after();
        const uint64_t ad = adesc0 + (uint64_t)stage * sstep;
        const uint64_t bd = ad + bofs;
        const uint32_t acc = kb > 0 ? 1u : 0u;
        if (two) {
          umma_bf16_pair(tm0, ad, bd, idesc, acc);
          umma_bf16_pair(tm1, ad, bd + mofs, idesc, acc);
#pragma unroll
          for (int kk = 1; kk < kLmBK / 16; ++kk) {
            umma_bf16_pair(tm0, ad + 2 * kk, bd + 2 * kk, idesc, 1u);
            umma_bf16_pair(tm1, ad + 2 * kk, bd + mofs + 2 * kk, idesc, 1u);
          }
        } else {
          umma_bf16_pair(tm0, ad, bd, idesc, acc);
#pragma unroll
          for (int kk = 1; kk < kLmBK / 16; ++kk)
            umma_bf16_pair(tm0, ad + 2 * kk, bd + 2 * kk, idesc, 1u);
        }
        umma_commit_both(&empty[stage]);  // the stage is free in both CTAs once these finish
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      umma_commit_both(&acc_full[j & 1]);  // the tile's accumulators are complete in both CTAs
    }
    // every MMA this thread issued has completed before tensor memory is freed
    umma_commit_own(&drain);
    mbar_wait_bounded(&drain, 0);
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    // Accumulator lane = vocabulary entry of the tile, column = row.  Argmax
    // and statistics reduce each warp's 32 lanes per column with a butterfly
    // that leaves column c's result in lane c; the four quadrants' results
    // meet in shared memory and each epilogue thread keeps the running
    // result of rows e, e + 256 over the CTA's tiles.
    const int q = warp & 3;          // tensor-memory lane quadrant of this warp
    const int e = threadIdx.x - 64;  // 0..255 among the epilogue threads
    constexpr int kPer = (kLmMaxRows + kLmEpiThreads - 1) / kLmEpiThreads;  // rows per thread
    float best[kPer];
    int bidx[kPer];
    StatsState run[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      best[j] = -INFINITY;
      bidx[j] = 0x7FFFFFFF;
    }
    const uint32_t slot_empty0 = cluster_addr(&slot_empty[0], 0);  // the leader's barriers
    const int nblk = nper / 32;  // column blocks of one slot
    // The two warps of a quadrant take alternate column blocks, so that the
    // slot of the tile's first MMA -- the one the next tile's second MMA
    // reuses -- is read after about half of the epilogue.
    const int cb0 = warp >= 6 ? 1 : 0;
    const int ncb = R / 32;
    for (int j = 0; j < nsteps; ++j) {
      // every epilogue thread takes the same decision, so none is left at a
      // named barrier the others no longer reach
      const unsigned ok = mbar_wait_bounded(&acc_full[j & 1], (unsigned)((j >> 1) & 1)) ? 1u : 0u;
      unsigned all_ok;
      asm volatile(
          "{\n .reg .pred a, b;\n setp.ne.u32 a, %1, 0;\n bar.red.and.pred b, 1, 256, a;\n"
          " selp.u32 %0, 1, 0, b;\n}"
          : "=r"(all_ok)
          : "r"(ok)
          : "memory");
      if (!all_ok) {
        s_abort = 1;
        set_flag(p.flags, kFlagTimeout);
        break;
      }
      tmem_fence_after();
      const int vocab = (T0 + j) * kLmPairBV + (int)rank * kLmBV + 32 * q + lane;
      const bool valid = vocab < p.V;
      // one 32-column block's reduction (or, for the logits, its stores)
      auto block = [&](const int cb, const uint32_t (&r)[32]) {
        if constexpr (Mode == kLmArgmax) {
          float v[32];
          int ix[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            v[c] = valid ? __uint_as_float(r[c]) : -INFINITY;
            ix[c] = valid ? vocab : 0x7FFFFFFF;
          }
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) {
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int jj = 0; jj < off; ++jj) {
              const float send_v = upper ? v[jj] : v[jj + off];
              const int send_i = upper ? ix[jj] : ix[jj + off];
              const float keep_v = upper ? v[jj + off] : v[jj];
              const int keep_i = upper ? ix[jj + off] : ix[jj];
              const float got_v = __shfl_xor_sync(0xffffffffu, send_v, off);
              const int got_i = __shfl_xor_sync(0xffffffffu, send_i, off);
              const bool take = lm_better(got_v, got_i, keep_v, keep_i);
              v[jj] = take ? got_v : keep_v;
              ix[jj] = take ? got_i : keep_i;
            }
          }
          red_v[q][cb * 32 + lane] = v[0];
          red_i[q][cb * 32 + lane] = ix[0];
        } else if constexpr (Mode == kLmStats) {
          float z[32], v[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            z[c] = valid ? __uint_as_float(r[c]) : -INFINITY;
            v[c] = z[c];
          }
          // the draft token's logit, from the lane that holds it
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int col = cb * 32 + c;
            if (valid && s_tok[col] == vocab && row0 + col < nrows)
              p.zx[lm_sample_row(p, second, row0 + col)] = z[c];
          }
          // per column: the quadrant's integer reference, then its sum
          lane_butterfly(v, [](float a, float b) { return fmaxf(a, b); });
          const int ref = exp_ref(v[0], p.scale);  // column (cb*32 + lane)
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float nref = -(float)__shfl_sync(0xffffffffu, ref, c);
            v[c] = ex2(__fmaf_rn(z[c], p.scale, nref));  // 2^-inf = 0 past the vocabulary
          }
          lane_butterfly(v, [](float a, float b) { return __fadd_rn(a, b); });
          red_v[q][cb * 32 + lane] = v[0];
          red_i[q][cb * 32 + lane] = ref;
        } else {
          // the logits: for each column (row) the warp's 32 lanes store 32
          // consecutive vocabulary entries
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int lr = row0 + cb * 32 + c;
            if (valid && lr < nrows)
              p.logits[(size_t)lr * p.V + vocab] = __uint_as_float(r[c]);
          }
        }
      };
      const uint32_t qbase = tmem_base + ((uint32_t)(32 * q) << 16);
      if (Mode == kLmArgmax && nmma == 2) {
        // Each warp loads all its blocks of a slot (at most three), waits
        // once and frees the slot before reducing them: the slot of the
        // first MMA is the one the next tile's second MMA waits for.  (The
        // statistics epilogue, with its larger register state, keeps the
        // per-block order below, which measured faster there.)
        for (int m = 0; m < 2; ++m) {
          const int slot = (j * 2 + m) % nslots;
          const int lo = m * nblk, hi = lo + nblk;
          const int c0 = lo + ((lo & 1) != cb0 ? 1 : 0), c1 = c0 + 2, c2 = c0 + 4;
          const uint32_t sbase = qbase + (uint32_t)(slot * nper - lo * 32);
          uint32_t r0[32], r1[32], r2[32];
          tmem_ld32_async(sbase + (uint32_t)(c0 * 32), r0);
          if (c1 < hi) tmem_ld32_async(sbase + (uint32_t)(c1 * 32), r1);
          if (c2 < hi) tmem_ld32_async(sbase + (uint32_t)(c2 * 32), r2);
          tmem_wait_ld(r0);
          if (c1 < hi) tmem_wait_ld(r1);
          if (c2 < hi) tmem_wait_ld(r2);
          tmem_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(slot_empty0 + 8u * (uint32_t)slot);
          block(c0, r0);
          if (c1 < hi) block(c1, r1);
          if (c2 < hi) block(c2, r2);
        }
      } else {
        for (int cb = cb0; cb < ncb; cb += 2) {
          const int m = cb / nblk, cbl = cb - m * nblk;
          const int slot = (j * nmma + m) % nslots;
          uint32_t r[32];
          tmem_ld32(qbase + (uint32_t)(slot * nper + cbl * 32), r);
          if (cbl >= nblk - 2) {  // this warp's last block of the slot
            // the slot is read (the load has completed): its next tile may start
            tmem_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(slot_empty0 + 8u * (uint32_t)slot);
          }
          block(cb, r);
        }
      }
      if constexpr (Mode != kLmLogits) {
        asm volatile("bar.sync 1, 256;" ::: "memory");  // the four quadrants' results are in
#pragma unroll
        for (int jj = 0; jj < kPer; ++jj) {
          const int c = e + kLmEpiThreads * jj;
          if (c < R) {
            if constexpr (Mode == kLmArgmax) {
#pragma unroll
              for (int qq = 0; qq < 4; ++qq)
                if (lm_better(red_v[qq][c], red_i[qq][c], best[jj], bidx[jj])) {
                  best[jj] = red_v[qq][c];
                  bidx[jj] = red_i[qq][c];
                }
            } else {
              // the tile's partial of this row: the four quadrants rescaled
              // (exactly, powers of two) to their largest reference
              int tref = kRefEmpty;
#pragma unroll
              for (int qq = 0; qq < 4; ++qq) tref = max(tref, red_i[qq][c]);
              float tsum = 0.0f;
#pragma unroll
              for (int qq = 0; qq < 4; ++qq)
                tsum = __fadd_rn(tsum, red_v[qq][c] * pow2i_f(red_i[qq][c] - tref));
              if (tref > run[jj].ref) {
                run[jj].acc.scale(pow2i_f(run[jj].ref - tref));
                run[jj].ref = tref;
              }
              run[jj].acc.add(tsum * pow2i_f(tref - run[jj].ref));
            }
          }
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");  // the scratch may be reused
      }
    }
    const int C = gridDim.x;
#pragma unroll
    for (int jj = 0; jj < kPer; ++jj) {
      const int lr = row0 + e + kLmEpiThreads * jj;
      if (e + kLmEpiThreads * jj < R && lr < nrows) {
        if constexpr (Mode == kLmArgmax) {
          p.part[(size_t)lr * C + blockIdx.x] = ArgPartial{best[jj], bidx[jj], nsteps > 0 ? 1 : 0, 0};
        } else if constexpr (Mode == kLmStats) {
          SoftmaxPartial sp;
          sp.ref = run[jj].ref;
          sp.nch = nsteps > 0 ? 1 : 0;
          sp.hi = run[jj].acc.hi;
          sp.lo = run[jj].acc.lo;
          p.spart[(size_t)lm_sample_row(p, second, lr) * C + blockIdx.x] = sp;
        }
      }
    }
  }
  // neither CTA frees its tensor memory or leaves while the leader's MMAs
  // or the peer's epilogue may still use it
  tmem_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tmem_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kLmTmemCols)
                 : "memory");
  }
}

// LM head fused with sampling verification, between the statistics GEMM and
// the recomputation of the drawn rows: one CTA per sequence merges its rows'
// records, runs the accept test, and copies the hidden states of the rows
// the draw needs into hbuf [2B, d] (row 2b: the target row of the drawn
// position, 2b + 1: its draft row, zero for the bonus draw).
__global__ void __launch_bounds__(kThreads) lm_sample_gather_kernel(const SampleParams p,
                                                                    const uint16_t* h_target,
                                                                    const uint16_t* h_draft,
                                                                    uint16_t* hbuf, int d) {
  __shared__ RowStats s_rows[kMaxSeqRows];
  __shared__ int s_n;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the statistics records
  asm volatile("griddepcontrol.launch_dependents;");
  const int b = blockIdx.x, warp = threadIdx.x >> 5;
  const int rows_per_seq = 2 * p.k + 1;
  for (int r = warp; r < rows_per_seq; r += kWarps)
    finalize_stats_row<F32>(p, b * rows_per_seq + r, &s_rows[r]);
  __syncthreads();
  if (warp == 0) {
    const DrawDesc dd = resolve_sample_seq(p, b, [&](int r) { return s_rows[r]; }, false);
    if ((threadIdx.x & 31) == 0) s_n = dd.n;
  }
  __syncthreads();
  const int n = s_n;
  const uint4* src_t =
      reinterpret_cast<const uint4*>(h_target + ((size_t)b * (p.k + 1) + n) * (size_t)d);
  const uint4* src_d =
      n < p.k ? reinterpret_cast<const uint4*>(h_draft + ((size_t)b * p.k + n) * (size_t)d)
              : nullptr;
  uint4* dst_t = reinterpret_cast<uint4*>(hbuf + (size_t)(2 * b) * d);
  uint4* dst_d = reinterpret_cast<uint4*>(hbuf + (size_t)(2 * b + 1) * d);
  for (int i = threadIdx.x; i < d / 8; i += kThreads) {
    dst_t[i] = src_t[i];
    dst_d[i] = src_d ? src_d[i] : make_uint4(0, 0, 0, 0);
  }
}

}  // namespace sv
