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
//   Z tile^T = W_LM[v0 : v0+128, :] x H[rows, :]^T   (both K-major, bf16)
//
// The vocabulary is the MMA's M (128 tensor-memory lanes per tile) and the
// rows are its N (up to 384 columns, one or two MMAs of N <= 256), so rows
// are padded only to a multiple of 64.  One CTA per SM walks a contiguous
// range of vocabulary tiles for a group of rows; every CTA loads its own
// operands (no cluster, no multicast).  Warp roles (192 threads):
//   warp 0     TMA producer: per 64-wide K step, the tile's W slice and the
//              rows' H slice (128-byte swizzled) into a 3-stage ring
//   warp 1     allocates tensor memory; lane 0 issues tcgen05.mma
//              (M=128, N=rows/2 or rows, K=16) into a 128 x rows fp32
//              accumulator and commits stage releases and tile completion
//   warps 2-5  epilogue: tcgen05.ld of their 32-lane quadrant, a butterfly
//              reduction across lanes per column (row), a merge of the four
//              quadrants in shared memory and a running argmax per row
//              (lowest index wins ties); the accumulator is released as
//              soon as it has been read
// Each CTA writes one argmax record per row for its vocabulary segment, in
// the layout the greedy resolve kernel merges.  Every wait is bounded.
#pragma once

#include <cuda.h>

#include "sv_kernels.cuh"

namespace sv {

constexpr int kLmBV = 128;         // vocabulary per tile (UMMA M, tensor-memory lanes)
constexpr int kLmMaxRows = 384;    // rows per row group (UMMA N total, tensor-memory columns;
                                   // three stages of 16 KB + 48 KB fit in shared memory)
constexpr int kLmMaxN = 256;       // N of one MMA instruction
constexpr int kLmBK = 64;          // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kLmStages = 3;
constexpr int kLmThreads = 192;
constexpr int kLmABytes = kLmBV * kLmBK * 2;          // 16 KB: W slice
constexpr int kLmBBytes = kLmMaxRows * kLmBK * 2;     // up to 48 KB: H slice
constexpr int kLmHBox = 64;                           // rows per H box (TMA)
constexpr int kLmTmemCols = 512;

// What the epilogue makes of each accumulator tile.
enum LmMode : int {
  kLmArgmax = 0,  // running (max, lowest index) per row: greedy verification
  kLmStats = 1,   // running softmax partial per row and the draft token's logit: sampling
  kLmLogits = 2,  // the logits themselves, fp32 (the rows a sampling draw re-reads)
};

struct LmHeadParams {
  int rows, d, V;       // rows of the first matrix (argmax: B * (k+1))
  int ntiles;           // ceil(V / kLmBV)
  int grp_rows;         // rows per row group of the first matrix (multiple of kLmHBox)
  int stage_bytes;      // kLmABytes + grp_rows * 128 (the largest group)
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

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
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
__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap map_h,
                  const __grid_constant__ CUtensorMap map_h1,
                  const __grid_constant__ CUtensorMap map_w, const LmHeadParams p) {
  extern __shared__ uint8_t lm_raw[];
  __shared__ uint64_t full[kLmStages], empty[kLmStages];
  __shared__ uint64_t acc_full, acc_empty, drain;
  __shared__ uint32_t tmem_base_holder;
  __shared__ int s_abort;
  __shared__ float red_v[4][kLmMaxRows];  // per-quadrant column results of one tile
  __shared__ int red_i[4][kLmMaxRows];
  __shared__ int s_tok[kLmMaxRows];       // kLmStats: the draft token of each column (row)

  // 1024-byte aligned operand ring (128-byte swizzle atoms)
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(lm_raw) + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the CTA's row group: of the first matrix, or (sampling) of the second
  const bool second = (int)blockIdx.y >= p.ngroups0;
  const int R = second ? p.grp_rows1 : p.grp_rows;  // columns used (rows past the end read as 0)
  const int row0 = second ? ((int)blockIdx.y - p.ngroups0) * p.grp_rows1 : blockIdx.y * p.grp_rows;
  const int nrows = second ? p.rows1 : p.rows;
  const CUtensorMap* hmap = second ? &map_h1 : &map_h;
  const int stage_bytes = kLmABytes + R * 128;
  // the CTA owns the vocabulary tiles [T0, T1)
  int T0, T1;
  {
    const long long G = gridDim.x, g = blockIdx.x;
    T0 = (int)((long long)p.ntiles * g / G);
    T1 = (int)((long long)p.ntiles * (g + 1) / G);
  }
  const int nsteps = T1 - T0;
  const int nk = (p.d + kLmBK - 1) / kLmBK;
  const int nmma = (R + kLmMaxN - 1) / kLmMaxN;  // MMAs per K step of 16
  const int nper = R / nmma;                     // N of each (a multiple of 16)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kLmStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);  // released by the MMAs that read the stage
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, 4);
    mbar_init(&drain, 1);
    s_abort = 0;
    mbar_init_fence();
  }
  if (warp == 1) {  // tensor memory for the accumulators (whole warp)
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
            smem_addr(&tmem_base_holder)),
        "r"(kLmTmemCols)
        : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tmem_fence_before();
  __syncthreads();
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
    // ---------------- TMA producer ----------------
    int stage = 0, issued = 0;
    unsigned phase = 0;
    const unsigned bytes = (unsigned)stage_bytes;
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
        mbar_expect_tx(&full[stage], bytes);
        tma_load_2d(st, &map_w, kb * kLmBK, t * kLmBV, &full[stage]);
        for (int r = 0; r < R; r += kLmHBox)
          tma_load_2d(st + kLmABytes + r * 128, hmap, kb * kLmBK, row0 + r, &full[stage]);
        if (++stage == kLmStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // every copy this thread issued has landed before the CTA can leave
    for (int j = max(0, issued - kLmStages); j < issued; ++j)
      mbar_wait_bounded(&full[j % kLmStages], (unsigned)((j / kLmStages) & 1));
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = umma_idesc_bf16_f32(kLmBV, nper);
    int stage = 0;
    unsigned phase = 0, acc_phase = 0;
    for (int j = 0; j < nsteps && !*(volatile int*)&s_abort; ++j) {
      if (!mbar_wait_bounded(&acc_empty, acc_phase ^ 1u)) {
        s_abort = 1;
        set_flag(p.flags, kFlagTimeout);
        break;
      }
      tmem_fence_after();
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait_bounded(&full[stage], phase)) {
          s_abort = 1;
          set_flag(p.flags, kFlagTimeout);
          break;
        }
        tmem_fence_after();
        const uint32_t ast = smem_addr(ring + (size_t)stage * p.stage_bytes);
        const uint32_t bst = ast + kLmABytes;
#pragma unroll
        for (int kk = 0; kk < kLmBK / 16; ++kk)
          for (int m = 0; m < nmma; ++m)
            umma_bf16(tmem_base + m * nper, umma_desc_sw128(ast + kk * 32),
                      umma_desc_sw128(bst + m * nper * 128 + kk * 32), idesc,
                      (kb > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&empty[stage]);  // the stage is free once these finish
        if (++stage == kLmStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      umma_commit(&acc_full);  // the tile's accumulators are complete
      acc_phase ^= 1u;
    }
    // every MMA this thread issued has completed before tensor memory is freed
    umma_commit(&drain);
    mbar_wait_bounded(&drain, 0);
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    // Accumulator lane = vocabulary entry of the tile, column = row.  Argmax
    // and statistics reduce each warp's 32 lanes per column with a butterfly
    // that leaves column c's result in lane c; the four quadrants' results
    // meet in shared memory and each epilogue thread keeps the running
    // result of rows e, e + 128, ... over the CTA's tiles.
    const int q = warp & 3;   // tensor-memory lane quadrant of this warp
    const int e = threadIdx.x - 64;  // 0..127 among the epilogue threads
    float best[kLmMaxRows / 128];
    int bidx[kLmMaxRows / 128];
    StatsState run[kLmMaxRows / 128];
#pragma unroll
    for (int j = 0; j < kLmMaxRows / 128; ++j) {
      best[j] = -INFINITY;
      bidx[j] = 0x7FFFFFFF;
    }
    unsigned acc_phase = 0;
    for (int j = 0; j < nsteps; ++j) {
      // every epilogue thread takes the same decision, so none is left at a
      // named barrier the others no longer reach
      const unsigned ok = mbar_wait_bounded(&acc_full, acc_phase) ? 1u : 0u;
      unsigned all_ok;
      asm volatile(
          "{\n .reg .pred a, b;\n setp.ne.u32 a, %1, 0;\n bar.red.and.pred b, 1, 128, a;\n"
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
      const int vocab = (T0 + j) * kLmBV + 32 * q + lane;
      const bool valid = vocab < p.V;
      for (int cb = 0; cb < R / 32; ++cb) {
        uint32_t r[32];
        tmem_ld32(tmem_base + ((uint32_t)(32 * q) << 16) + cb * 32, r);
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
      }
      tmem_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty);  // tensor memory read: next tile may start
      if constexpr (Mode != kLmLogits) {
        asm volatile("bar.sync 1, 128;" ::: "memory");  // the four quadrants' results are in
#pragma unroll
        for (int jj = 0; jj < kLmMaxRows / 128; ++jj) {
          const int c = e + 128 * jj;
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
        asm volatile("bar.sync 1, 128;" ::: "memory");  // the scratch may be reused
      }
      acc_phase ^= 1u;
    }
    const int C = gridDim.x;
#pragma unroll
    for (int jj = 0; jj < kLmMaxRows / 128; ++jj) {
      const int lr = row0 + e + 128 * jj;
      if (e + 128 * jj < R && lr < nrows) {
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
  tmem_fence_before();
  __syncthreads();
  if (warp == 1) {
    tmem_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
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
