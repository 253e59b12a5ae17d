// spec_verify.cu -- C ABI of libspecverify (declared in include/spec_verify.h):
// host-side argument checks, workspace layout and kernel launches.
//
// Workspace layout (all offsets 256-byte aligned):
//   [0, 256)     header; word 0 = sticky device flag bits
//   [256, ...)   per-call scratch records; every record a kernel reads was
//                written earlier in the same call, so the contents on entry
//                do not matter and calls of any shape can share a workspace.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "spec_verify.h"
#include "sv_kernels.cuh"
#include "sv_tree.cuh"
#include "sv_lmhead.cuh"
#include "sv_grow.cuh"

static_assert(sv::kMaxDraft == SPEC_MAX_K, "finish kernel buffers are sized for SPEC_MAX_K");

namespace {

std::atomic<uint64_t> g_launches{0};
// limit of the verification kernels' waits on their bulk copies
// (spec_verify_set_wait_limit_ns)
std::atomic<uint64_t> g_wait_limit_ns{sv::kWaitLimitNs};

constexpr size_t kAlign = 256;
constexpr size_t kHeaderBytes = 256;
constexpr size_t kDataOffset = kHeaderBytes;
constexpr int kLmMaxGrid = 1024;  // CTAs (records per row) of the fused LM-head kernel

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int elem_bytes(int dtype) { return dtype == SPEC_DTYPE_BF16 ? 2 : 4; }
int chunk_elems(int dtype) {
  return dtype == SPEC_DTYPE_BF16 ? sv::BF16::kChunk : sv::F32::kChunk;
}

struct Layout {
  size_t bytes = 0;
  int rows = 0, nchunks = 0;
  size_t off_part = 0, off_desc = 0, off_csum = 0, off_csum_p = 0, off_zx = 0;  // sample
  size_t off_gsum = 0, off_gsum_p = 0;
  size_t off_arg = 0;                                            // greedy / tree
  size_t off_log = 0;  // LM head + sampling: the drawn rows' logits
};

// Returns false for arguments outside the documented limits.
bool make_layout(int mode, int B, int kN, int V, int dtype, Layout* L) {
  if (mode == SPEC_MODE_TREE_MASK || mode == SPEC_MODE_KV_COMMIT) {  // the flag header only
    if (B < 0 || kN < 1 || kN > SPEC_MAX_TREE_NODES) return false;
    L->bytes = kHeaderBytes;
    return true;
  }
  if (mode == SPEC_MODE_TREE_GROW) {  // kN = K (children per node); records and node arrays
    const int K = kN;
    if (B < 0 || K < 1 || K > sv::kGrowMaxK || V < K || V > SPEC_MAX_V) return false;
    if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return false;
    const int C = (V + chunk_elems(dtype) - 1) / chunk_elems(dtype);
    if ((long long)C * K > sv::kGrowMaxCand) return false;
    L->nchunks = C;
    size_t off = kDataOffset;
    L->off_part = off;  // GrowRec [B, 1 + (kGrowMaxD - 1) K, C]: every row of up to 16 layers
    off = align_up(off + (size_t)B * (1 + (sv::kGrowMaxD - 1) * K) * C * sizeof(sv::GrowRec));
    L->off_desc = off;  // node values, float64 [B, kGrowMaxNodes]
    off = align_up(off + (size_t)B * sv::kGrowMaxNodes * sizeof(double));
    L->off_gsum = off;  // parent, token, depth [3][B, kGrowMaxNodes]
    off = align_up(off + 3 * (size_t)B * sv::kGrowMaxNodes * sizeof(int32_t));
    L->bytes = off;
    return true;
  }
  if (mode == SPEC_MODE_LM_HEAD_SAMPLE) {
    // statistics records of up to kLmMaxGrid CTAs per row, captured token
    // logits, the draw's structures over fp32 rows, the drawn rows' hidden
    // states [2B, d <= SPEC_LM_MAX_D] and their logits [2B, V] fp32
    if (B < 0 || kN < 0 || kN > SPEC_MAX_K || V < 1 || V > SPEC_MAX_V) return false;
    const long long rows = (long long)B * (2LL * kN + 1);
    if (rows * kLmMaxGrid > 0x7FFFFFFFLL) return false;
    const int C = (V + sv::F32::kChunk - 1) / sv::F32::kChunk;
    if ((long long)B * C * sv::kVecPerChunk > 0x7FFFFFFFLL) return false;
    L->rows = (int)rows;
    L->nchunks = C;
    size_t off = kDataOffset;
    L->off_part = off;
    off = align_up(off + (size_t)rows * kLmMaxGrid * sizeof(sv::SoftmaxPartial));
    L->off_zx = off;
    off = align_up(off + (size_t)rows * sizeof(float));
    L->off_desc = off;
    off = align_up(off + (size_t)B * sizeof(sv::DrawDesc));
    const size_t bc = (size_t)B * C;
    L->off_csum = off;
    off = align_up(off + bc * sizeof(sv::FSum));
    L->off_csum_p = off;
    off = align_up(off + bc * sizeof(sv::FSum));
    L->off_gsum = off;
    off = align_up(off + bc * sv::kVecPerChunk * sizeof(float));
    L->off_gsum_p = off;
    off = align_up(off + bc * sv::kVecPerChunk * sizeof(float));
    L->off_arg = off;
    off = align_up(off + (size_t)2 * B * SPEC_LM_MAX_D * sizeof(uint16_t));
    L->off_log = off;
    off = align_up(off + (size_t)2 * B * V * sizeof(float));
    L->bytes = off;
    return true;
  }
  if (mode == SPEC_MODE_LM_HEAD_GREEDY) {  // argmax records of up to kLmMaxGrid CTAs per row
    if (B < 0 || kN < 0 || kN > SPEC_MAX_K || V < 1 || V > SPEC_MAX_V) return false;
    const long long rows = (long long)B * (kN + 1);
    if (rows * kLmMaxGrid > 0x7FFFFFFFLL) return false;
    L->rows = (int)rows;
    L->nchunks = kLmMaxGrid;
    size_t off = kDataOffset;
    L->off_part = off;
    off = align_up(off + (size_t)rows * kLmMaxGrid * sizeof(sv::ArgPartial));
    L->off_arg = off;
    off = align_up(off + (size_t)rows * sizeof(int32_t));
    L->bytes = off;
    return true;
  }
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return false;
  if (B < 0 || V < 1 || V > SPEC_MAX_V) return false;
  const int C = (V + chunk_elems(dtype) - 1) / chunk_elems(dtype);
  long long rows;
  if (mode == SPEC_MODE_SAMPLE) {
    if (kN < 0 || kN > SPEC_MAX_K) return false;
    rows = (long long)B * (2LL * kN + 1);
  } else if (mode == SPEC_MODE_GREEDY) {
    if (kN < 0 || kN > SPEC_MAX_K) return false;
    rows = (long long)B * (kN + 1LL);
  } else if (mode == SPEC_MODE_TREE_GREEDY) {
    if (kN < 1 || kN > SPEC_MAX_TREE_NODES) return false;
    rows = (long long)B * kN;
  } else {
    return false;
  }
  if (rows * C > 0x7FFFFFFFLL || (long long)B * C * sv::kVecPerChunk > 0x7FFFFFFFLL) return false;
  L->rows = (int)rows;
  L->nchunks = C;
  size_t off = kDataOffset;
  if (mode == SPEC_MODE_SAMPLE) {
    L->off_part = off;
    off = align_up(off + (size_t)rows * C * sizeof(sv::SoftmaxPartial));
    L->off_desc = off;
    off = align_up(off + (size_t)B * sizeof(sv::DrawDesc));
    const size_t bc = (size_t)B * C;
    L->off_csum = off;
    off = align_up(off + bc * sizeof(sv::FSum));
    L->off_csum_p = off;
    off = align_up(off + bc * sizeof(sv::FSum));
    L->off_gsum = off;
    off = align_up(off + bc * sv::kVecPerChunk * sizeof(float));
    L->off_gsum_p = off;
    off = align_up(off + bc * sv::kVecPerChunk * sizeof(float));
    L->off_zx = off;
    off = align_up(off + (size_t)rows * sizeof(float));
  } else {
    L->off_part = off;
    off = align_up(off + (size_t)rows * C * sizeof(sv::ArgPartial));
    L->off_arg = off;
    off = align_up(off + (size_t)rows * sizeof(int32_t));
  }
  L->bytes = off;
  return true;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// 16-byte vector path: base aligned and every row a whole number of vectors.
bool vec_ok(const void* p, int V, int dtype) {
  return aligned(p, 16) && ((size_t)V * elem_bytes(dtype)) % 16 == 0;
}

template <typename KernelT, typename ParamT>
spec_status_t launch(KernelT kernel, int grid, size_t smem, const ParamT& prm, void* stream,
                     bool pdl, int cluster = 1, int threads = sv::kThreads) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = na ? attr : nullptr;
  cfg.numAttrs = na;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, prm);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return SPEC_OK;
}

// Launch configuration of a programmatic dependent launch (the kernel waits
// for the preceding kernel in the stream with griddepcontrol.wait).
void pdl_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, dim3 grid, dim3 block,
                size_t smem, void* stream) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = grid;
  cfg->blockDim = block;
  cfg->dynamicSmemBytes = smem;
  cfg->stream = (cudaStream_t)stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
}

// Per-device state the library caches (shared-memory opt-ins, launch shapes,
// the no-allocation array's address) belongs to the device's current context:
// each cache entry records the context's unique id and is redone when the id
// changes (after cudaDeviceReset, for example).
constexpr int kMaxDevices = 64;
constexpr size_t kStreamSmem = (size_t)sv::kStages * sv::kChunkBytes;
std::mutex g_shape_mu;
std::mutex g_ctx_mu;
CUresult (*g_ctx_current)(CUcontext*) = nullptr;
CUresult (*g_ctx_id)(CUcontext, unsigned long long*) = nullptr;

// The current device and the unique id of its (primary) context, creating
// that context if the runtime has not yet done so.
spec_status_t current_context(int* dev, unsigned long long* id) {
  if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return SPEC_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(g_ctx_mu);
    if (!g_ctx_current || !g_ctx_id) {
      void* f1 = nullptr;
      void* f2 = nullptr;
      cudaDriverEntryPointQueryResult q1, q2;
      if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 4000, cudaEnableDefault,
                                           &q1) != cudaSuccess ||
          q1 != cudaDriverEntryPointSuccess || !f1 ||
          cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
              cudaSuccess ||
          q2 != cudaDriverEntryPointSuccess || !f2)
        return SPEC_ERR_CUDA;
      g_ctx_current = reinterpret_cast<CUresult (*)(CUcontext*)>(f1);
      g_ctx_id = reinterpret_cast<CUresult (*)(CUcontext, unsigned long long*)>(f2);
    }
  }
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return SPEC_ERR_CUDA;
  if (ctx == nullptr) {  // the runtime has not made the device's context current yet
    if (cudaSetDevice(*dev) != cudaSuccess || g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx)
      return SPEC_ERR_CUDA;
  }
  return g_ctx_id(ctx, id) == CUDA_SUCCESS ? SPEC_OK : SPEC_ERR_CUDA;
}

// Per-device launch shape of a persistent streaming kernel: the shared-memory
// opt-in is set once per device context, the grid is SMs x resident CTAs per
// SM.
template <auto kernel>
spec_status_t persistent_grid(int items, int* grid) {
  static int cached[kMaxDevices] = {0};  // one table per kernel instantiation
  static unsigned long long cached_ctx[kMaxDevices] = {0};
  int dev = 0;
  unsigned long long ctx = 0;
  if (current_context(&dev, &ctx) != SPEC_OK) return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_shape_mu);
  if (cached[dev] == 0 || cached_ctx[dev] != ctx) {
    int sms = 0, per_sm = 0;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kStreamSmem) != cudaSuccess)
      return SPEC_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SPEC_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, sv::kThreads,
                                                      kStreamSmem) != cudaSuccess)
      return SPEC_ERR_CUDA;
    cached[dev] = std::max(1, sms * std::max(1, per_sm));
    cached_ctx[dev] = ctx;
  }
  *grid = std::min(items, cached[dev]);
  return SPEC_OK;
}

// Dynamic shared-memory opt-in for a kernel, once per device context.
template <auto kernel>
spec_status_t ensure_smem(size_t bytes) {
  static bool done[kMaxDevices] = {false};
  static unsigned long long done_ctx[kMaxDevices] = {0};
  int dev = 0;
  unsigned long long ctx = 0;
  if (current_context(&dev, &ctx) != SPEC_OK) return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_shape_mu);
  if (!done[dev] || done_ctx[dev] != ctx) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
        cudaSuccess)
      return SPEC_ERR_CUDA;
    done[dev] = true;
    done_ctx[dev] = ctx;
  }
  return SPEC_OK;
}

// TMA descriptor of a row-major bf16 matrix [outer, inner] read as K-major
// boxes of 64 x box_outer with 128-byte swizzle (out-of-range rows and
// columns read as zero).  The driver's encoder is looked up once.
std::mutex g_encode_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

spec_status_t encode_bf16_kmajor(CUtensorMap* map, const void* base, int inner, int outer,
                                 int box_outer) {
  {
    std::lock_guard<std::mutex> lock(g_encode_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return SPEC_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  const cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  const cuuint32_t box[2] = {(cuuint32_t)sv::kLmBK, (cuuint32_t)box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SPEC_OK : SPEC_ERR_INVALID_ARG;
}

// Row groups of an LM-head GEMM: at most kLmMaxRows rows each, split evenly,
// each a multiple of the 64-row H box (so two MMAs of equal N stay multiples
// of 16).  Returns false when the rows need more groups than a grid allows.
bool lm_row_groups(int rows, int* ngroups, int* grp) {
  if (rows <= 0) {
    *ngroups = 0;
    *grp = sv::kLmHBox;
    return true;
  }
  const int gy = (rows + sv::kLmMaxRows - 1) / sv::kLmMaxRows;
  if (gy > 32768) return false;
  *ngroups = gy;
  *grp = ((rows + gy - 1) / gy + sv::kLmHBox - 1) / sv::kLmHBox * sv::kLmHBox;
  return true;
}

// One CTA per SM (the kernel holds the SM's tensor memory and most of its
// shared memory), in pairs: as many pairs as can be resident at once, at most
// one per 256-entry vocabulary tile.  The number of co-resident pairs is
// asked of the runtime once per device and context.
template <int Mode>
spec_status_t lm_grid_x(int ntiles, int* gx) {
  static int pairs_cached[kMaxDevices] = {0};
  static unsigned long long pairs_ctx[kMaxDevices] = {0};
  int dev = 0;
  unsigned long long ctx = 0;
  if (current_context(&dev, &ctx) != SPEC_OK) return SPEC_ERR_CUDA;
  int pairs = 0;
  {
    std::lock_guard<std::mutex> lock(g_shape_mu);
    if (pairs_ctx[dev] == ctx && pairs_cached[dev] > 0) pairs = pairs_cached[dev];
  }
  if (pairs == 0) {
    // the occupancy query sees the kernel's shared-memory opt-in
    const spec_status_t st = ensure_smem<sv::lmhead_kernel<Mode>>((size_t)sv::kLmRingBytes + 1024);
    if (st != SPEC_OK) return st;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SPEC_ERR_CUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(2 * std::max(1, sms / 2)), 1, 1);
    cfg.blockDim = dim3(sv::kLmThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)sv::kLmRingBytes + 1024;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, sv::lmhead_kernel<Mode>, &cfg) != cudaSuccess)
      return SPEC_ERR_CUDA;
    pairs = std::max(1, std::min(clusters, sms / 2));
    std::lock_guard<std::mutex> lock(g_shape_mu);
    pairs_cached[dev] = pairs;
    pairs_ctx[dev] = ctx;
  }
  *gx = 2 * std::max(1, std::min(std::min(pairs, ntiles), kLmMaxGrid / 2));
  return SPEC_OK;
}

template <int Mode>
spec_status_t launch_lmhead(const CUtensorMap& map_h, const CUtensorMap& map_h1,
                            const CUtensorMap& map_w, const sv::LmHeadParams& lp, int gx, int gy,
                            void* stream) {
  const spec_status_t st =
      ensure_smem<sv::lmhead_kernel<Mode>>((size_t)sv::kLmRingBytes + 1024);
  if (st != SPEC_OK) return st;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  pdl_config(&cfg, attr, dim3((unsigned)gx, (unsigned)gy, 1), dim3(sv::kLmThreads, 1, 1),
             (size_t)lp.nstages * lp.stage_bytes + 1024, stream);
  if (cudaLaunchKernelEx(&cfg, sv::lmhead_kernel<Mode>, map_h, map_h1, map_w, lp) != cudaSuccess)
    return SPEC_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return SPEC_OK;
}

template <typename E, bool kVec>
spec_status_t run_finish(const sv::SampleParams& prm, void* stream) {
  if (prm.nchunks <= sv::kClusterMaxChunks) {
    const spec_status_t st = ensure_smem<sv::sample_finish_kernel<E, kVec>>(sv::kFinishSmem);
    if (st != SPEC_OK) return st;
    return launch(sv::sample_finish_kernel<E, kVec>, prm.B * sv::kClusterCTAs, sv::kFinishSmem,
                  prm, stream, true, sv::kClusterCTAs);
  }
  const spec_status_t st =
      launch(sv::draw_kernel<E, kVec>, prm.B * prm.nchunks, 0, prm, stream, true);
  if (st != SPEC_OK) return st;
  return launch(sv::draw_resolve_kernel<E, kVec>, prm.B, 0, prm, stream, true);
}

// L2 budget for the rows streamed with a keep hint (well under the 129 MB L2
// of a GB300, so that the rest of the stream does not evict them).
constexpr double kKeepBytes = 80.0 * (1 << 20);

template <typename E>
spec_status_t run_sample(sv::SampleParams prm, int rows, bool vec, void* stream) {
  prm.items = rows * prm.nchunks;
  prm.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  {
    const double pair = 2.0 * prm.B * (double)prm.V * sizeof(typename E::storage);
    prm.keep_pos = pair > 0 ? std::min(prm.k + 1, (int)(kKeepBytes / pair)) : 0;
  }
  spec_status_t st;
  if (vec) {
    int grid = 0;
    st = persistent_grid<sv::stream_stats_kernel<E, false>>(prm.items, &grid);
    if (st != SPEC_OK) return st;
    if (prm.items / grid < sv::kFrontLoadItems) {  // short ranges: start before the wait
      st = persistent_grid<sv::stream_stats_kernel<E, true>>(prm.items, &grid);
      if (st != SPEC_OK) return st;
      st = launch(sv::stream_stats_kernel<E, true>, grid, kStreamSmem, prm, stream, true);
    } else {
      st = launch(sv::stream_stats_kernel<E, false>, grid, kStreamSmem, prm, stream, true);
    }
  } else {
    st = launch(sv::chunk_stats_kernel<E, false>, prm.items, 0, prm, stream, false);
  }
  if (st != SPEC_OK) return st;
  return vec ? run_finish<E, true>(prm, stream) : run_finish<E, false>(prm, stream);
}

template <typename E>
spec_status_t run_argmax(sv::ArgmaxParams prm, int rows, bool vec, void* stream) {
  prm.items = rows * prm.nchunks;
  prm.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  if (vec) {
    int grid = 0;
    spec_status_t st = persistent_grid<sv::stream_argmax_kernel<E>>(prm.items, &grid);
    if (st != SPEC_OK) return st;
    st = launch(sv::stream_argmax_kernel<E>, grid, kStreamSmem, prm, stream, true);
    if (st != SPEC_OK) return st;
  } else {
    const spec_status_t st =
        launch(sv::chunk_argmax_kernel<E, false>, prm.items, 0, prm, stream, false);
    if (st != SPEC_OK) return st;
  }
  return launch(sv::argmax_resolve_kernel, prm.B, 0, prm, stream, true);
}

// Scratch of spec_verify_greedy_noalloc: a fixed array in the library's own
// device memory (one copy per device that loads the library).  Host code may
// not use the symbol as an address; its device address is looked up with
// cudaGetSymbolAddress while the device is current, once per device context.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];
void* g_noalloc_addr[kMaxDevices] = {nullptr};
unsigned long long g_noalloc_ctx[kMaxDevices] = {0};
std::mutex g_noalloc_mu;

spec_status_t noalloc_scratch(void** addr) {
  int dev = 0;
  unsigned long long ctx = 0;
  if (current_context(&dev, &ctx) != SPEC_OK) return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr || g_noalloc_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return SPEC_ERR_CUDA;
    g_noalloc_addr[dev] = p;
    g_noalloc_ctx[dev] = ctx;
  }
  *addr = g_noalloc_addr[dev];
  return SPEC_OK;
}

}  // namespace

extern "C" {

size_t spec_verify_workspace_bytes(int mode, int B, int k_or_N, int V, int dtype) {
  Layout L;
  if (!make_layout(mode, B, k_or_N, V, dtype, &L)) return 0;
  return L.bytes;
}

spec_status_t spec_verify_sample(const void* target_logits, const void* draft_logits, int dtype,
                                 const int32_t* draft_tokens, const float* u_accept,
                                 const float* u_sample, float temperature, int B, int k, int V,
                                 int32_t* accepted_len, int32_t* out_tokens, float* p_out,
                                 float* q_out, float* resid_mass, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_INVALID_ARG;
  if (B < 0 || k < 0 || k > SPEC_MAX_K || V < 1 || V > SPEC_MAX_V) return SPEC_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return SPEC_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(SPEC_MODE_SAMPLE, B, k, V, dtype, &L)) return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!target_logits || !u_sample || !accepted_len || !out_tokens || !resid_mass)
    return SPEC_ERR_INVALID_ARG;
  if (k > 0 && (!draft_logits || !draft_tokens || !u_accept || !p_out || !q_out))
    return SPEC_ERR_INVALID_ARG;
  const int eb = elem_bytes(dtype);
  if (!aligned(target_logits, eb) || (k > 0 && !aligned(draft_logits, eb)))
    return SPEC_ERR_ALIGNMENT;
  if (!aligned(accepted_len, 4) || !aligned(out_tokens, 4) || !aligned(u_sample, 4) ||
      !aligned(resid_mass, 4) ||
      (k > 0 && (!aligned(draft_tokens, 4) || !aligned(u_accept, 4) || !aligned(p_out, 4) ||
                 !aligned(q_out, 4))))
    return SPEC_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < L.bytes) return SPEC_ERR_WORKSPACE;
  if (!aligned(workspace, kAlign)) return SPEC_ERR_ALIGNMENT;

  char* ws = static_cast<char*>(workspace);
  sv::SampleParams prm;
  prm.target = target_logits;
  prm.draft = draft_logits;
  prm.tokens = draft_tokens;
  prm.u_accept = u_accept;
  prm.u_sample = u_sample;
  prm.scale = (float)(1.4426950408889634 / (double)temperature);
  prm.B = B;
  prm.k = k;
  prm.V = V;
  prm.nchunks = L.nchunks;
  prm.accepted_len = accepted_len;
  prm.out_tokens = out_tokens;
  prm.p_out = p_out;
  prm.q_out = q_out;
  prm.resid_mass = resid_mass;
  prm.flags = reinterpret_cast<unsigned*>(ws);
  prm.part = reinterpret_cast<sv::SoftmaxPartial*>(ws + L.off_part);
  prm.desc = reinterpret_cast<sv::DrawDesc*>(ws + L.off_desc);
  prm.csum = reinterpret_cast<sv::FSum*>(ws + L.off_csum);
  prm.csum_p = reinterpret_cast<sv::FSum*>(ws + L.off_csum_p);
  prm.gsum = reinterpret_cast<float*>(ws + L.off_gsum);
  prm.gsum_p = reinterpret_cast<float*>(ws + L.off_gsum_p);
  prm.zx = reinterpret_cast<float*>(ws + L.off_zx);
  prm.nrec = L.nchunks;
  prm.drawn = nullptr;

  const bool vec = vec_ok(target_logits, V, dtype) && (k == 0 || vec_ok(draft_logits, V, dtype));
  if (dtype == SPEC_DTYPE_BF16) return run_sample<sv::BF16>(prm, L.rows, vec, stream);
  return run_sample<sv::F32>(prm, L.rows, vec, stream);
}

static spec_status_t argmax_common(sv::ArgmaxParams& prm, const Layout& L, void* workspace,
                                   int dtype, void* stream) {
  char* ws = static_cast<char*>(workspace);
  prm.flags = reinterpret_cast<unsigned*>(ws);
  prm.part = reinterpret_cast<sv::ArgPartial*>(ws + L.off_part);
  prm.rowarg = reinterpret_cast<int32_t*>(ws + L.off_arg);
  prm.nchunks = L.nchunks;
  const bool vec = vec_ok(prm.target, prm.V, dtype);
  if (dtype == SPEC_DTYPE_BF16) return run_argmax<sv::BF16>(prm, L.rows, vec, stream);
  return run_argmax<sv::F32>(prm, L.rows, vec, stream);
}

spec_status_t spec_verify_greedy(const void* target_logits, int dtype,
                                 const int32_t* draft_tokens, int B, int k, int V,
                                 int32_t* accepted_len, int32_t* out_tokens, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_INVALID_ARG;
  if (B < 0 || k < 0 || k > SPEC_MAX_K || V < 1 || V > SPEC_MAX_V) return SPEC_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(SPEC_MODE_GREEDY, B, k, V, dtype, &L)) return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!target_logits || !accepted_len || !out_tokens || (k > 0 && !draft_tokens))
    return SPEC_ERR_INVALID_ARG;
  if (!aligned(target_logits, elem_bytes(dtype)) || !aligned(accepted_len, 4) ||
      !aligned(out_tokens, 4) || (k > 0 && !aligned(draft_tokens, 4)))
    return SPEC_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < L.bytes) return SPEC_ERR_WORKSPACE;
  if (!aligned(workspace, kAlign)) return SPEC_ERR_ALIGNMENT;
  sv::ArgmaxParams prm;
  std::memset(&prm, 0, sizeof prm);
  prm.target = target_logits;
  prm.tokens = draft_tokens;
  prm.parents = nullptr;
  prm.B = B;
  prm.rows_per_seq = k + 1;
  prm.V = V;
  prm.tree = 0;
  prm.max_depth = 0;
  prm.accepted_len = accepted_len;
  prm.out_tokens = out_tokens;
  prm.path_nodes = nullptr;
  return argmax_common(prm, L, workspace, dtype, stream);
}

spec_status_t spec_verify_tree_greedy(const void* target_logits, int dtype,
                                      const int32_t* node_tokens, const int32_t* parents, int B,
                                      int N, int V, int max_depth, int32_t* accepted_len,
                                      int32_t* path_nodes, int32_t* out_tokens, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_INVALID_ARG;
  if (B < 0 || N < 1 || N > SPEC_MAX_TREE_NODES || V < 1 || V > SPEC_MAX_V)
    return SPEC_ERR_INVALID_ARG;
  if (max_depth < 0 || max_depth > SPEC_MAX_TREE_DEPTH) return SPEC_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(SPEC_MODE_TREE_GREEDY, B, N, V, dtype, &L)) return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!target_logits || !node_tokens || !parents || !accepted_len || !path_nodes || !out_tokens)
    return SPEC_ERR_INVALID_ARG;
  if (!aligned(target_logits, elem_bytes(dtype)) || !aligned(node_tokens, 4) ||
      !aligned(parents, 4) || !aligned(accepted_len, 4) || !aligned(path_nodes, 4) ||
      !aligned(out_tokens, 4))
    return SPEC_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < L.bytes) return SPEC_ERR_WORKSPACE;
  if (!aligned(workspace, kAlign)) return SPEC_ERR_ALIGNMENT;
  sv::ArgmaxParams prm;
  std::memset(&prm, 0, sizeof prm);
  prm.target = target_logits;
  prm.tokens = node_tokens;
  prm.parents = parents;
  prm.B = B;
  prm.rows_per_seq = N;
  prm.V = V;
  prm.tree = 1;
  prm.max_depth = max_depth;
  prm.accepted_len = accepted_len;
  prm.out_tokens = out_tokens;
  prm.path_nodes = path_nodes;
  return argmax_common(prm, L, workspace, dtype, stream);
}

spec_status_t spec_tree_attention_mask(const int32_t* parents, int B, int N, uint32_t* mask,
                                       int32_t* depth, void* workspace, size_t workspace_bytes,
                                       void* stream) {
  if (B < 0 || N < 1 || N > SPEC_MAX_TREE_NODES) return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!parents || !mask) return SPEC_ERR_INVALID_ARG;
  if (!aligned(parents, 4) || !aligned(mask, 4) || (depth && !aligned(depth, 4)))
    return SPEC_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < kHeaderBytes) return SPEC_ERR_WORKSPACE;
  if (!aligned(workspace, kAlign)) return SPEC_ERR_ALIGNMENT;
  const int W = (N + 31) / 32;
  const long long threads = (long long)B * N * W;
  const long long blocks = (threads + sv::kMaskThreads - 1) / sv::kMaskThreads;
  if (blocks > 0x7FFFFFFFLL) return SPEC_ERR_INVALID_ARG;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  pdl_config(&cfg, attr, dim3((unsigned)blocks), dim3(sv::kMaskThreads), 0, stream);
  if (cudaLaunchKernelEx(&cfg, sv::tree_mask_kernel, parents, B, N, W, mask, depth,
                         reinterpret_cast<unsigned*>(workspace)) != cudaSuccess)
    return SPEC_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return SPEC_OK;
}

spec_status_t spec_kv_commit_path(void* cache, int B, int planes, long long plane_stride,
                                  long long seq_stride, int entry_bytes, int L, int N,
                                  const int32_t* base_len, const int32_t* accepted_len,
                                  const int32_t* path_nodes, int max_depth, int32_t* new_len,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || planes < 1 || planes > 65535 || entry_bytes < 16 || L < 1 || N < 1 ||
      N > SPEC_MAX_TREE_NODES || max_depth < 0 || max_depth > SPEC_MAX_TREE_DEPTH ||
      plane_stride < 0 || seq_stride < 0)
    return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!cache || !base_len || !accepted_len || !path_nodes || !new_len)
    return SPEC_ERR_INVALID_ARG;
  if (!aligned(cache, 16) || entry_bytes % 16 || plane_stride % 16 || seq_stride % 16 ||
      !aligned(base_len, 4) || !aligned(accepted_len, 4) || !aligned(path_nodes, 4) ||
      !aligned(new_len, 4))
    return SPEC_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < kHeaderBytes) return SPEC_ERR_WORKSPACE;
  if (!aligned(workspace, kAlign)) return SPEC_ERR_ALIGNMENT;
  sv::KvCommitParams prm;
  prm.cache = static_cast<uint8_t*>(cache);
  prm.plane_stride = plane_stride;
  prm.seq_stride = seq_stride;
  prm.entry_bytes = entry_bytes;
  prm.L = L;
  prm.N = N;
  prm.max_depth = max_depth;
  prm.planes = planes;
  prm.base_len = base_len;
  prm.accepted_len = accepted_len;
  prm.path_nodes = path_nodes;
  prm.new_len = new_len;
  prm.flags = reinterpret_cast<unsigned*>(workspace);
  // stage every moved entry of a pass in at most 40 KB of dynamic shared
  // memory (under the 48 KB default with the kernel's static arrays)
  constexpr int kStageBytes = 40 * 1024;
  const int moves = std::max(1, std::min(max_depth, sv::kKvMaxMoves));
  prm.slice_bytes = std::min(entry_bytes, kStageBytes / moves / 16 * 16);
  const size_t smem = (size_t)prm.slice_bytes * moves;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  pdl_config(&cfg, attr, dim3((unsigned)B, (unsigned)planes), dim3(sv::kKvThreads), smem,
             stream);
  if (cudaLaunchKernelEx(&cfg, sv::kv_commit_kernel, prm) != cudaSuccess) return SPEC_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return SPEC_OK;
}

spec_status_t spec_lm_head_verify_greedy(const void* hidden, const void* w_lm,
                                         const int32_t* draft_tokens, int B, int k, int d, int V,
                                         int32_t* accepted_len, int32_t* out_tokens,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || k < 0 || k > SPEC_MAX_K || d < 8 || d > (1 << 20) || d % 8 || V < 1 ||
      V > SPEC_MAX_V)
    return SPEC_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(SPEC_MODE_LM_HEAD_GREEDY, B, k, V, SPEC_DTYPE_BF16, &L))
    return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!hidden || !w_lm || !accepted_len || !out_tokens || (k > 0 && !draft_tokens))
    return SPEC_ERR_INVALID_ARG;
  if (!aligned(hidden, 16) || !aligned(w_lm, 16) || !aligned(accepted_len, 4) ||
      !aligned(out_tokens, 4) || (k > 0 && !aligned(draft_tokens, 4)))
    return SPEC_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < L.bytes) return SPEC_ERR_WORKSPACE;
  if (!aligned(workspace, kAlign)) return SPEC_ERR_ALIGNMENT;
  const int rows = L.rows;
  const int ntiles = (V + sv::kLmPairBV - 1) / sv::kLmPairBV;
  int gy = 0, grp = 0, gx = 0;
  if (!lm_row_groups(rows, &gy, &grp)) return SPEC_ERR_INVALID_ARG;
  spec_status_t st = lm_grid_x<sv::kLmArgmax>(ntiles, &gx);
  if (st != SPEC_OK) return st;
  CUtensorMap map_h, map_w;
  st = encode_bf16_kmajor(&map_h, hidden, d, rows, sv::lm_half_rows(grp));
  if (st != SPEC_OK) return st;
  st = encode_bf16_kmajor(&map_w, w_lm, d, V, sv::kLmBV);
  if (st != SPEC_OK) return st;
  char* ws = static_cast<char*>(workspace);
  sv::LmHeadParams lp;
  std::memset(&lp, 0, sizeof lp);
  lp.rows = rows;
  lp.d = d;
  lp.V = V;
  lp.ntiles = ntiles;
  lp.grp_rows = grp;
  lp.stage_bytes = sv::lm_stage_bytes(grp);
  lp.nstages = sv::lm_stages(lp.stage_bytes);
  lp.part = reinterpret_cast<sv::ArgPartial*>(ws + L.off_part);
  lp.flags = reinterpret_cast<unsigned*>(ws);
  lp.ngroups0 = gy;
  lp.grp_rows1 = sv::kLmHBox;
  st = launch_lmhead<sv::kLmArgmax>(map_h, map_h, map_w, lp, gx, gy, stream);
  if (st != SPEC_OK) return st;
  // merge the per-CTA records and resolve the chains (the greedy resolve)
  sv::ArgmaxParams prm;
  std::memset(&prm, 0, sizeof prm);
  prm.tokens = draft_tokens;
  prm.B = B;
  prm.rows_per_seq = k + 1;
  prm.V = V;
  prm.nchunks = gx;
  prm.tree = 0;
  prm.accepted_len = accepted_len;
  prm.out_tokens = out_tokens;
  prm.flags = lp.flags;
  prm.part = lp.part;
  prm.rowarg = reinterpret_cast<int32_t*>(ws + L.off_arg);
  prm.wait_ns = sv::kWaitLimitNs;
  return launch(sv::argmax_resolve_kernel, B, 0, prm, stream, true);
}

spec_status_t spec_lm_head_verify_sample(
    const void* hidden_target, const void* hidden_draft, const void* w_lm,
    const int32_t* draft_tokens, const float* u_accept, const float* u_sample, float temperature,
    int B, int k, int d, int V, int32_t* accepted_len, int32_t* out_tokens, float* p_out,
    float* q_out, float* resid_mass, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || k < 0 || k > SPEC_MAX_K || d < 8 || d > SPEC_LM_MAX_D || d % 8 || V < 1 ||
      V > SPEC_MAX_V)
    return SPEC_ERR_INVALID_ARG;
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return SPEC_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(SPEC_MODE_LM_HEAD_SAMPLE, B, k, V, SPEC_DTYPE_BF16, &L))
    return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!hidden_target || !w_lm || !u_sample || !accepted_len || !out_tokens || !resid_mass)
    return SPEC_ERR_INVALID_ARG;
  if (k > 0 && (!hidden_draft || !draft_tokens || !u_accept || !p_out || !q_out))
    return SPEC_ERR_INVALID_ARG;
  if (!aligned(hidden_target, 16) || !aligned(w_lm, 16) || (k > 0 && !aligned(hidden_draft, 16)))
    return SPEC_ERR_ALIGNMENT;
  if (!aligned(accepted_len, 4) || !aligned(out_tokens, 4) || !aligned(u_sample, 4) ||
      !aligned(resid_mass, 4) ||
      (k > 0 && (!aligned(draft_tokens, 4) || !aligned(u_accept, 4) || !aligned(p_out, 4) ||
                 !aligned(q_out, 4))))
    return SPEC_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < L.bytes) return SPEC_ERR_WORKSPACE;
  if (!aligned(workspace, kAlign)) return SPEC_ERR_ALIGNMENT;
  const int rows_t = B * (k + 1), rows_d = B * k, rows_2 = 2 * B;
  const int ntiles = (V + sv::kLmPairBV - 1) / sv::kLmPairBV;
  int gy0 = 0, grp0 = 0, gy1 = 0, grp1 = 0, gy2 = 0, grp2 = 0, gx = 0;
  if (!lm_row_groups(rows_t, &gy0, &grp0) || !lm_row_groups(rows_d, &gy1, &grp1) ||
      !lm_row_groups(rows_2, &gy2, &grp2) || gy0 + gy1 > 65535)
    return SPEC_ERR_INVALID_ARG;
  spec_status_t st = lm_grid_x<sv::kLmStats>(ntiles, &gx);
  if (st != SPEC_OK) return st;
  char* ws = static_cast<char*>(workspace);
  uint16_t* hbuf = reinterpret_cast<uint16_t*>(ws + L.off_arg);
  float* lbuf = reinterpret_cast<float*>(ws + L.off_log);
  CUtensorMap map_ht, map_hd, map_w, map_hb;
  st = encode_bf16_kmajor(&map_ht, hidden_target, d, rows_t, sv::lm_half_rows(grp0));
  if (st != SPEC_OK) return st;
  st = k > 0 ? encode_bf16_kmajor(&map_hd, hidden_draft, d, rows_d, sv::lm_half_rows(grp1))
             : SPEC_OK;
  if (k == 0) map_hd = map_ht;  // no draft rows: never read
  if (st != SPEC_OK) return st;
  st = encode_bf16_kmajor(&map_w, w_lm, d, V, sv::kLmBV);
  if (st != SPEC_OK) return st;
  st = encode_bf16_kmajor(&map_hb, hbuf, d, rows_2, sv::lm_half_rows(grp2));
  if (st != SPEC_OK) return st;

  // 1. softmax statistics of every target and draft row, and the draft
  // tokens' logits, from the tensor cores' accumulators
  sv::LmHeadParams lp;
  std::memset(&lp, 0, sizeof lp);
  lp.rows = rows_t;
  lp.d = d;
  lp.V = V;
  lp.ntiles = ntiles;
  lp.grp_rows = grp0;
  lp.stage_bytes = sv::lm_stage_bytes(std::max(grp0, grp1));
  lp.nstages = sv::lm_stages(lp.stage_bytes);
  lp.flags = reinterpret_cast<unsigned*>(ws);
  lp.ngroups0 = gy0;
  lp.rows1 = rows_d;
  lp.grp_rows1 = grp1;
  lp.k = k;
  lp.scale = (float)(1.4426950408889634 / (double)temperature);
  lp.tokens = draft_tokens;
  lp.spart = reinterpret_cast<sv::SoftmaxPartial*>(ws + L.off_part);
  lp.zx = reinterpret_cast<float*>(ws + L.off_zx);
  st = launch_lmhead<sv::kLmStats>(map_ht, map_hd, map_w, lp, gx, gy0 + gy1, stream);
  if (st != SPEC_OK) return st;

  // 2. accept test; hidden states of the rows each sequence draws from
  sv::SampleParams prm;
  std::memset(&prm, 0, sizeof prm);
  prm.target = lbuf;
  prm.draft = lbuf;
  prm.tokens = draft_tokens;
  prm.u_accept = u_accept;
  prm.u_sample = u_sample;
  prm.scale = lp.scale;
  prm.B = B;
  prm.k = k;
  prm.V = V;
  prm.nchunks = L.nchunks;
  prm.nrec = gx;
  prm.accepted_len = accepted_len;
  prm.out_tokens = out_tokens;
  prm.p_out = p_out;
  prm.q_out = q_out;
  prm.resid_mass = resid_mass;
  prm.flags = lp.flags;
  prm.part = lp.spart;
  prm.desc = reinterpret_cast<sv::DrawDesc*>(ws + L.off_desc);
  prm.csum = reinterpret_cast<sv::FSum*>(ws + L.off_csum);
  prm.csum_p = reinterpret_cast<sv::FSum*>(ws + L.off_csum_p);
  prm.gsum = reinterpret_cast<float*>(ws + L.off_gsum);
  prm.gsum_p = reinterpret_cast<float*>(ws + L.off_gsum_p);
  prm.zx = lp.zx;
  prm.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  prm.drawn = lbuf;
  {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    pdl_config(&cfg, attr, dim3((unsigned)B, 1, 1), dim3(sv::kThreads, 1, 1), 0, stream);
    if (cudaLaunchKernelEx(&cfg, sv::lm_sample_gather_kernel, prm,
                           static_cast<const uint16_t*>(hidden_target),
                           static_cast<const uint16_t*>(hidden_draft), hbuf, d) != cudaSuccess)
      return SPEC_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }

  // 3. those rows' logits, fp32
  sv::LmHeadParams lq = lp;
  lq.rows = rows_2;
  lq.grp_rows = grp2;
  lq.stage_bytes = sv::lm_stage_bytes(grp2);
  lq.nstages = sv::lm_stages(lq.stage_bytes);
  lq.ngroups0 = gy2;
  lq.rows1 = 0;
  lq.grp_rows1 = sv::kLmHBox;
  lq.logits = lbuf;
  st = launch_lmhead<sv::kLmLogits>(map_hb, map_hb, map_w, lq, gx, gy2, stream);
  if (st != SPEC_OK) return st;

  // 4. the residual or bonus draw (the accept test again, then the draw over
  // the recomputed rows), as spec_verify_sample's
  if (vec_ok(lbuf, V, SPEC_DTYPE_F32)) return run_finish<sv::F32, true>(prm, stream);
  return run_finish<sv::F32, false>(prm, stream);
}

spec_status_t spec_tree_grow(const void* draft_logits, int dtype, float temperature, int B,
                             int D, int K, int V, int M, int32_t* tokens, int32_t* parents,
                             int32_t* depth, float* values, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_INVALID_ARG;
  if (B < 0 || D < 1 || D > sv::kGrowMaxD || K < 1 || K > sv::kGrowMaxK || V < K ||
      V > SPEC_MAX_V || !(temperature > 0.0f) || !std::isfinite(temperature))
    return SPEC_ERR_INVALID_ARG;
  const int nnodes = 1 + K + (D - 1) * K * K;
  if (M < 0 || M > nnodes - 1) return SPEC_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(SPEC_MODE_TREE_GROW, B, K, V, dtype, &L)) return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!draft_logits || !tokens || !parents || !depth || !values) return SPEC_ERR_INVALID_ARG;
  if (!aligned(draft_logits, elem_bytes(dtype)) || !aligned(tokens, 4) || !aligned(parents, 4) ||
      !aligned(depth, 4) || !aligned(values, 4))
    return SPEC_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < L.bytes) return SPEC_ERR_WORKSPACE;
  if (!aligned(workspace, kAlign)) return SPEC_ERR_ALIGNMENT;
  char* ws = static_cast<char*>(workspace);
  sv::GrowParams prm;
  std::memset(&prm, 0, sizeof prm);
  prm.logits = draft_logits;
  prm.scale = (float)(1.4426950408889634 / (double)temperature);
  prm.B = B;
  prm.D = D;
  prm.K = K;
  prm.V = V;
  prm.M = M;
  prm.nchunks = L.nchunks;
  prm.rec = reinterpret_cast<sv::GrowRec*>(ws + L.off_part);
  prm.nval = reinterpret_cast<double*>(ws + L.off_desc);
  prm.npar = reinterpret_cast<int32_t*>(ws + L.off_gsum);
  prm.ntok = prm.npar + (size_t)B * sv::kGrowMaxNodes;
  prm.ndep = prm.ntok + (size_t)B * sv::kGrowMaxNodes;
  prm.tokens = tokens;
  prm.parents = parents;
  prm.depth = depth;
  prm.values = values;
  prm.flags = reinterpret_cast<unsigned*>(ws);
  // every draft row the growth reads, reduced in one streaming launch
  prm.rows_per_tree = 1 + (D - 1) * K;
  if ((long long)B * prm.rows_per_tree * prm.nchunks > INT32_MAX) return SPEC_ERR_INVALID_ARG;
  prm.items = B * prm.rows_per_tree * prm.nchunks;
  const bool vec = vec_ok(draft_logits, V, dtype);  // whole 16-byte vectors per row
  spec_status_t st;
  if (vec) {
    int grid = 0;
    if (dtype == SPEC_DTYPE_BF16) {
      st = persistent_grid<sv::grow_topk_stream_kernel<sv::BF16>>(prm.items, &grid);
      if (st == SPEC_OK)
        st = launch(sv::grow_topk_stream_kernel<sv::BF16>, grid, kStreamSmem, prm, stream, true);
    } else {
      st = persistent_grid<sv::grow_topk_stream_kernel<sv::F32>>(prm.items, &grid);
      if (st == SPEC_OK)
        st = launch(sv::grow_topk_stream_kernel<sv::F32>, grid, kStreamSmem, prm, stream, true);
    }
  } else if (dtype == SPEC_DTYPE_BF16) {
    st = launch(sv::grow_topk_kernel<sv::BF16, false>, prm.items, 0, prm, stream, true);
  } else {
    st = launch(sv::grow_topk_kernel<sv::F32, false>, prm.items, 0, prm, stream, true);
  }
  if (st != SPEC_OK) return st;
  // the node bookkeeping of every layer and the final ranking, one CTA per tree
  st = ensure_smem<sv::grow_tree_kernel>(sv::kGrowTreeSmem);
  if (st != SPEC_OK) return st;
  return launch(sv::grow_tree_kernel, B * sv::kGrowTreeCluster,
                sv::grow_tree_smem(L.nchunks, K, prm.rows_per_tree, nnodes), prm, stream,
                true, sv::kGrowTreeCluster, sv::kGrowTreeThreads);
}

spec_status_t spec_verify_read_flags(void* workspace, uint32_t* host_flags, int clear,
                                     void* stream) {
  if (!workspace || !host_flags) return SPEC_ERR_INVALID_ARG;
  if (!aligned(workspace, kAlign)) return SPEC_ERR_ALIGNMENT;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(host_flags, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return SPEC_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SPEC_ERR_CUDA;
  if (clear && cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

spec_status_t spec_verify_greedy_noalloc(const void* target_logits, int dtype,
                                         const int32_t* draft_tokens, int B, int k, int V,
                                         int32_t* accepted_len, int32_t* out_tokens, void* stream) {
  if (dtype != SPEC_DTYPE_F32 && dtype != SPEC_DTYPE_BF16) return SPEC_ERR_INVALID_ARG;
  if (B < 0 || k < 0 || k > SPEC_MAX_K || V < 1 || V > SPEC_MAX_V) return SPEC_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(SPEC_MODE_GREEDY, B, k, V, dtype, &L)) return SPEC_ERR_INVALID_ARG;
  if (L.bytes > (size_t)SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_ERR_TOO_LARGE;
  if (B == 0) return SPEC_OK;
  if (!target_logits || !accepted_len || !out_tokens || (k > 0 && !draft_tokens))
    return SPEC_ERR_INVALID_ARG;
  if (!aligned(target_logits, elem_bytes(dtype)) || !aligned(accepted_len, 4) ||
      !aligned(out_tokens, 4) || (k > 0 && !aligned(draft_tokens, 4)))
    return SPEC_ERR_ALIGNMENT;
  void* scratch = nullptr;
  const spec_status_t st = noalloc_scratch(&scratch);
  if (st != SPEC_OK) return st;
  // the flag word starts clear on every call (nothing else needs zeroing)
  if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), (cudaStream_t)stream) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return spec_verify_greedy(target_logits, dtype, draft_tokens, B, k, V, accepted_len, out_tokens,
                            scratch, (size_t)SPEC_NOALLOC_SCRATCH_BYTES, stream);
}

spec_status_t spec_verify_selftest_exp2(const float* x, float* y_fma, float* y_sfu, int n,
                                        void* stream) {
  if (n < 0 || (n > 0 && (!x || !y_fma || !y_sfu))) return SPEC_ERR_INVALID_ARG;
  if (n == 0) return SPEC_OK;
  sv::selftest_exp2_kernel<<<(n + 255) / 256, 256, 0, (cudaStream_t)stream>>>(x, y_fma, y_sfu, n);
  if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return SPEC_OK;
}

uint64_t spec_verify_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void spec_verify_set_wait_limit_ns(uint64_t limit_ns) {
  g_wait_limit_ns.store(limit_ns == 0 ? sv::kWaitLimitNs : limit_ns, std::memory_order_relaxed);
}

const char* spec_status_string(int status) {
  switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_ALIGNMENT: return "misaligned pointer";
    case SPEC_ERR_WORKSPACE: return "workspace missing or too small";
    case SPEC_ERR_CUDA: return "CUDA error";
    case SPEC_ERR_TOO_LARGE: return "call exceeds the fixed no-allocation scratch";
    default: return "unknown status";
  }
}

int spec_verify_abi_version(void) { return SPEC_VERIFY_ABI_VERSION; }

}  // extern "C"
