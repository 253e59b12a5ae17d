// sv_device.cuh -- device helpers shared by the verification kernels.
//
// Layout model: every logits row is cut into chunks of kChunk elements (32 KB
// of logits).  A chunk is 2048 16-byte vectors; in a CTA of kThreads threads,
// thread t owns vectors vi = q * kThreads + t (q < kVecPerThread), so each
// warp touches 512 contiguous bytes per q.  Cross-CTA hand-off uses the "last
// CTA to arrive finishes the row" pattern with an atomic counter: no kernel
// waits on another CTA.  The only waits are on this CTA's own bulk copies.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kVecPerThread = 4;
constexpr int kVecPerChunk = kThreads * kVecPerThread;  // 2048 vectors = 32 KB
constexpr int kChunkBytes = kVecPerChunk * 16;
constexpr int kStages = 3;                              // bulk-copy ring depth per CTA
constexpr int kRefEmpty = -(1 << 30);                   // reference of an empty slice
constexpr uint64_t kWaitLimitNs = 200000000ull;         // 0.2 s per bulk-copy wait
constexpr uint32_t kSuspendHintNs = 1000000u;           // longest sleep inside one try_wait

// Flag bits (mirrors include/spec_verify.h).
constexpr unsigned kFlagTokenRange = 1u;
constexpr unsigned kFlagBadParent = 2u;
constexpr unsigned kFlagDepth = 4u;
constexpr unsigned kFlagResidualFallback = 8u;
constexpr unsigned kFlagTimeout = 16u;
constexpr unsigned kFlagBadPath = 32u;

// Element storage traits: 16-byte vectors hold kEPV elements; kNegInf is a
// vector of -inf used to pad past the end of a row.
struct F32 {
  using storage = float;
  static constexpr int kEPV = 4;
  static constexpr int kChunk = kVecPerChunk * kEPV;  // 8192
  static constexpr uint32_t kNegInfWord = 0xFF800000u;
  static __device__ __forceinline__ float load1(const storage* p) { return __ldg(p); }
  static __device__ __forceinline__ float elem(const uint4& v, int e) {
    const uint32_t w = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
    return __uint_as_float(w);
  }
};

struct BF16 {
  using storage = uint16_t;
  static constexpr int kEPV = 8;
  static constexpr int kChunk = kVecPerChunk * kEPV;  // 16384
  static constexpr uint32_t kNegInfWord = 0xFF80FF80u;
  static __device__ __forceinline__ float load1(const storage* p) {
    return __uint_as_float(((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p))) << 16);
  }
  static __device__ __forceinline__ float elem(const uint4& v, int e) {
    const uint32_t w = (e >> 1) == 0 ? v.x : (e >> 1) == 1 ? v.y : (e >> 1) == 2 ? v.z : v.w;
    return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
};

// Streaming 16-byte load through the read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 2^x on the special-function unit (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Exact 2^d for an integer d <= 0 (0 below the normal range).
__device__ __forceinline__ float pow2i_f(int d) {
  return d < -126 ? 0.0f : __int_as_float((d + 127) << 23);
}
__device__ __forceinline__ double pow2i_d(int d) {
  return d < -1022 ? 0.0 : __longlong_as_double((long long)(d + 1023) << 52);
}

// Integer reference for the exponent shift: ceil(m * s), clamped; the empty
// slice (m = -inf) maps to kRefEmpty.
__device__ __forceinline__ int exp_ref(float m, float s) {
  float v = ceilf(m * s);
  v = fminf(fmaxf(v, (float)kRefEmpty), (float)(1 << 30));
  return (int)v;
}

__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// (value, index) argmax order: larger value first, then lower index.
__device__ __forceinline__ bool better(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(v2, i2, v, i)) {
      v = v2;
      i = i2;
    }
  }
}

// Error-free accumulation of non-negative float terms: hi + lo is the running
// sum to about 2^-48 relative (Knuth's two-sum).
struct FSum {
  float hi, lo;  // plain aggregate (usable in __shared__ storage); start from zero()
  static __device__ __forceinline__ FSum zero() { return FSum{0.0f, 0.0f}; }
  __device__ __forceinline__ void add(float b) {
    const float s = __fadd_rn(hi, b);
    const float bb = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    hi = s;
    lo = __fadd_rn(lo, err);
  }
  __device__ __forceinline__ double value() const { return (double)hi + (double)lo; }
  __device__ __forceinline__ void scale(float f) {  // exact for powers of two
    hi *= f;
    lo *= f;
  }
};

// a + b for double-float values (two-sum of the high parts, then a fast
// renormalisation); about 2^-44 relative, float-pipe arithmetic only.
__device__ __forceinline__ FSum df_add(const FSum& a, const FSum& b) {
  const float s = __fadd_rn(a.hi, b.hi);
  const float bb = __fsub_rn(s, a.hi);
  float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  FSum r;
  r.hi = __fadd_rn(s, e);
  r.lo = __fsub_rn(e, __fsub_rn(r.hi, s));
  return r;
}

__device__ __forceinline__ FSum warp_sum_df(FSum v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    FSum y;
    y.hi = __shfl_xor_sync(0xffffffffu, v.hi, o);
    y.lo = __shfl_xor_sync(0xffffffffu, v.lo, o);
    v = df_add(v, y);
  }
  return v;
}

// Normalised double-float (|lo| <= half an ulp of hi), so that values compare
// lexicographically.
__device__ __forceinline__ FSum df_norm(const FSum& a) {
  FSum r;
  r.hi = __fadd_rn(a.hi, a.lo);
  r.lo = __fsub_rn(a.lo, __fsub_rn(r.hi, a.hi));
  return r;
}
// a < b for normalised double-floats.
__device__ __forceinline__ bool df_less(const FSum& a, const FSum& b) {
  return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}
// u * a for a float u >= 0 and a double-float a (two-product via FMA).
__device__ __forceinline__ FSum df_mul_f(float u, const FSum& a) {
  const float p = __fmul_rn(u, a.hi);
  float e = __fmaf_rn(u, a.hi, -p);
  e = __fmaf_rn(u, a.lo, e);
  FSum r;
  r.hi = __fadd_rn(p, e);
  r.lo = __fsub_rn(e, __fsub_rn(r.hi, p));
  return r;
}
__device__ __forceinline__ FSum df_from(float x) { return FSum{x, 0.0f}; }

// Inclusive warp scan of double-float values in lane order.
__device__ __forceinline__ FSum warp_scan_df(FSum v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    FSum y;
    y.hi = __shfl_up_sync(0xffffffffu, v.hi, o);
    y.lo = __shfl_up_sync(0xffffffffu, v.lo, o);
    if (lane >= o) v = df_add(y, v);
  }
  return v;
}

__device__ __forceinline__ void set_flag(unsigned* flags, unsigned bit) { atomicOr(flags, bit); }

// 2^x on the FMA pipe, for x <= 0.5: Cody-Waite reduction x = n + f with
// n = round(x) (the 1.5 * 2^23 shifter), f in [-1/2, 1/2], then a degree-5
// minimax polynomial for 2^f (relative error below 2e-7; coefficients from
// fit_exp2_poly.py) and n added to the exponent field.  Inputs below -126
// are clamped, giving at most 2^-125.5 where 2^x would underflow.
__device__ __forceinline__ float exp2_fma(float x) {
  x = fmaxf(x, -126.0f);
  const float shifter = 12582912.0f;  // 1.5 * 2^23
  const float t = __fadd_rn(x, shifter);
  const float n = __fsub_rn(t, shifter);
  const float f = __fsub_rn(x, n);
  float q = 1.3276472454890609e-3f;
  q = __fmaf_rn(q, f, 9.675540961325169e-3f);
  q = __fmaf_rn(q, f, 5.550713092088699e-2f);
  q = __fmaf_rn(q, f, 2.4022120237350464e-1f);
  q = __fmaf_rn(q, f, 6.931469440460205e-1f);
  q = __fmaf_rn(q, f, 1.0000001192092896f);
  const int ni = __float_as_int(t) - 0x4B400000;  // round(x) as an integer
  return __int_as_float(__float_as_int(q) + (ni << 23));
}

// Packed pairs of floats (f32x2) for the FMA pipe's two-wide instructions.
__device__ __forceinline__ unsigned long long f2pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Largest of the elements of 4 vectors, as float.
template <typename E>
__device__ __forceinline__ float vec4_max(const uint4 (&raw)[4]);

template <>
__device__ __forceinline__ float vec4_max<F32>(const uint4 (&raw)[4]) {
  float m[4];
#pragma unroll
  for (int q = 0; q < 4; ++q)
    m[q] = fmaxf(fmaxf(__uint_as_float(raw[q].x), __uint_as_float(raw[q].y)),
                 fmaxf(__uint_as_float(raw[q].z), __uint_as_float(raw[q].w)));
  return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

template <>
__device__ __forceinline__ float vec4_max<BF16>(const uint4 (&raw)[4]) {
  uint32_t m[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) m[q] = bmax2(bmax2(raw[q].x, raw[q].y), bmax2(raw[q].z, raw[q].w));
  const uint32_t w = bmax2(bmax2(m[0], m[1]), bmax2(m[2], m[3]));
  return fmaxf(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// ---------------------------------------------------------------------------
// Bulk asynchronous copies (global -> shared) completed on an mbarrier.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// L2 cache policies for bulk copies: lines that will be read again soon
// (evict_last) and lines read once (evict_first).
__device__ __forceinline__ uint64_t l2_policy_keep() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_stream() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, unsigned bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Test a barrier phase; the thread may sleep up to `hint_ns` (at most ~1 ms)
// in the instruction while the phase is incomplete (woken when it completes),
// so waiting warps do not spin through the issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity,
                                              uint32_t hint_ns = kSuspendHintNs) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for a barrier phase; give up after limit_ns (returns false).  With the
// default limit a sleeping try_wait is woken by the phase's completion; a
// shorter limit also shortens each sleep, so that the limit is observed.  A
// limit of 1 ns gives up as soon as one test finds the phase incomplete
// (shorter than the resolution of the global timer).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  const uint32_t hint = limit_ns < kSuspendHintNs ? (uint32_t)limit_ns : kSuspendHintNs;
  if (mbar_try_wait(bar, parity, hint)) return true;
  if (limit_ns <= 1) return false;
  const uint64_t t0 = global_ns();
  for (unsigned it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity, hint)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
  return false;
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}

}  // namespace sv
