// sv_device.cuh -- device helpers shared by the verification kernels.
//
// Layout model: every logits row is cut into chunks of kChunk elements (16 KB
// of logits).  One CTA of kThreads threads handles one (row, chunk) item: each
// thread owns kVecPerThread 16-byte vectors, vector index vi = q * kThreads +
// tid, so a warp's loads are 512 contiguous bytes.  Cross-CTA hand-off uses the
// "last CTA to arrive finishes the row" pattern with an atomic counter, never a
// wait, so no kernel here spins on another CTA.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kVecPerThread = 4;
constexpr int kGroupsPerChunk = kThreads * kVecPerThread;  // 1024 vectors = groups
constexpr int kRefEmpty = -(1 << 30);                      // reference of an empty slice

// Element storage traits: 16-byte vectors hold kEPV elements.
struct F32 {
  using storage = float;
  static constexpr int kEPV = 4;
  static constexpr int kChunk = kThreads * kVecPerThread * kEPV;  // 4096
  static __device__ __forceinline__ float load1(const storage* p) { return __ldg(p); }
  static __device__ __forceinline__ void unpack(const uint4& v, float (&z)[kEPV]) {
    z[0] = __uint_as_float(v.x);
    z[1] = __uint_as_float(v.y);
    z[2] = __uint_as_float(v.z);
    z[3] = __uint_as_float(v.w);
  }
};

struct BF16 {
  using storage = uint16_t;
  static constexpr int kEPV = 8;
  static constexpr int kChunk = kThreads * kVecPerThread * kEPV;  // 8192
  static __device__ __forceinline__ float load1(const storage* p) {
    return __uint_as_float(((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p))) << 16);
  }
  static __device__ __forceinline__ void unpack(const uint4& v, float (&z)[kEPV]) {
    z[0] = __uint_as_float(v.x << 16);
    z[1] = __uint_as_float(v.x & 0xFFFF0000u);
    z[2] = __uint_as_float(v.y << 16);
    z[3] = __uint_as_float(v.y & 0xFFFF0000u);
    z[4] = __uint_as_float(v.z << 16);
    z[5] = __uint_as_float(v.z & 0xFFFF0000u);
    z[6] = __uint_as_float(v.w << 16);
    z[7] = __uint_as_float(v.w & 0xFFFF0000u);
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

// One chunk of one row, held in registers: z[q][e] is element
// j0 + (q * kThreads + tid) * kEPV + e; slots past the row end hold -inf.
template <typename E, bool kVec>
__device__ __forceinline__ void load_chunk(const typename E::storage* __restrict__ row, int j0,
                                           int j1, float (&z)[kVecPerThread][E::kEPV]) {
  const int tid = threadIdx.x;
  if constexpr (kVec) {
    const int nvec = (j1 - j0) / E::kEPV;  // rows are whole vectors on this path
    uint4 raw[kVecPerThread];
#pragma unroll
    for (int q = 0; q < kVecPerThread; ++q) {
      const int vi = q * kThreads + tid;
      if (vi < nvec)
        raw[q] = ldg_stream(row + j0 + vi * E::kEPV);
      else
        raw[q] = make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int q = 0; q < kVecPerThread; ++q) {
      const int vi = q * kThreads + tid;
      E::unpack(raw[q], z[q]);
      if (vi >= nvec) {
#pragma unroll
        for (int e = 0; e < E::kEPV; ++e) z[q][e] = -INFINITY;
      }
    }
  } else {
#pragma unroll
    for (int q = 0; q < kVecPerThread; ++q) {
      const int base = j0 + (q * kThreads + tid) * E::kEPV;
#pragma unroll
      for (int e = 0; e < E::kEPV; ++e)
        z[q][e] = (base + e < j1) ? E::load1(row + base + e) : -INFINITY;
    }
  }
}

// 2^x on the special-function unit (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Exact 2^d for an integer d <= 0 (0 below the float normal range).
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

// Error-free accumulation of positive float terms: (hi, lo) with hi + lo the
// running sum to about 2^-48 relative (Knuth's two-sum).
struct FSum {
  float hi = 0.0f, lo = 0.0f;
  __device__ __forceinline__ void add(float b) {
    const float s = __fadd_rn(hi, b);
    const float bb = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    hi = s;
    lo = __fadd_rn(lo, err);
  }
  __device__ __forceinline__ double value() const { return (double)hi + (double)lo; }
};

// Release this CTA's global writes, count its arrival, and tell whether it
// arrived last (then acquire the other arrivals' writes and reset the counter).
// Called by every thread of the CTA.
__device__ __forceinline__ bool arrive_last(unsigned* counter, unsigned expected, int* s_flag) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned old = atomicAdd(counter, 1u);
    const bool last = (old == expected - 1u);
    if (last) {
      __threadfence();
      *counter = 0u;  // every call leaves its counters at zero
    }
    *s_flag = last ? 1 : 0;
  }
  __syncthreads();
  const bool last = *s_flag != 0;
  if (last) __threadfence();
  return last;
}

__device__ __forceinline__ void set_flag(unsigned* flags, unsigned bit) { atomicOr(flags, bit); }

}  // namespace sv
