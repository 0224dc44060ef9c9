// Device-side helpers shared by the kernels: vector loads, element loads of
// the supported input dtypes, warp reductions, and the device error word.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace qlin {

// Error codes recorded in the device error word (first one wins).
enum : int32_t {
  kDevErrNone = 0,
  kDevErrTimeoutBase = 0x1000,  // + site id: a bounded barrier wait expired
  kDevErrBadIndex = 0x2000,     // an index argument (e.g. a channel permutation) was out of range
};

__device__ __forceinline__ void record_device_error(int32_t* err, int32_t code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

// x / d rounded to nearest even from r = __frcp_rn(d), by one FMA correction
// step (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", 1990): q0 = x r, e = x - q0 d, q = q0 + e r.  With r
// the correctly rounded reciprocal this equals __fdiv_rn(x, d) whenever d,
// r and the quotient are normal numbers; a quotient below the normal range
// comes out as a tiny number (or zero) with the sign of x.  A zero dividend
// returns q0 = x r, the correctly signed zero (the correction would add
// +0 and -0 and lose the sign).  Four operations per element instead of a
// full division when many elements share d.
__device__ __forceinline__ float div_by_rcp(float x, float d, float r) {
  const float q0 = __fmul_rn(x, r);
  const float e = __fmaf_rn(-q0, d, x);
  const float q = __fmaf_rn(e, r, q0);
  return x == 0.0f ? q0 : q;
}

// True when div_by_rcp may replace the division by d (d and 1/d normal).
__device__ __forceinline__ bool rcp_division_ok(float d, float r) {
  const float kMinNormal = 1.17549435e-38f, kMaxFinite = 3.40282347e38f;
  return fabsf(d) >= kMinNormal && fabsf(d) <= kMaxFinite && fabsf(r) >= kMinNormal && fabsf(r) <= kMaxFinite;
}

// Programmatic dependent launch: let the next kernel in the stream start
// launching, and wait for the previous one before touching data it writes.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// 16-byte read-only load that does not allocate in L1 (streamed weights).
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 16-byte read-only load through L1 (small operands reused across warps).
__device__ __forceinline__ uint4 ldg_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// 16-byte load cached in L2 only.  For data the previous kernel in the stream
// writes while this one is already resident (programmatic dependent launch):
// an L1 line filled before that kernel finished could be stale.
__device__ __forceinline__ uint4 ldg_cg_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Eight consecutive input elements of the given dtype, widened to float32
// (exact for fp16 and bf16).  `p` must be 16-byte aligned for F16/BF16 and
// 32-byte aligned (two 16-byte loads) for F32.
template <int DT>
struct Vec8Loader;

template <>
struct Vec8Loader<0> {  // F16
  static __device__ __forceinline__ void load(const void* p, float* v) {
    uint4 u = ldg_v4(p);
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __half22float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
};

template <>
struct Vec8Loader<1> {  // BF16
  static __device__ __forceinline__ void load(const void* p, float* v) {
    uint4 u = ldg_v4(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
};

template <>
struct Vec8Loader<2> {  // F32
  static __device__ __forceinline__ void load(const void* p, float* v) {
    uint4 a = ldg_v4(p);
    uint4 b = ldg_v4(static_cast<const char*>(p) + 16);
    v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
    v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
    v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
    v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
  }
};

// One element of the given dtype as float32.
template <int DT>
__device__ __forceinline__ float load_elem(const void* base, int64_t i) {
  if constexpr (DT == 0) return __half2float(static_cast<const __half*>(base)[i]);
  else if constexpr (DT == 1) return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[i]);
  else return static_cast<const float*>(base)[i];
}

template <int DT>
__host__ __device__ constexpr int elem_bytes() { return DT == 2 ? 4 : 2; }

}  // namespace qlin
