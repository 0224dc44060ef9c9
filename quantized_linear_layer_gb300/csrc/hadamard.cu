// Online Hadamard rotation of activation rows before 4-bit quantization.
//
// The operation: every group of n consecutive elements of a row times the
// normalized Hadamard matrix H_n / sqrt(n), then times signs[k] (+-1 per
// column, QuaRot's diag(+-1)) if given, rounded once to the output type.
//   Sylvester H_n ("LLM and AIGC quantization", QuaRot section): computed
//     by the fast Walsh-Hadamard transform, log2(n) butterfly stages, stage
//     h mapping the pair (a, b) at distance h to (a + b, a - b);
//   regular H_n, n = 4^k (ConvRot section: the Kronecker power of
//     H4 = [[1,1,1,-1],[1,1,-1,1],[1,-1,1,1],[-1,1,1,1]]): computed by
//     radix-4 stages at strides 1, 4, 16, ..., each quad (x0, x1, x2, x3)
//     becoming y_i = s - 2 x_(3-i) with s = (x0 + x1) + (x2 + x3) (H4 is the
//     all-ones matrix minus twice the anti-diagonal).
// The stages run in float32, then one multiply by c = float32(1/sqrt(n)) and
// the signs; the result is within float32 rounding of the exact rotation and
// the same on every run.
//
// HBM-bound (read and write the rows once; a few float32 operations per
// element and stage), so no tensor cores: the pages' ConvRot multiplies by the
// dense N0 x N0 matrix on tensor cores, 2 N0 flops per element, where the
// butterflies need log2(N0).  Each thread holds 8 consecutive elements;
// stages inside them run in registers, stages across lanes by shuffles
// (Sylvester up to n = 256, the regular transform up to 256), and Sylvester
// stages beyond 256 elements through shared memory, one CTA of n/8 threads
// per group.
//
// The kernels do not trigger a programmatic dependent launch: the quantizers
// that read the rotated rows are launched without it and read x at their
// start.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <type_traits>

#include "device_common.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace {

constexpr int kHdThreads = 256;

// Eight elements as float32 through the coherent path (not the read-only
// one: the rotation may run in place).
template <int DT>
__device__ __forceinline__ void load8(const void* p, float* v) {
  if constexpr (DT == 2) {
    const float4 a = static_cast<const float4*>(p)[0], b = static_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 u = *static_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f;
      if constexpr (DT == 0) f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      else f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
}

template <int DT>
__device__ __forceinline__ void store8(void* p, const float* v) {
  if constexpr (DT == 2) {
    float4* q = static_cast<float4*>(p);
    q[0] = make_float4(v[0], v[1], v[2], v[3]);
    q[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (DT == 0) {
        __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&h);
      } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&h);
      }
    }
    *static_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Sylvester stages h = 1, 2, 4 (inside the thread's 8 elements), up to n/2.
__device__ __forceinline__ void fwht_in_thread(float* v, int n) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
    if (h >= n) break;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i & h) continue;
      const float a = v[i], b = v[i + h];
      v[i] = __fadd_rn(a, b);
      v[i + h] = __fsub_rn(a, b);
    }
  }
}

// Sylvester stages h = 8 m for lane bits m = 1 .. 16 while h < min(n, 256).
__device__ __forceinline__ void fwht_across_lanes(float* v, int n, int lane) {
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    if (8 * m >= n) break;
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
      v[i] = upper ? __fsub_rn(o, v[i]) : __fadd_rn(v[i], o);  // (a + b, a - b), a the lower index
    }
  }
}

__device__ __forceinline__ float quad_out(float q0, float q1, float q2, float q3, int pos) {
  const float s = __fadd_rn(__fadd_rn(q0, q1), __fadd_rn(q2, q3));
  const float x = pos == 0 ? q3 : pos == 1 ? q2 : pos == 2 ? q1 : q0;  // x_(3 - pos)
  return __fsub_rn(s, 2.0f * x);
}

// Regular-Hadamard radix-4 stages at strides 1, 4, 16, 64 while the stride is < n.
__device__ __forceinline__ void regular_stages(float* v, int n, int lane) {
  // stride 1: quads (0..3) and (4..7) of the thread
  {
    float y[8];
#pragma unroll
    for (int b = 0; b < 8; b += 4)
#pragma unroll
      for (int p = 0; p < 4; ++p) y[b + p] = quad_out(v[b], v[b + 1], v[b + 2], v[b + 3], p);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = y[i];
  }
  if (n <= 4) return;
  // stride 4: quad (r, r + 4, r + 8, r + 12) of a 16-element block = this
  // lane's elements r, r + 4 and the neighbour lane's (lane ^ 1)
  {
    const bool odd = (lane & 1) != 0;
    float y[8];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float o0 = __shfl_xor_sync(0xffffffffu, v[r], 1);
      const float o1 = __shfl_xor_sync(0xffffffffu, v[r + 4], 1);
      const float q0 = odd ? o0 : v[r], q1 = odd ? o1 : v[r + 4];
      const float q2 = odd ? v[r] : o0, q3 = odd ? v[r + 4] : o1;
      y[r] = quad_out(q0, q1, q2, q3, odd ? 2 : 0);
      y[r + 4] = quad_out(q0, q1, q2, q3, odd ? 3 : 1);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = y[i];
  }
  // strides 16 and 64: the quad's members are the lanes that differ in two
  // lane bits (1-2, then 3-4), same element index.  Three shuffles give the
  // pair sum (q0 + q1 or q2 + q3), then s, then x_(3 - pos), the lane whose
  // position is pos ^ 3; float addition is commutative, so every lane of the
  // quad holds the same s = (q0 + q1) + (q2 + q3).
#pragma unroll
  for (int shift = 1; shift <= 3; shift += 2) {
    if ((8 << shift) >= n) break;  // stride 8 . 2^shift
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float pair = __fadd_rn(v[i], __shfl_xor_sync(0xffffffffu, v[i], 1 << shift));
      const float sum = __fadd_rn(pair, __shfl_xor_sync(0xffffffffu, pair, 2 << shift));
      const float mirror = __shfl_xor_sync(0xffffffffu, v[i], 3 << shift);
      v[i] = __fsub_rn(sum, 2.0f * mirror);
    }
  }
}

__device__ __forceinline__ void scale_and_sign(float* v, float c, const int8_t* __restrict__ signs, int64_t col0) {
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], c);
  if (signs != nullptr) {
    const uint2 sg = __ldg(reinterpret_cast<const uint2*>(signs + col0));
    const uint32_t w[2] = {sg.x, sg.y};
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (static_cast<int8_t>((w[i >> 2] >> (8 * (i & 3))) & 0xFF) < 0) v[i] = -v[i];
  }
}

// Groups of n <= 256: one warp walks 256 consecutive elements (all its groups),
// grid-stride over the rows' 8-element vectors; every lane of a warp runs the
// same iterations (the shuffles need the whole warp), and a group is all in
// range or all out (K is a multiple of n).
template <int DT, int KIND>
__global__ void __launch_bounds__(kHdThreads) hadamard_warp_kernel(const void* x, int64_t nvec, int K,
                                                                  int n, float c, const int8_t* __restrict__ signs,
                                                                  void* y) {
  // x and y may be the same rows (in place): every element is read by the
  // thread that later writes it, before the write
  constexpr int EB = DT == 2 ? 4 : 2;
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kHdThreads;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kHdThreads + (threadIdx.x & ~31); base < nvec;
       base += stride) {
    const int64_t vi = base + lane;
    const bool active = vi < nvec;
    float v[8];
    if (active) {
      load8<DT>(static_cast<const char*>(x) + vi * 8 * EB, v);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    }
    if constexpr (KIND == 0) {
      fwht_in_thread(v, n);
      fwht_across_lanes(v, n, lane);
    } else {
      regular_stages(v, n, lane);
    }
    if (!active) continue;
    scale_and_sign(v, c, signs, (vi * 8) % K);
    store8<DT>(static_cast<char*>(y) + vi * 8 * EB, v);
  }
}

// Sylvester groups of 512 .. 8192: one CTA of n / 8 threads per group, the
// stages h >= 256 through shared memory (each thread keeps its own 8 values
// in registers and reads the 8 partners).
template <int DT>
__global__ void __launch_bounds__(1024) hadamard_cta_kernel(const void* x, int64_t groups, int K, int n,
                                                            float c, const int8_t* __restrict__ signs,
                                                            void* y) {
  extern __shared__ __align__(16) float buf[];
  constexpr int EB = DT == 2 ? 4 : 2;
  const int tid = threadIdx.x, lane = tid & 31;
  for (int64_t g = blockIdx.x; g < groups; g += gridDim.x) {
    const int64_t e0 = g * n + 8 * tid;  // first element of this thread
    float v[8];
    load8<DT>(static_cast<const char*>(x) + e0 * EB, v);
    fwht_in_thread(v, n);
    fwht_across_lanes(v, n, lane);
    for (int h = 256; h < n; h <<= 1) {
      // 32-byte rows per thread, written and read as two 16-byte pieces
      float4* mine = reinterpret_cast<float4*>(buf + 8 * tid);
      mine[0] = make_float4(v[0], v[1], v[2], v[3]);
      mine[1] = make_float4(v[4], v[5], v[6], v[7]);
      __syncthreads();
      const int j0 = 8 * tid;  // the 8 elements share bit h (h >= 256 > 7)
      const bool upper = (j0 & h) != 0;
      const float4* other = reinterpret_cast<const float4*>(buf + (j0 ^ h));
      const float4 o0 = other[0], o1 = other[1];
      const float o[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = upper ? __fsub_rn(o[i], v[i]) : __fadd_rn(v[i], o[i]);
      __syncthreads();
    }
    scale_and_sign(v, c, signs, e0 % K);
    store8<DT>(static_cast<char*>(y) + e0 * EB, v);
  }
}

}  // namespace

cudaError_t launch_hadamard(const void* x, qlin_dtype dtype, int64_t rows, int64_t K, qlin_hadamard_kind kind,
                            int64_t n, const int8_t* signs, void* y, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const float c = static_cast<float>(1.0 / std::sqrt(static_cast<double>(n)));
  const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
  auto go = [&](auto dt) -> cudaError_t {
    constexpr int DT = decltype(dt)::value;
    if (n <= 256) {
      const int64_t nvec = rows * (K / 8);
      const int64_t want = (nvec + kHdThreads - 1) / kHdThreads;
      const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
      if (kind == QLIN_HADAMARD_SYLVESTER)
        hadamard_warp_kernel<DT, 0><<<grid, kHdThreads, 0, stream>>>(x, nvec, static_cast<int>(K),
                                                                       static_cast<int>(n), c, signs, y);
      else
        hadamard_warp_kernel<DT, 1><<<grid, kHdThreads, 0, stream>>>(x, nvec, static_cast<int>(K),
                                                                       static_cast<int>(n), c, signs, y);
      return cudaGetLastError();
    }
    const int64_t groups = rows * (K / n);
    const unsigned grid = static_cast<unsigned>(groups < cap ? groups : cap);
    const size_t smem = static_cast<size_t>(n) * sizeof(float);
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(hadamard_cta_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    hadamard_cta_kernel<DT><<<grid, static_cast<unsigned>(n / 8), smem, stream>>>(x, groups, static_cast<int>(K),
                                                                                static_cast<int>(n), c, signs, y);
    return cudaGetLastError();
  };
  switch (dtype) {
    case QLIN_F16: return go(std::integral_constant<int, 0>{});
    case QLIN_BF16: return go(std::integral_constant<int, 1>{});
    default: return go(std::integral_constant<int, 2>{});
  }
}

}  // namespace qlin
