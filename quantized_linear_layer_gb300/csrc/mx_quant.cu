// MX quantization: MXFP8 (E4M3 elements) and MXFP4 (E2M1 elements), one E8M0
// scale per 32 consecutive elements of a row.
//
// Per block ("LLM and AIGC quantization: from number formats to W4A4",
// block-scaled formats: the shared scale is a power of two,
// 2^(floor(log2 absmax) - e_max), e_max = 8 for E4M3 and 2 for E2M1):
//   e    = floor(log2 max|x|) - e_max, clamped to [-127, 127] (-127 for a
//          zero block, and wherever the maximum is below 2^(e_max - 127))
//   sf   = e + 127                               (the E8M0 code)
//   q    = E4M3 / E2M1( x . 2^-e )               (float32 multiply; RNE, saturating)
// The multiply by 2^-e is exact unless the product is below the float32
// normal range, where both element formats round it to zero anyway.
//
// Memory-bound: four lanes share one block (eight elements each, one
// 16-byte or two 16-byte loads), the block maximum by two xor shuffles, the
// codes stored as 8 bytes (E4M3) or 4 bytes (E2M1) per lane, so each warp
// reads and writes contiguous runs.  Grid-stride over the 8-element vectors;
// all lanes of a warp run the same number of iterations (the shuffles need
// the whole warp), and a block's four vectors are all in range or all out
// (K is a multiple of 32).
#include <type_traits>

#include "device_common.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace {

constexpr int kMxThreads = 256;

// Two floats -> two E4M3 codes, `lo` in the low byte.
__device__ __forceinline__ uint32_t mx_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two floats -> one byte of two E2M1 codes, `lo` in bits 0-3.
__device__ __forceinline__ uint32_t mx_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// FMT 0: MXFP8 (E4M3 codes, [rows][K] bytes); FMT 1: MXFP4 (E2M1 codes packed
// two per byte, element 2i in the low nibble, [rows][K/2]).
template <int DT, int FMT>
__global__ void __launch_bounds__(kMxThreads) mx_quant_kernel(const void* __restrict__ x, int64_t nvec, int K,
                                                                uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                                int sf_mma) {
  pdl_launch_dependents();  // the GEMM that reads the codes may start setting up
  constexpr int EB = elem_bytes<DT>();
  constexpr int kEmax = FMT == 0 ? 8 : 2;
  const int lane = threadIdx.x & 31;
  const int vpr = K / 8;                      // 8-element vectors per row
  const int kg = (K / 32 + 3) / 4;            // 4-scale groups per row in the MMA layout
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kMxThreads;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kMxThreads + (threadIdx.x & ~31); base < nvec;
       base += stride) {
    const int64_t v = base + lane;
    const bool active = v < nvec;
    float e[8];
    if (active) {
      Vec8Loader<DT>::load(static_cast<const char*>(x) + v * 8 * EB, e);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) e[i] = 0.0f;
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(e[i]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    // floor(log2 m) is the unbiased exponent field for a normal m; a zero or
    // subnormal maximum lies below 2^-126 and takes the clamp
    const int biased = static_cast<int>(__float_as_uint(m) >> 23) & 0xFF;
    const int ex = biased == 0 ? -127 : max(biased - 127 - kEmax, -127);
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - ex) << 23);  // 2^-ex, 127 - ex in [2, 254]
    if (!active) continue;
    const int64_t row = v / vpr;
    const int cv = static_cast<int>(v - row * vpr);
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(e[i], inv);
    if constexpr (FMT == 0) {
      const uint32_t w0 = mx_e4m3x2(y[0], y[1]) | (mx_e4m3x2(y[2], y[3]) << 16);
      const uint32_t w1 = mx_e4m3x2(y[4], y[5]) | (mx_e4m3x2(y[6], y[7]) << 16);
      *reinterpret_cast<uint2*>(q + row * K + cv * 8) = make_uint2(w0, w1);
    } else {
      const uint32_t w = mx_e2m1x2(y[0], y[1]) | (mx_e2m1x2(y[2], y[3]) << 8) | (mx_e2m1x2(y[4], y[5]) << 16) |
                         (mx_e2m1x2(y[6], y[7]) << 24);
      *reinterpret_cast<uint32_t*>(q + row * (K / 2) + cv * 4) = w;
    }
    if ((lane & 3) == 0) {
      const int j = cv >> 2;  // the row's 32-element block
      const int64_t at = sf_mma ? ((row >> 7) * kg + (j >> 2)) * 512 + 16 * (row & 31) + 4 * ((row & 127) >> 5) + (j & 3)
                                : row * (K / 32) + j;
      sf[at] = static_cast<uint8_t>(ex + 127);
    }
  }
}

}  // namespace

// Launched without the programmatic-serialization attribute: the kernel reads
// x at its start, with no griddepcontrol.wait before it, so it must not
// overlap the kernel that writes x.
cudaError_t launch_quant_mx(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, qlin_mx_fmt fmt, uint8_t* q,
                            uint8_t* sf, qlin_sf_layout sf_layout, cudaStream_t stream) {
  const int64_t nvec = rows * (K / 8);
  if (nvec == 0) return cudaSuccess;
  const int64_t want = (nvec + kMxThreads - 1) / kMxThreads;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  const int mma = sf_layout == QLIN_SF_MMA ? 1 : 0;
  auto go = [&](auto dt, auto f) -> cudaError_t {
    mx_quant_kernel<decltype(dt)::value, decltype(f)::value><<<grid, kMxThreads, 0, stream>>>(
        x, nvec, static_cast<int>(K), q, sf, mma);
    return cudaGetLastError();
  };
  auto with_fmt = [&](auto dt) -> cudaError_t {
    return fmt == QLIN_MX_FP8_E4M3 ? go(dt, std::integral_constant<int, 0>{}) : go(dt, std::integral_constant<int, 1>{});
  };
  switch (x_dtype) {
    case QLIN_F16: return with_fmt(std::integral_constant<int, 0>{});
    case QLIN_BF16: return with_fmt(std::integral_constant<int, 1>{});
    default: return with_fmt(std::integral_constant<int, 2>{});
  }
}

}  // namespace qlin
