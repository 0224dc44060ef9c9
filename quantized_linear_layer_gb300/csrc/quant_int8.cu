// Per-token int8 activation quantization (symmetric absmax or asymmetric with
// an integer zero-point), the int8 row sum used as the W8A8 zero-point
// adjustment, the asymmetric 4-bit group weight quantizer, and the per-row
// FP8 E4M3 quantizer of FP8 W8A8.
//
// Symmetric: s = max|x| / 127, q = clamp(rint(x / s), -127, 127)
//   ("LLM and AIGC quantization: from number formats to W4A4", symmetric
//   quantization with q_max = 2^(b-1) - 1, per-token dynamic scales).
// Asymmetric: the row range [min(x,0), max(x,0)] is mapped onto [-128, 127]
//   with an integer zero-point z so that 0 is exact; q = round(x/s) + z
//   ("Chapter 9 - Quantization kernels", 9.2: zero-point added on quantize).
// FP8 E4M3, per token or per output channel: s = max|x| / 448 (1 for an
//   all-zero row), q = E4M3(x / s), nearest, ties to even, saturating
//   ("LLM and AIGC quantization", "W4A4, FP8 and block-scaled formats": x/s
//   converted to E4M3 instead of rounded to INT8; "FP8: robustness from
//   dynamic range": the per-tensor example [0.6, -45.0, 1.1, -0.8] -> 6, -448,
//   11, -8, whose printed quotients this scale reproduces).
// 4-bit weights: s = fp16(max(max - min, 1e-5) / 15), z = rint(-min / s),
//   q = clamp(rint(w / s) + z, 0, 15) per 128-element group (the AWQ offline
//   flow's pseudo_quant on the same page).
//
// The rounding decisions are taken in IEEE float32 exactly as written: true
// division (__fdiv_rn), round-half-to-even (__float2int_rn), and no fused
// multiply-add anywhere a result feeds a rounding decision.
#include <algorithm>

#include "device_common.cuh"
#include "exact_sumsq.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kMaxVecPerThread = 4;  // 4 x 8 elements held in registers
// The row quantizers are bound by the latency of each CTA's life (row loads,
// the max reduction and its barrier, the divisions), so their rate is the
// rows each SM holds at once: 48 registers per thread fit five CTAs per SM
// instead of four (a few bytes of spill; FP8 4% faster), and the int8 kernel
// for rows of up to 4096 elements, holding two vectors per thread, fits six
// at 40 registers (int8 2048 x 4096: 9.75 -> 7.8 us, 4096 x 4096 with
// zero-points: 18.2 -> 14.0 us).
constexpr int kQuantMinCtasPerSm = 5;

// F16: the codes are written as the fp16 numbers of the same values (exact,
// |q| <= 128), the operand form of the W8A8 GEMM that widens nothing on chip.
// V: 8-element vectors of the row held in registers per thread (2 for rows of
// up to 4096 elements, which leaves room for a sixth CTA per SM; else 4).
template <int DT, bool ASYM, bool F16, int V>
__global__ void __launch_bounds__(kQuantThreads, V == 2 ? 6 : kQuantMinCtasPerSm) quant_int8_rows_kernel(const void* __restrict__ x, int K,
                                                                         void* __restrict__ q,
                                                                         float* __restrict__ scale,
                                                                         int32_t* __restrict__ azp) {
  pdl_launch_dependents();  // the GEMM that reads the codes may start setting up
  const int64_t row = blockIdx.x;
  const int tid = threadIdx.x;
  const int nvec = K / 8;
  const char* xr = static_cast<const char*>(x) + row * (int64_t)K * elem_bytes<DT>();
  unsigned char* qr = static_cast<unsigned char*>(q) + row * (int64_t)K * (F16 ? 2 : 1);

  float v[V][8];
  // Running absmax (symmetric) or running min / max (asymmetric).  Both start
  // at 0, which makes the asymmetric range include 0.
  float s0 = 0.0f;
  float s1 = 0.0f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int idx = tid + i * kQuantThreads;
    if (idx < nvec) {
      Vec8Loader<DT>::load(xr + (int64_t)idx * 8 * elem_bytes<DT>(), v[i]);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (ASYM) { s0 = fminf(s0, v[i][j]); s1 = fmaxf(s1, v[i][j]); }
        else s0 = fmaxf(s0, fabsf(v[i][j]));
      }
    }
  }
  for (int idx = tid + V * kQuantThreads; idx < nvec; idx += kQuantThreads) {
    float t[8];
    Vec8Loader<DT>::load(xr + (int64_t)idx * 8 * elem_bytes<DT>(), t);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (ASYM) { s0 = fminf(s0, t[j]); s1 = fmaxf(s1, t[j]); }
      else s0 = fmaxf(s0, fabsf(t[j]));
    }
  }

  // Block reduction (min/max are exact, so the order does not matter).
  __shared__ float red0[kQuantThreads / 32], red1[kQuantThreads / 32];
  __shared__ float s_scale;
  __shared__ int s_zero;
  if (ASYM) { s0 = warp_min(s0); s1 = warp_max(s1); } else { s0 = warp_max(s0); }
  if ((tid & 31) == 0) { red0[tid >> 5] = s0; red1[tid >> 5] = s1; }
  __syncthreads();
  if (tid == 0) {
    float a = red0[0], b = red1[0];
    for (int w = 1; w < kQuantThreads / 32; ++w) {
      if (ASYM) { a = fminf(a, red0[w]); b = fmaxf(b, red1[w]); } else { a = fmaxf(a, red0[w]); }
    }
    if (ASYM) {
      // a = min(min x, 0), b = max(max x, 0)
      const float range = fmaxf(__fsub_rn(b, a), 1e-5f);
      const float s = __fdiv_rn(range, 255.0f);
      const int z = -128 - __float2int_rn(__fdiv_rn(a, s));
      s_scale = s;
      s_zero = z;
      scale[row] = s;
      azp[row] = z;
    } else {
      const float s = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 127.0f);
      s_scale = s;
      s_zero = 0;
      scale[row] = s;
    }
  }
  __syncthreads();
  const float s = s_scale;
  const int z = s_zero;
  // Every element of the row is divided by s: through the correctly rounded
  // reciprocal and one FMA correction, which gives the IEEE quotient wherever
  // it can change the rounded code (tiny quotients round to 0 either way).
  const float rs = __frcp_rn(s);
  const bool rcp_ok = rcp_division_ok(s, rs);

  auto quant8 = [&](const float* t, int64_t idx) {
    int r[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      r[j] = __float2int_rn(rcp_ok ? div_by_rcp(t[j], s, rs) : __fdiv_rn(t[j], s));
      if (ASYM) r[j] = min(max(r[j] + z, -128), 127);
      else r[j] = min(max(r[j], -127), 127);
    }
    if (F16) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 h = __halves2half2(__int2half_rn(r[2 * j]), __int2half_rn(r[2 * j + 1]));
        w[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
      *reinterpret_cast<uint4*>(qr + idx * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      uint32_t w0 = 0, w1 = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t byte = static_cast<uint32_t>(r[j]) & 0xffu;
        if (j < 4) w0 |= byte << (8 * j); else w1 |= byte << (8 * (j - 4));
      }
      *reinterpret_cast<uint2*>(qr + idx * 8) = make_uint2(w0, w1);
    }
  };
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int idx = tid + i * kQuantThreads;
    if (idx < nvec) quant8(v[i], idx);
  }
  for (int idx = tid + V * kQuantThreads; idx < nvec; idx += kQuantThreads) {
    float t[8];
    Vec8Loader<DT>::load(xr + (int64_t)idx * 8 * elem_bytes<DT>(), t);
    quant8(t, idx);
  }
}

// Two floats -> two E4M3-FN codes in one 16-bit word, `lo` in bits 0-7
// (hardware round-to-nearest-even, saturating at 448).
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// One CTA per row, the same shape as the int8 quantizer: 16-byte loads kept
// in registers, block absmax, then IEEE division and the E4M3 encode.
template <int DT>
__global__ void __launch_bounds__(kQuantThreads, kQuantMinCtasPerSm) quant_fp8_rows_kernel(const void* __restrict__ x, int K,
                                                                      uint8_t* __restrict__ q,
                                                                      float* __restrict__ scale) {
  pdl_launch_dependents();  // the GEMM that reads the codes may start setting up
  const int64_t row = blockIdx.x;
  const int tid = threadIdx.x;
  const int nvec = K / 8;
  const char* xr = static_cast<const char*>(x) + row * (int64_t)K * elem_bytes<DT>();
  uint8_t* qr = q + row * (int64_t)K;

  float v[kMaxVecPerThread][8];
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxVecPerThread; ++i) {
    const int idx = tid + i * kQuantThreads;
    if (idx < nvec) {
      Vec8Loader<DT>::load(xr + (int64_t)idx * 8 * elem_bytes<DT>(), v[i]);
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[i][j]));
    }
  }
  for (int idx = tid + kMaxVecPerThread * kQuantThreads; idx < nvec; idx += kQuantThreads) {
    float t[8];
    Vec8Loader<DT>::load(xr + (int64_t)idx * 8 * elem_bytes<DT>(), t);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(t[j]));
  }
  __shared__ float red[kQuantThreads / 32];
  __shared__ float s_scale;
  m = warp_max(m);
  if ((tid & 31) == 0) red[tid >> 5] = m;
  __syncthreads();
  if (tid == 0) {
    float a = red[0];
    for (int w = 1; w < kQuantThreads / 32; ++w) a = fmaxf(a, red[w]);
    const float s = (a == 0.0f) ? 1.0f : __fdiv_rn(a, 448.0f);
    s_scale = s;
    scale[row] = s;
  }
  __syncthreads();
  const float s = s_scale;
  // x / s through the correctly rounded reciprocal and one FMA correction
  // (the IEEE quotient wherever it can change the code; quotients below the
  // normal range encode to a signed zero either way)
  const float rs = __frcp_rn(s);
  const bool rcp_ok = rcp_division_ok(s, rs);
  auto quant8 = [&](const float* t, int64_t idx) {
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float a0 = t[4 * h + 2 * j], a1 = t[4 * h + 2 * j + 1];
        const uint32_t pair = f32x2_to_e4m3x2(rcp_ok ? div_by_rcp(a0, s, rs) : __fdiv_rn(a0, s),
                                              rcp_ok ? div_by_rcp(a1, s, rs) : __fdiv_rn(a1, s));
        if (j == 0) lo = pair; else hi = pair;
      }
      w[h] = lo | (hi << 16);
    }
    *reinterpret_cast<uint2*>(qr + idx * 8) = make_uint2(w[0], w[1]);
  };
#pragma unroll
  for (int i = 0; i < kMaxVecPerThread; ++i) {
    const int idx = tid + i * kQuantThreads;
    if (idx < nvec) quant8(v[i], idx);
  }
  for (int idx = tid + kMaxVecPerThread * kQuantThreads; idx < nvec; idx += kQuantThreads) {
    float t[8];
    Vec8Loader<DT>::load(xr + (int64_t)idx * 8 * elem_bytes<DT>(), t);
    quant8(t, idx);
  }
}

// RMSNorm fused with the per-token quantizers ("Chapter 9 - Quantization
// kernels", practical notes: the per-row max and the quantization fused into
// the upstream operator; "LLM and AIGC quantization", "Static and dynamic
// quantization": the per-token reduction is usually fused into the
// preceding RMSNorm): y = (x / sqrt(mean(x^2) + eps)) . gamma, then the
// symmetric int8 (FMT 0) or the E4M3 (FMT 1) quantization of y, without
// rounding y to the input dtype.  The row is read once.  y is computed as
// (x . inv) . gamma with inv = 1 / sqrt(mean(x^2) + eps) (one correctly
// rounded square root and division per row); a row whose mean(x^2) + eps is
// 0 normalizes to 0.
// The mean of squares is the exact sum of the row's squares rounded once to
// float32 (exact_sum_squares_cta), divided by K in float32: the result does
// not depend on the number of threads or on the order of the additions.
template <int DT, int FMT>
__global__ void __launch_bounds__(kQuantThreads) rmsnorm_quant_kernel(const void* __restrict__ x,
                                                                     const void* __restrict__ gamma, int K,
                                                                     float eps, void* __restrict__ q,
                                                                     float* __restrict__ scale) {
  pdl_launch_dependents();  // the GEMM that reads the codes may start setting up
  const int64_t row = blockIdx.x;
  const int tid = threadIdx.x;
  const int nvec = K / 8;
  constexpr int EB = elem_bytes<DT>();
  const char* xr = static_cast<const char*>(x) + row * (int64_t)K * EB;
  const char* gr = static_cast<const char*>(gamma);

  float v[kMaxVecPerThread][8];
#pragma unroll
  for (int i = 0; i < kMaxVecPerThread; ++i) {
    const int c = tid + i * kQuantThreads;
    if (c < nvec) Vec8Loader<DT>::load(xr + (int64_t)c * 8 * EB, v[i]);
  }
  // every element of this thread's share: the chunks held in registers, then
  // (rows longer than the registers hold) the rest read again
  auto for_each = [&](auto f) {
#pragma unroll
    for (int i = 0; i < kMaxVecPerThread; ++i) {
      const int c = tid + i * kQuantThreads;
      if (c < nvec) {
#pragma unroll
        for (int j = 0; j < 8; ++j) f(v[i][j]);
      }
    }
    for (int c = tid + kMaxVecPerThread * kQuantThreads; c < nvec; c += kQuantThreads) {
      float t[8];
      Vec8Loader<DT>::load(xr + (int64_t)c * 8 * EB, t);
#pragma unroll
      for (int j = 0; j < 8; ++j) f(t[j]);
    }
  };
  __shared__ ExactSqScratch<kQuantThreads / 32> sq;
  __shared__ float red[kQuantThreads / 32];
  __shared__ float s_scale;
  float sumsq;
  if constexpr (DT == 0)
    sumsq = exact_sum_squares_f16_cta<kQuantThreads / 32>(for_each, sq);
  else
    sumsq = exact_sum_squares_cta<kQuantThreads / 32, DT == 1 ? 32 : 0>(for_each, sq);
  const float ms = __fdiv_rn(sumsq, static_cast<float>(K));
  const float r = __fsqrt_rn(__fadd_rn(ms, eps));
  const float s_inv = r == 0.0f ? 0.0f : __fdiv_rn(1.0f, r);
  const float inv = s_inv;
  // y = (x . inv) . gamma
  auto normalize = [&](float* t, int c) {
    float gv[8];
    Vec8Loader<DT>::load(gr + (int64_t)c * 8 * EB, gv);
#pragma unroll
    for (int j = 0; j < 8; ++j) t[j] = __fmul_rn(__fmul_rn(t[j], inv), gv[j]);
  };
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxVecPerThread; ++i) {
    const int c = tid + i * kQuantThreads;
    if (c < nvec) {
      normalize(v[i], c);
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[i][j]));
    }
  }
  for (int c = tid + kMaxVecPerThread * kQuantThreads; c < nvec; c += kQuantThreads) {
    float t[8];
    Vec8Loader<DT>::load(xr + (int64_t)c * 8 * EB, t);
    normalize(t, c);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(t[j]));
  }
  // max is exact, so this reduction's order does not matter
  m = warp_max(m);
  if ((tid & 31) == 0) red[tid >> 5] = m;
  __syncthreads();
  if (tid == 0) {
    float a = red[0];
    for (int w = 1; w < kQuantThreads / 32; ++w) a = fmaxf(a, red[w]);
    const float sv = (a == 0.0f) ? 1.0f : __fdiv_rn(a, FMT == 0 ? 127.0f : 448.0f);
    s_scale = sv;
    scale[row] = sv;
  }
  __syncthreads();
  const float s = s_scale;
  const float rs = __frcp_rn(s);
  const bool srcp_ok = rcp_division_ok(s, rs);
  auto quant8 = [&](const float* t, int c) {
    uint32_t w0 = 0, w1 = 0;
    if (FMT == 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        int qi = __float2int_rn(srcp_ok ? div_by_rcp(t[j], s, rs) : __fdiv_rn(t[j], s));
        qi = min(max(qi, -127), 127);
        const uint32_t byte = static_cast<uint32_t>(qi) & 0xffu;
        if (j < 4) w0 |= byte << (8 * j); else w1 |= byte << (8 * (j - 4));
      }
    } else {
      uint32_t pr[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        pr[j] = f32x2_to_e4m3x2(srcp_ok ? div_by_rcp(t[2 * j], s, rs) : __fdiv_rn(t[2 * j], s),
                                srcp_ok ? div_by_rcp(t[2 * j + 1], s, rs) : __fdiv_rn(t[2 * j + 1], s));
      w0 = pr[0] | (pr[1] << 16);
      w1 = pr[2] | (pr[3] << 16);
    }
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(q) + row * (int64_t)K + (int64_t)c * 8) = make_uint2(w0, w1);
  };
#pragma unroll
  for (int i = 0; i < kMaxVecPerThread; ++i) {
    const int c = tid + i * kQuantThreads;
    if (c < nvec) quant8(v[i], c);
  }
  for (int c = tid + kMaxVecPerThread * kQuantThreads; c < nvec; c += kQuantThreads) {
    float t[8];
    Vec8Loader<DT>::load(xr + (int64_t)c * 8 * EB, t);
    normalize(t, c);
    quant8(t, c);
  }
}

// Exact fp16 copies of int8 codes: 16 codes per thread (one 16-byte load,
// two 16-byte stores), grid-stride; the last count % 16 codes one by one.
__global__ void int8_to_f16_kernel(const int8_t* __restrict__ src, int64_t count, __half* __restrict__ dst) {
  const int64_t nvec = count / 16;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < nvec; v += stride) {
    const uint4 u = ldg_v4(src + v * 16);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t h[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 lo = __halves2half2(__short2half_rn(static_cast<int8_t>(w[i] & 0xFF)),
                                        __short2half_rn(static_cast<int8_t>((w[i] >> 8) & 0xFF)));
      const __half2 hi = __halves2half2(__short2half_rn(static_cast<int8_t>((w[i] >> 16) & 0xFF)),
                                        __short2half_rn(static_cast<int8_t>(w[i] >> 24)));
      h[2 * i] = *reinterpret_cast<const uint32_t*>(&lo);
      h[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&hi);
    }
    uint4* d = reinterpret_cast<uint4*>(dst + v * 16);
    d[0] = make_uint4(h[0], h[1], h[2], h[3]);
    d[1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
  if (blockIdx.x == 0)
    for (int64_t i = nvec * 16 + threadIdx.x; i < count; i += blockDim.x) dst[i] = __short2half_rn(src[i]);
}

// azp_adj[n] = sum_k b[n,k]: one warp per row, 16 bytes per lane per step.
__global__ void int8_row_sum_kernel(const int8_t* __restrict__ b, int64_t N, int K, int32_t* __restrict__ out) {
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= N) return;
  const int8_t* br = b + row * (int64_t)K;
  int acc = 0;
  for (int off = lane * 16; off < K; off += 32 * 16) {
    const uint4 u = ldg_v4(br + off);
    acc = __dp4a(static_cast<int>(u.x), 0x01010101, acc);
    acc = __dp4a(static_cast<int>(u.y), 0x01010101, acc);
    acc = __dp4a(static_cast<int>(u.z), 0x01010101, acc);
    acc = __dp4a(static_cast<int>(u.w), 0x01010101, acc);
  }
  acc = warp_sum_int(acc);
  if (lane == 0) out[row] = acc;
}

// Asymmetric 4-bit group quantization: one warp per row and pair of
// 128-element groups; lane l covers 8 consecutive elements, lanes 0-15 the
// first group and 16-31 the second.
template <int DT>
__global__ void quant_w4_g128_kernel(const void* __restrict__ w, int64_t N, int K, uint8_t* __restrict__ wq,
                                     __half* __restrict__ scales, uint8_t* __restrict__ zeros) {
  const int G = K / 128;
  const int pairs = (G + 1) / 2;
  const int64_t item = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (item >= N * pairs) return;
  const int64_t row = item / pairs;
  const int p = static_cast<int>(item % pairs);
  const int lane = threadIdx.x & 31;
  const int grp = 2 * p + (lane >> 4);
  const bool active = grp < G;
  const int k0 = grp * 128 + (lane & 15) * 8;

  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float mn = 0.0f, mx = 0.0f;
  if (active) {
    Vec8Loader<DT>::load(static_cast<const char*>(w) + (row * (int64_t)K + k0) * elem_bytes<DT>(), v);
    mn = v[0]; mx = v[0];
#pragma unroll
    for (int j = 1; j < 8; ++j) { mn = fminf(mn, v[j]); mx = fmaxf(mx, v[j]); }
  }
  // reduce within each 16-lane half
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const __half s16 = __float2half_rn(__fdiv_rn(fmaxf(__fsub_rn(mx, mn), 1e-5f), 15.0f));
  const float s = __half2float(s16);
  const int z = min(max(__float2int_rn(__fdiv_rn(-mn, s)), 0), 15);
  uint32_t packed = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int c = min(max(__float2int_rn(__fdiv_rn(v[j], s)) + z, 0), 15);
    packed |= static_cast<uint32_t>(c) << (4 * j);
  }
  const int z_hi = __shfl_down_sync(0xffffffffu, z, 16);
  if (active) {
    *reinterpret_cast<uint32_t*>(wq + row * (int64_t)(K / 2) + k0 / 2) = packed;
    if ((lane & 15) == 0) scales[row * G + grp] = s16;
  }
  if (lane == 0) {
    const int hi = (2 * p + 1 < G) ? z_hi : 0;
    zeros[row * (int64_t)pairs + p] = static_cast<uint8_t>(z | (hi << 4));
  }
}

}  // namespace

// Launched without the programmatic-serialization attribute: the kernel reads
// x at its start, with no griddepcontrol.wait before it, so it must not
// overlap the kernel that writes x.
namespace {
template <bool F16>
void quant_act_int8_dispatch(const void* x, qlin_dtype x_dtype, int64_t T, int64_t K, void* q, float* scale,
                             int32_t* azp, cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(T)), block(kQuantThreads);
  const int k = static_cast<int>(K);
  const bool asym = azp != nullptr;
  switch (x_dtype) {
    case QLIN_F16:
      if (k <= 2 * 8 * kQuantThreads) {
        if (asym) quant_int8_rows_kernel<0, true, F16, 2><<<grid, block, 0, stream>>>(x, k, q, scale, azp);
        else quant_int8_rows_kernel<0, false, F16, 2><<<grid, block, 0, stream>>>(x, k, q, scale, azp);
      } else {
        if (asym) quant_int8_rows_kernel<0, true, F16, 4><<<grid, block, 0, stream>>>(x, k, q, scale, azp);
        else quant_int8_rows_kernel<0, false, F16, 4><<<grid, block, 0, stream>>>(x, k, q, scale, azp);
      }
      break;
    case QLIN_BF16:
      if (k <= 2 * 8 * kQuantThreads) {
        if (asym) quant_int8_rows_kernel<1, true, F16, 2><<<grid, block, 0, stream>>>(x, k, q, scale, azp);
        else quant_int8_rows_kernel<1, false, F16, 2><<<grid, block, 0, stream>>>(x, k, q, scale, azp);
      } else {
        if (asym) quant_int8_rows_kernel<1, true, F16, 4><<<grid, block, 0, stream>>>(x, k, q, scale, azp);
        else quant_int8_rows_kernel<1, false, F16, 4><<<grid, block, 0, stream>>>(x, k, q, scale, azp);
      }
      break;
    default:
      if (k <= 2 * 8 * kQuantThreads) {
        if (asym) quant_int8_rows_kernel<2, true, F16, 2><<<grid, block, 0, stream>>>(x, k, q, scale, azp);
        else quant_int8_rows_kernel<2, false, F16, 2><<<grid, block, 0, stream>>>(x, k, q, scale, azp);
      } else {
        if (asym) quant_int8_rows_kernel<2, true, F16, 4><<<grid, block, 0, stream>>>(x, k, q, scale, azp);
        else quant_int8_rows_kernel<2, false, F16, 4><<<grid, block, 0, stream>>>(x, k, q, scale, azp);
      }
      break;
  }
}
}  // namespace

cudaError_t launch_quant_act_int8(const void* x, qlin_dtype x_dtype, int64_t T, int64_t K, void* q, bool f16_codes,
                                  float* scale, int32_t* azp, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  if (f16_codes) quant_act_int8_dispatch<true>(x, x_dtype, T, K, q, scale, azp, stream);
  else quant_act_int8_dispatch<false>(x, x_dtype, T, K, q, scale, azp, stream);
  return cudaGetLastError();
}

// Launched without the programmatic-serialization attribute: the kernel reads
// x at its start, with no griddepcontrol.wait before it, so it must not
// overlap the kernel that writes x.
cudaError_t launch_quant_fp8(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, uint8_t* q, float* scale,
                             cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(rows)), block(kQuantThreads);
  const int k = static_cast<int>(K);
  switch (x_dtype) {
    case QLIN_F16: quant_fp8_rows_kernel<0><<<grid, block, 0, stream>>>(x, k, q, scale); break;
    case QLIN_BF16: quant_fp8_rows_kernel<1><<<grid, block, 0, stream>>>(x, k, q, scale); break;
    default: quant_fp8_rows_kernel<2><<<grid, block, 0, stream>>>(x, k, q, scale); break;
  }
  return cudaGetLastError();
}

// Launched without the programmatic-serialization attribute: the kernel reads
// x at its start, with no griddepcontrol.wait before it, so it must not
// overlap the kernel that writes x.
cudaError_t launch_rmsnorm_quant(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, const void* gamma,
                                 float eps, qlin_qfmt fmt, void* q, float* scale, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>(rows)), block(kQuantThreads);
  const int k = static_cast<int>(K);
  const bool fp8 = fmt == QLIN_QFMT_FP8_E4M3;
  switch (x_dtype) {
    case QLIN_F16:
      if (fp8) rmsnorm_quant_kernel<0, 1><<<grid, block, 0, stream>>>(x, gamma, k, eps, q, scale);
      else rmsnorm_quant_kernel<0, 0><<<grid, block, 0, stream>>>(x, gamma, k, eps, q, scale);
      break;
    case QLIN_BF16:
      if (fp8) rmsnorm_quant_kernel<1, 1><<<grid, block, 0, stream>>>(x, gamma, k, eps, q, scale);
      else rmsnorm_quant_kernel<1, 0><<<grid, block, 0, stream>>>(x, gamma, k, eps, q, scale);
      break;
    default:
      if (fp8) rmsnorm_quant_kernel<2, 1><<<grid, block, 0, stream>>>(x, gamma, k, eps, q, scale);
      else rmsnorm_quant_kernel<2, 0><<<grid, block, 0, stream>>>(x, gamma, k, eps, q, scale);
      break;
  }
  return cudaGetLastError();
}

cudaError_t launch_int8_to_f16(const int8_t* src, int64_t count, void* dst, cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  const int64_t nvec = count / 16;
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((nvec + 255) / 256, 8 * sm_count()));
  int8_to_f16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(src, count, static_cast<__half*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_int8_row_sum(const int8_t* b, int64_t N, int64_t K, int32_t* out, cudaStream_t stream) {
  if (N == 0) return cudaSuccess;
  const int warps = 8;
  dim3 grid(static_cast<unsigned>((N + warps - 1) / warps)), block(32 * warps);
  int8_row_sum_kernel<<<grid, block, 0, stream>>>(b, N, static_cast<int>(K), out);
  return cudaGetLastError();
}

cudaError_t launch_quant_w4_g128(const void* w, qlin_dtype w_dtype, int64_t N, int64_t K, uint8_t* wq,
                                 void* scales, uint8_t* zeros, cudaStream_t stream) {
  if (N == 0) return cudaSuccess;
  const int64_t pairs = (K / 128 + 1) / 2;
  const int64_t items = N * pairs;
  const int warps = 8;
  dim3 grid(static_cast<unsigned>((items + warps - 1) / warps)), block(32 * warps);
  __half* s = static_cast<__half*>(scales);
  const int k = static_cast<int>(K);
  switch (w_dtype) {
    case QLIN_F16: quant_w4_g128_kernel<0><<<grid, block, 0, stream>>>(w, N, k, wq, s, zeros); break;
    case QLIN_BF16: quant_w4_g128_kernel<1><<<grid, block, 0, stream>>>(w, N, k, wq, s, zeros); break;
    default: quant_w4_g128_kernel<2><<<grid, block, 0, stream>>>(w, N, k, wq, s, zeros); break;
  }
  return cudaGetLastError();
}

}  // namespace qlin
