// NVFP4 quantization with ARCQuant residual channels, and its two set-up
// helpers (per-tensor scale, channel order).
//
// Per 16-element block b of a row of the reordered channels xs = x[:, perm]
// ("LLM and AIGC quantization: from number formats to W4A4", block-scaled
// formats, the 16-element NVFP4 example; "NVFP4 quantization and ARCQuant",
// sections 2.1 and 3.1):
//   sf_b = E4M3( (max_b |xs| / 6) / g )     round-to-nearest-even, saturating
//   d_b  = dec(sf_b) . g
//   q    = E2M1( xs / d_b )                 round-to-nearest-even, saturating
// The first S reordered channels then get, in columns K .. K+S-1, either the
// NVFP4 re-quantization of the residual r = xs - e2m1(q) . d_b (activations)
// or a copy of their codes and scales (weights: "copy rather than compute").
//
// Every rounding decision is taken in IEEE float32 as written (true division,
// separate multiply and subtract; the 16 divisions of a block by its d go
// through the correctly rounded reciprocal plus one FMA correction, which
// gives the same quotients); the E4M3 and E2M1 encodes use the hardware's
// round-to-nearest-even saturating conversions.
#include <type_traits>

#include "device_common.cuh"
#include "exact_sumsq.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace {

constexpr int kNvThreads = 256;

__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}

__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  uint32_t h2;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h2) : "r"(code));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// Two floats -> one byte of two E2M1 codes, `lo` in bits 0-3, `hi` in 4-7.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// One byte of two E2M1 codes -> the two values (low nibble first).
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t byte) {
  uint32_t h2;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h2) : "r"(byte));
  const __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// x / d from r = __frcp_rn(d) by one FMA correction step (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", 1990), with the sign taken from x.  Equal to __fdiv_rn(x, d)
// when d, r and the quotient are normal; a quotient below the normal range
// comes out as a tiny number or zero with the sign of x (a zero dividend
// keeps its sign, which the correction's +0 would otherwise drop).
__device__ __forceinline__ float div_rcp_signed(float x, float d, float r) {
  const float q0 = __fmul_rn(x, r);
  const float q = __fmaf_rn(__fmaf_rn(-q0, d, x), r, q0);
  return __int_as_float((__float_as_int(q) & 0x7FFFFFFF) | (__float_as_int(x) & static_cast<int>(0x80000000u)));
}

constexpr float kMinNormal = 1.17549435e-38f;
constexpr float kMaxFinite = 3.40282347e38f;

// Per-tensor scale g with its reciprocal, and whether s / g may go through
// the reciprocal (g and 1/g normal).
struct GlobalScale {
  float g, rg;
  bool fast;
};

__device__ __forceinline__ GlobalScale make_global_scale(float g) {
  GlobalScale gs;
  gs.g = g;
  gs.rg = __frcp_rn(g);
  gs.fast = fabsf(g) >= kMinNormal && fabsf(g) <= kMaxFinite && fabsf(gs.rg) >= kMinNormal && fabsf(gs.rg) <= kMaxFinite;
  return gs;
}

// (amax / 6) / g with both divisions correctly rounded.  The reciprocal path
// is taken only where it provably gives the same float (normal operands and
// quotients); every other case uses the division itself.
__device__ __forceinline__ float block_scale_value(float amax, const GlobalScale& gs) {
  if (amax == 0.0f) return 0.0f;
  const float r6 = 0.166666672f;  // float nearest 1/6
  const float s1 = (amax >= 6.0f * kMinNormal && amax <= kMaxFinite)
                       ? __fmaf_rn(__fmaf_rn(-__fmul_rn(amax, r6), 6.0f, amax), r6, __fmul_rn(amax, r6))
                       : __fdiv_rn(amax, 6.0f);
  if (gs.fast) {
    const float s2 = __fmaf_rn(__fmaf_rn(-__fmul_rn(s1, gs.rg), gs.g, s1), gs.rg, __fmul_rn(s1, gs.rg));
    if (s2 >= kMinNormal && s2 <= kMaxFinite) return s2;
  }
  return __fdiv_rn(s1, gs.g);
}

// Quantize one 16-element block; returns the scale code, writes 8 code bytes.
__device__ __forceinline__ uint32_t quant_block16(const float* v, const GlobalScale& gs, uint32_t* packed /*[2]*/,
                                                  float* d_out) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint32_t sfc = f32_to_e4m3(block_scale_value(amax, gs));
  const float d = __fmul_rn(e4m3_to_f32(sfc), gs.g);
  packed[0] = 0u;
  packed[1] = 0u;
  if (d != 0.0f) {
    // The 16 quotients share d.  Through the reciprocal when d and 1/d are
    // normal and no quotient can overflow (|x r| <= amax r finite): a
    // quotient below the normal range rounds to a zero code either way.
    const float rd = __frcp_rn(d);
    if (fabsf(d) >= kMinNormal && rd >= kMinNormal && __fmul_rn(amax, rd) <= 1.0e38f) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t byte = f32x2_to_e2m1x2(div_rcp_signed(v[2 * i], d, rd), div_rcp_signed(v[2 * i + 1], d, rd));
        packed[i >> 2] |= byte << (8 * (i & 3));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t byte = f32x2_to_e2m1x2(__fdiv_rn(v[2 * i], d), __fdiv_rn(v[2 * i + 1], d));
        packed[i >> 2] |= byte << (8 * (i & 3));
      }
    }
  }
  *d_out = d;
  return sfc;
}

// Eight consecutive staged elements (16 or 32 bytes of shared memory) as float32.
template <int DT>
__device__ __forceinline__ void smem_chunk8(const unsigned char* p, float* v) {
  if constexpr (DT == 2) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 c = *reinterpret_cast<const float4*>(p + 16);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
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

// 1 / sqrt(mean(x^2) + eps) of each of the nr staged rows into inv[] (0 where
// the root is 0), every thread of the CTA taking part: the mean of squares is
// the exact sum of the row's squares rounded once to float32, divided by K
// (the definition of the fused RMSNorm quantizers; exact_sum_squares_cta).
template <int DT, int R>
__device__ void staged_rows_inv_rms(const unsigned char* rows_smem, int row_bytes, int nr, int K, float eps,
                                    ExactSqScratch<kNvThreads / 32>& sq, float* inv) {
  constexpr int EB = elem_bytes<DT>();
  const int tid = threadIdx.x;
#pragma unroll
  for (int rr = 0; rr < R; ++rr) {
    if (rr >= nr) break;  // uniform over the CTA
    const unsigned char* rs = rows_smem + rr * row_bytes;
    auto for_each = [&](auto f) {
      for (int c = tid; c * 8 < K; c += kNvThreads) {
        float v[8];
        smem_chunk8<DT>(rs + c * 8 * EB, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) f(v[i]);
      }
    };
    float sumsq;
    if constexpr (DT == 0)
      sumsq = exact_sum_squares_f16_cta<kNvThreads / 32>(for_each, sq);
    else
      sumsq = exact_sum_squares_cta<kNvThreads / 32, DT == 1 ? 32 : 0>(for_each, sq);
    if (tid == 0) {
      const float r = __fsqrt_rn(__fadd_rn(__fdiv_rn(sumsq, static_cast<float>(K)), eps));
      inv[rr] = r == 0.0f ? 0.0f : __fdiv_rn(1.0f, r);
    }
  }
  __syncthreads();
}

// R rows per CTA: the rows are staged in shared memory in their input dtype,
// then each thread quantizes 16-element blocks of the reordered rows; the
// block's 16 channel offsets are loaded and checked once for all R rows.
// NORM: RMSNorm fused in front (gamma staged after the rows, in its own
// order, and gathered with the same offsets as the row elements).
template <int DT, int R, bool NORM>
__global__ void __launch_bounds__(kNvThreads) nvfp4_quant_kernel(const void* __restrict__ x, int64_t rows, int K,
                                                                  const int32_t* __restrict__ perm, int S,
                                                                  int mode, const float* __restrict__ gp,
                                                                  uint8_t* __restrict__ q,
                                                                  uint8_t* __restrict__ sf, int sf_mma,
                                                                  const void* __restrict__ gamma, float eps,
                                                                  int32_t* __restrict__ err) {
  extern __shared__ __align__(16) unsigned char row_smem[];
  pdl_launch_dependents();  // the GEMM that reads the codes may start setting up
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * R;
  const int nr = static_cast<int>(min(static_cast<int64_t>(R), rows - row0));
  const int tid = threadIdx.x;
  constexpr int EB = elem_bytes<DT>();
  const int row_bytes = K * EB;
  unsigned char* gamma_smem = row_smem + R * row_bytes;
  {
    const char* xr = static_cast<const char*>(x) + row0 * row_bytes;
    for (int off = tid * 16; off < nr * row_bytes; off += kNvThreads * 16)
      *reinterpret_cast<uint4*>(row_smem + off) = ldg_v4(xr + off);
    if constexpr (NORM) {
      for (int off = tid * 16; off < row_bytes; off += kNvThreads * 16)
        *reinterpret_cast<uint4*>(gamma_smem + off) = ldg_v4(static_cast<const char*>(gamma) + off);
    }
  }
  __syncthreads();
  // fused RMSNorm: each staged row's 1 / rms
  __shared__ float inv_rms[R];
  if constexpr (NORM) {
    __shared__ ExactSqScratch<kNvThreads / 32> sq;
    staged_rows_inv_rms<DT, R>(row_smem, row_bytes, nr, K, eps, sq, inv_rms);
  }

  const GlobalScale gs = make_global_scale(__ldg(gp));
  const int Kaug = K + S;
  const int nblk = K / 16;
  const int sblk = S / 16;
  for (int b = tid; b < nblk; b += kNvThreads) {
    // byte offsets of the block's channels in a staged row; a channel index
    // outside [0, K) is recorded in the device error word and read as K-1,
    // so the shared-memory gather stays in bounds
    uint32_t off[16];
    if (perm != nullptr) {
      const int4* pp = reinterpret_cast<const int4*>(perm + b * 16);
      uint32_t pmax = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int4 p4 = __ldg(pp + i);
        const uint32_t c[4] = {static_cast<uint32_t>(p4.x), static_cast<uint32_t>(p4.y),
                               static_cast<uint32_t>(p4.z), static_cast<uint32_t>(p4.w)};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          pmax = max(pmax, c[j]);
          off[4 * i + j] = min(c[j], static_cast<uint32_t>(K - 1)) * EB;
        }
      }
      if (pmax >= static_cast<uint32_t>(K)) record_device_error(err, kDevErrBadIndex);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) off[i] = (b * 16 + i) * EB;
    }
    // fused RMSNorm: the block's gamma at the channels' original positions
    float gv[16];
    if constexpr (NORM) {
#pragma unroll
      for (int i = 0; i < 16; ++i) gv[i] = load_elem<DT>(gamma_smem + off[i], 0);
    }
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      if (rr >= nr) break;
      const int64_t row = row0 + rr;
      const unsigned char* rs = row_smem + rr * row_bytes;
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = load_elem<DT>(rs + off[i], 0);
      if constexpr (NORM) {
        const float inv = inv_rms[rr];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(__fmul_rn(v[i], inv), gv[i]);
      }
      uint32_t packed[2];
      float d;
      const uint32_t sfc = quant_block16(v, gs, packed, &d);
      uint8_t* qr = q + row * (int64_t)(Kaug / 2);
      // position of the scale of block j of this row in either layout
      const int64_t sf_row_base = sf_mma ? ((row >> 7) * (int64_t)(Kaug / 64)) * 512 + 16 * (row & 31) +
                                               4 * ((row & 127) >> 5)
                                         : row * (int64_t)(Kaug / 16);
      auto sf_at = [&](int j) -> uint8_t& {
        return sf_mma ? sf[sf_row_base + (int64_t)(j >> 2) * 512 + (j & 3)] : sf[sf_row_base + j];
      };
      *reinterpret_cast<uint2*>(qr + b * 8) = make_uint2(packed[0], packed[1]);
      sf_at(b) = static_cast<uint8_t>(sfc);
      if (b < sblk) {
        if (mode == QLIN_NVFP4_DUPLICATE) {
          *reinterpret_cast<uint2*>(qr + (K / 2) + b * 8) = make_uint2(packed[0], packed[1]);
          sf_at(nblk + b) = static_cast<uint8_t>(sfc);
        } else {
          // residual r = x - e2m1(q) * d, one float32 multiply then one subtract
          float r[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float2 e = e2m1x2_to_f32x2((packed[i >> 2] >> (8 * (i & 3))) & 0xFFu);
            r[2 * i] = __fsub_rn(v[2 * i], __fmul_rn(e.x, d));
            r[2 * i + 1] = __fsub_rn(v[2 * i + 1], __fmul_rn(e.y, d));
          }
          uint32_t rp[2];
          float rd;
          const uint32_t rsf = quant_block16(r, gs, rp, &rd);
          *reinterpret_cast<uint2*>(qr + (K / 2) + b * 8) = make_uint2(rp[0], rp[1]);
          sf_at(nblk + b) = static_cast<uint8_t>(rsf);
        }
      }
    }
  }
}

// max |x| over the tensor into the bits of *g (non-negative floats order like
// their bit patterns); *g must be zero beforehand.
template <int DT>
__global__ void absmax_bits_kernel(const void* __restrict__ x, int64_t nvec, unsigned int* __restrict__ out) {
  float m = 0.0f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += (int64_t)gridDim.x * blockDim.x) {
    float v[8];
    Vec8Loader<DT>::load(static_cast<const char*>(x) + i * 8 * elem_bytes<DT>(), v);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) atomicMax(out, __float_as_uint(m));
}

__global__ void global_scale_finish_kernel(float* g) {
  *g = __fdiv_rn(*g, 2688.0f);  // 6 * 448
}

// Column maxima of |x| into the bits of perm[k]; perm must be zero beforehand.
// Thread handles 8 consecutive columns over a slice of rows.
template <int DT>
__global__ void col_absmax_kernel(const void* __restrict__ x, int64_t rows, int K, int rows_per_cta,
                                  unsigned int* __restrict__ out) {
  const int vec = blockIdx.x * blockDim.x + threadIdx.x;
  if (vec * 8 >= K) return;
  const int64_t r0 = (int64_t)blockIdx.y * rows_per_cta;
  const int64_t r1 = min(rows, r0 + rows_per_cta);
  float m[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int64_t r = r0; r < r1; ++r) {
    float v[8];
    Vec8Loader<DT>::load(static_cast<const char*>(x) + (r * K + (int64_t)vec * 8) * elem_bytes<DT>(), v);
#pragma unroll
    for (int j = 0; j < 8; ++j) m[j] = fmaxf(m[j], fabsf(v[j]));
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) atomicMax(out + vec * 8 + j, __float_as_uint(m[j]));
}

// Single-CTA bitonic sort of (statistic, channel) keys: ascending order of
// (~bits << 32 | channel) is descending statistic with ties by channel.
__global__ void __launch_bounds__(1024) perm_sort_kernel(int32_t* __restrict__ perm, int K, int n_pow2) {
  extern __shared__ unsigned long long keys[];
  for (int i = threadIdx.x; i < n_pow2; i += blockDim.x) {
    keys[i] = (i < K) ? ((static_cast<unsigned long long>(~static_cast<unsigned int>(perm[i])) << 32) |
                         static_cast<unsigned int>(i))
                      : ~0ull;
  }
  __syncthreads();
  for (int size = 2; size <= n_pow2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n_pow2; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;
          const unsigned long long a = keys[i], b = keys[j];
          if ((a > b) == up) { keys[i] = b; keys[j] = a; }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < K; i += blockDim.x) perm[i] = static_cast<int32_t>(keys[i] & 0xFFFFFFFFull);
}

// Row-major scales [rows][K/16] -> the MMA layout: one thread per (padded
// row, 64-element K block) moves 4 bytes; rows past `rows` are zero.
__global__ void sf_to_mma_kernel(const uint8_t* __restrict__ src, int rows, int K, uint8_t* __restrict__ dst) {
  const int KG = K / 64;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t prow = ((int64_t)rows + 127) / 128 * 128;
  if (i >= prow * KG) return;
  const int row = static_cast<int>(i / KG), kg = static_cast<int>(i % KG);
  const uint32_t v = row < rows ? *reinterpret_cast<const uint32_t*>(src + (int64_t)row * (K / 16) + 4 * kg) : 0u;
  const int64_t off = ((int64_t)(row >> 7) * KG + kg) * 512 + 16 * (row & 31) + 4 * ((row & 127) >> 5);
  *reinterpret_cast<uint32_t*>(dst + off) = v;
}

template <typename F>
cudaError_t dispatch_dtype(qlin_dtype dt, F&& f) {
  switch (dt) {
    case QLIN_F16: return f(std::integral_constant<int, 0>{});
    case QLIN_BF16: return f(std::integral_constant<int, 1>{});
    default: return f(std::integral_constant<int, 2>{});
  }
}

}  // namespace

// Launched without the programmatic-serialization attribute: the kernel reads
// x at its start, with no griddepcontrol.wait before it, so it must not
// overlap the kernel that writes x.
cudaError_t launch_quant_nvfp4(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, const int32_t* perm,
                               int64_t S, qlin_nvfp4_mode mode, const float* g, uint8_t* q, uint8_t* sf,
                               qlin_sf_layout sf_layout, const void* gamma, float eps, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  return dispatch_dtype(x_dtype, [&](auto dt) -> cudaError_t {
    constexpr int DT = decltype(dt)::value;
    const size_t row_smem = static_cast<size_t>(K) * elem_bytes<DT>();
    auto launch = [&](auto rows_per_cta, auto norm) -> cudaError_t {
      constexpr int R = decltype(rows_per_cta)::value;
      constexpr bool NORM = decltype(norm)::value;
      const size_t smem = row_smem * (R + (NORM ? 1 : 0));
      auto kern = nvfp4_quant_kernel<DT, R, NORM>;
      // the opt-in covers dynamic plus static shared memory above the 48 KB default
      if (smem + 4 * 1024 > 48 * 1024) {
        cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern));
        if (e != cudaSuccess) return e;
      }
      kern<<<static_cast<unsigned>((rows + R - 1) / R), kNvThreads, smem, stream>>>(
          x, rows, static_cast<int>(K), perm, static_cast<int>(S), static_cast<int>(mode), g, q, sf,
          sf_layout == QLIN_SF_MMA ? 1 : 0, gamma, eps, device_error_word());
      return cudaGetLastError();
    };
    // two rows per CTA share the channel offsets (and gamma) while both fit comfortably
    const bool two = 2 * row_smem <= 96 * 1024;
    if (gamma != nullptr)
      return two ? launch(std::integral_constant<int, 2>{}, std::true_type{})
                 : launch(std::integral_constant<int, 1>{}, std::true_type{});
    return two ? launch(std::integral_constant<int, 2>{}, std::false_type{})
               : launch(std::integral_constant<int, 1>{}, std::false_type{});
  });
}

cudaError_t launch_nvfp4_sf_to_mma(const uint8_t* src, int64_t rows, int64_t K, uint8_t* dst, cudaStream_t stream) {
  const int64_t n = (rows + 127) / 128 * 128 * (K / 64);
  if (n == 0) return cudaSuccess;
  sf_to_mma_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(src, static_cast<int>(rows),
                                                                              static_cast<int>(K), dst);
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_global_scale(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, float* g,
                                      cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(g, 0, sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const int64_t nvec = rows * K / 8;
  if (nvec > 0) {
    e = dispatch_dtype(x_dtype, [&](auto dt) -> cudaError_t {
      constexpr int DT = decltype(dt)::value;
      int64_t blocks = (nvec + 255) / 256;
      const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
      if (blocks > cap) blocks = cap;
      absmax_bits_kernel<DT><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
          x, nvec, reinterpret_cast<unsigned int*>(g));
      return cudaGetLastError();
    });
    if (e != cudaSuccess) return e;
  }
  global_scale_finish_kernel<<<1, 1, 0, stream>>>(g);
  return cudaGetLastError();
}

cudaError_t launch_arc_perm(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, int32_t* perm,
                            cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(perm, 0, sizeof(int32_t) * K, stream);
  if (e != cudaSuccess) return e;
  if (rows > 0) {
    e = dispatch_dtype(x_dtype, [&](auto dt) -> cudaError_t {
      constexpr int DT = decltype(dt)::value;
      const int vecs = static_cast<int>(K / 8);
      const int threads = 128;
      const int rows_per_cta = 64;
      dim3 grid((vecs + threads - 1) / threads, static_cast<unsigned>((rows + rows_per_cta - 1) / rows_per_cta));
      col_absmax_kernel<DT><<<grid, threads, 0, stream>>>(x, rows, static_cast<int>(K), rows_per_cta,
                                                          reinterpret_cast<unsigned int*>(perm));
      return cudaGetLastError();
    });
    if (e != cudaSuccess) return e;
  }
  int n = 1;
  while (n < K) n <<= 1;
  const size_t smem = sizeof(unsigned long long) * n;
  if (smem > 48 * 1024) {
    e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(perm_sort_kernel));
    if (e != cudaSuccess) return e;
  }
  perm_sort_kernel<<<1, 1024, smem, stream>>>(perm, static_cast<int>(K), n);
  return cudaGetLastError();
}

}  // namespace qlin
