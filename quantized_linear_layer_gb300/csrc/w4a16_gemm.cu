// W4A16 fused dequant GEMV / skinny GEMM for decode shapes (T <= 64).
//
//   Y[t,n] = sum_g s[n,g] . sum_{k in g} X[t,k] . (q[n,k] - z[n,g])
//
// ("Chapter 9 - Quantization kernels", 9.5: dequantize in registers right
// before the tensor core, HBM and SMEM only ever hold the 4-bit codes; 9.6:
// the magic-number unpack; "LLM and AIGC quantization", W4A16 section.)
//
// Design for GB300.  Decode reads every weight byte once, so the kernel is
// bound by HBM: it streams the packed codes with 16-byte non-allocating loads
// (each thread keeps several in flight) and spends as few instructions per
// code as possible.  The 4-bit codes are turned into exact fp16 integers
// (q - z) with two bit operations and one half2 subtract / fma per pair of
// codes, the zero-point folded into that subtract (the constants are built
// from z with integer ops).  The exact fp16 values feed the warp-level
// m16n8k16 tensor-core MMA with the weight rows as the M side and the tokens
// as the N side, so a decode token costs no CUDA-core FMAs at all: products
// are exact and accumulate in fp32 inside one 128-element group; the group
// scale is applied once per group in fp32.  Warps of a CTA split K; their
// partial sums are added in a fixed order through shared memory.
//
// Fragment mapping.  Thread (g, c) = (lane / 4, lane % 4) loads 16 bytes (32
// codes) of rows g and g + 8 at K offset 32c within a group.  Each 32-bit word
// holds eight consecutive codes k .. k+7; the unpack yields the half2 pairs
// (k, k+4), (k+1, k+5), (k+2, k+6), (k+3, k+7).  These pairs are assigned to
// the MMA's logical K slots (2c, 2c+1) and (2c+8, 2c+9); the activation
// fragment of the same thread is built with exactly the same assignment, so
// the product over a group covers every K index once.
#include "device_common.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace {

constexpr int kW4Group = 128;
constexpr int kW4Batch = 4;  // groups whose weight loads are in flight together

__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b),
                      *reinterpret_cast<__half2*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ void mma_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Exact fp16 (q - z) pairs from one word of eight codes.
//   out[0] = (k, k+4), out[1] = (k+1, k+5), out[2] = (k+2, k+6), out[3] = (k+3, k+7)
// 0x6400 is fp16 1024: OR-ing a nibble n into its low mantissa bits gives
// 1024 + n, and 1024 + 16n for the nibble one position higher.
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t sub, uint32_t add, uint32_t* out) {
  const uint32_t kLo = 0x000F000Fu, kHi = 0x00F000F0u, kEx = 0x64006400u, kSixteenth = 0x2C002C00u;
  out[0] = h2_sub((w & kLo) | kEx, sub);                 // (1024 + n) - (1024 + z)
  out[1] = h2_fma((w & kHi) | kEx, kSixteenth, add);     // (1024 + 16n) / 16 - (64 + z)
  const uint32_t w8 = w >> 8;
  out[2] = h2_sub((w8 & kLo) | kEx, sub);
  out[3] = h2_fma((w8 & kHi) | kEx, kSixteenth, add);
}

// Activation pairs (x[k+j], x[k+j+4]) for j = 0..3 from eight consecutive fp16.
__device__ __forceinline__ void pair_x(uint4 u, uint32_t* out) {
  out[0] = __byte_perm(u.x, u.z, 0x5410);
  out[1] = __byte_perm(u.x, u.z, 0x7632);
  out[2] = __byte_perm(u.y, u.w, 0x5410);
  out[3] = __byte_perm(u.y, u.w, 0x7632);
}

template <int NT>
__global__ void __launch_bounds__(256) w4a16_mma_kernel(const __half* __restrict__ x, int T, int N, int K,
                                                       const uint8_t* __restrict__ wq,
                                                       const __half* __restrict__ scales,
                                                       const uint8_t* __restrict__ zeros, int zpitch,
                                                       __half* __restrict__ y) {
  extern __shared__ float red[];  // [warps][32 lanes][NT * 4]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int G = K / kW4Group;
  const int rA = blockIdx.x * 16 + g, rB = rA + 8;
  // Rows past N read row N-1 (always in bounds); their results are not stored.
  const int rAc = min(rA, N - 1), rBc = min(rB, N - 1);
  const uint8_t* wA = wq + (int64_t)rAc * (K / 2) + c * 16;
  const uint8_t* wB = wq + (int64_t)rBc * (K / 2) + c * 16;

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;

  for (int gb = warp * kW4Batch; gb < G; gb += nwarps * kW4Batch) {
    uint4 qa[kW4Batch], qb[kW4Batch];
#pragma unroll
    for (int i = 0; i < kW4Batch; ++i) {
      if (gb + i < G) {
        qa[i] = ldg_stream_v4(wA + (gb + i) * (kW4Group / 2));
        qb[i] = ldg_stream_v4(wB + (gb + i) * (kW4Group / 2));
      }
    }
#pragma unroll
    for (int i = 0; i < kW4Batch; ++i) {
      const int grp = gb + i;
      if (grp >= G) break;
      uint32_t zA = 8, zB = 8;
      if (zeros != nullptr) {
        zA = (zeros[(int64_t)rAc * zpitch + (grp >> 1)] >> (4 * (grp & 1))) & 0xF;
        zB = (zeros[(int64_t)rBc * zpitch + (grp >> 1)] >> (4 * (grp & 1))) & 0xF;
      }
      const float sA = __half2float(scales[(int64_t)rAc * G + grp]);
      const float sB = __half2float(scales[(int64_t)rBc * G + grp]);
      // half2 constants 1024 + z and -(64 + z), built with integer ops
      const uint32_t subA = 0x64006400u | (zA << 16) | zA, addA = 0xD400D400u | (zA << 20) | (zA << 4);
      const uint32_t subB = 0x64006400u | (zB << 16) | zB, addB = 0xD400D400u | (zB << 20) | (zB << 4);

      // A fragments of the 8 MMAs of this group: MMA m uses word m/2 and
      // pairs 2(m%2), 2(m%2)+1.
      uint32_t fa[8][4];
      const uint32_t wa[4] = {qa[i].x, qa[i].y, qa[i].z, qa[i].w};
      const uint32_t wb[4] = {qb[i].x, qb[i].y, qb[i].z, qb[i].w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t pa[4], pb[4];
        unpack_word(wa[w], subA, addA, pa);
        unpack_word(wb[w], subB, addB, pb);
        fa[2 * w][0] = pa[0]; fa[2 * w][1] = pb[0]; fa[2 * w][2] = pa[1]; fa[2 * w][3] = pb[1];
        fa[2 * w + 1][0] = pa[2]; fa[2 * w + 1][1] = pb[2]; fa[2 * w + 1][2] = pa[3]; fa[2 * w + 1][3] = pb[3];
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tok = nt * 8 + g;
        uint32_t xp[4][4];  // [word w][pair j]
        if (tok < T) {
          const __half* xr = x + (int64_t)tok * K + grp * kW4Group + c * 32;
#pragma unroll
          for (int w = 0; w < 4; ++w) pair_x(ldg_v4(xr + 8 * w), xp[w]);
        } else {
#pragma unroll
          for (int w = 0; w < 4; ++w)
#pragma unroll
            for (int j = 0; j < 4; ++j) xp[w][j] = 0u;
        }
        float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int w = m >> 1, j0 = 2 * (m & 1);
          mma_16816(part, fa[m], xp[w][j0], xp[w][j0 + 1]);
        }
        acc[nt][0] = fmaf(sA, part[0], acc[nt][0]);
        acc[nt][1] = fmaf(sA, part[1], acc[nt][1]);
        acc[nt][2] = fmaf(sB, part[2], acc[nt][2]);
        acc[nt][3] = fmaf(sB, part[3], acc[nt][3]);
      }
    }
  }

  // Add the warps' partial sums in a fixed order.
  float* mine = red + ((size_t)warp * 32 + lane) * (NT * 4);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) mine[nt * 4 + i] = acc[nt][i];
  __syncthreads();
  if (warp != 0) return;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int wdx = 0; wdx < nwarps; ++wdx) {
      const float* p = red + ((size_t)wdx * 32 + lane) * (NT * 4) + nt * 4;
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] += p[i];
    }
    // c0, c1: row g, tokens 2c, 2c+1; c2, c3: row g + 8, same tokens.
    const int t0 = nt * 8 + 2 * c, t1 = t0 + 1;
    if (rA < N) {
      if (t0 < T) y[(int64_t)t0 * N + rA] = __float2half_rn(v[0]);
      if (t1 < T) y[(int64_t)t1 * N + rA] = __float2half_rn(v[1]);
    }
    if (rB < N) {
      if (t0 < T) y[(int64_t)t0 * N + rB] = __float2half_rn(v[2]);
      if (t1 < T) y[(int64_t)t1 * N + rB] = __float2half_rn(v[3]);
    }
  }
}

template <int NT>
cudaError_t launch_nt(const void* x, int T, int N, int K, const uint8_t* wq, const void* scales,
                      const uint8_t* zeros, void* y, cudaStream_t stream) {
  const int G = K / kW4Group;
  // Enough warps per CTA to split K; at most 8.
  int warps = (G + kW4Batch - 1) / kW4Batch;
  warps = warps < 1 ? 1 : (warps > 8 ? 8 : warps);
  const size_t smem = (size_t)warps * 32 * NT * 4 * sizeof(float);
  dim3 grid((N + 15) / 16), block(32 * warps);
  w4a16_mma_kernel<NT><<<grid, block, smem, stream>>>(
      static_cast<const __half*>(x), T, N, K, wq, static_cast<const __half*>(scales), zeros, (G + 1) / 2,
      static_cast<__half*>(y));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_w4a16_gemm(const void* x, int64_t T, int64_t N, int64_t K, const uint8_t* wq,
                              const void* scales, const uint8_t* zeros, void* y, cudaStream_t stream) {
  if (T == 0 || N == 0) return cudaSuccess;
  const int t = static_cast<int>(T), n = static_cast<int>(N), k = static_cast<int>(K);
  if (t <= 8) return launch_nt<1>(x, t, n, k, wq, scales, zeros, y, stream);
  if (t <= 16) return launch_nt<2>(x, t, n, k, wq, scales, zeros, y, stream);
  if (t <= 32) return launch_nt<4>(x, t, n, k, wq, scales, zeros, y, stream);
  return launch_nt<8>(x, t, n, k, wq, scales, zeros, y, stream);
}

}  // namespace qlin
