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
// The fragment mapping and the unpack are in w4a16_mma_common.cuh.
#include <mutex>

#include "device_common.cuh"
#include "qlin_internal.h"
#include "tc_common.cuh"
#include "w4a16_mma_common.cuh"

namespace qlin {
namespace {

using namespace w4mma;

constexpr int kW4Group = 128;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Wait until at most `pending` of this thread's most recent cp.async groups
// are still in flight (the count must be an immediate, hence the switch).
__device__ __forceinline__ void cp_async_wait_pending(int pending) {
  switch (pending) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
  }
}

// Groups one CTA handles at most; longer rows are split over a cluster.
constexpr int kW4MaxGroupsPerCta = 32;

// Shared-memory plan of one CTA (16 output rows, W warps, GPW groups per warp,
// GC groups of K, Tc tokens, C CTAs in the cluster).
struct W4Smem {
  int w_off, s_off, z_off, x_off, r_off, c_off, total;
};

__host__ __device__ inline W4Smem w4_smem_plan(int W, int GPW, int GC, int Tc, int NT, int C) {
  W4Smem p;
  p.w_off = 0;                                   // [W][GPW][2 rows][32 lanes] x 16 B
  p.s_off = p.w_off + W * GPW * 2 * 32 * 16;     // [16 rows][GC] fp16 scales
  p.z_off = p.s_off + ((16 * GC * 2 + 15) / 16) * 16;   // [16 rows][GC] zero-points, one per byte
  p.x_off = p.z_off + ((16 * GC + 15) / 16) * 16;       // [Tc][GC*16] activation chunks (16 B)
  p.r_off = p.x_off + Tc * GC * 16 * 16;                // [W][32][NT*4] fp32 partial sums
  p.c_off = p.r_off + W * 32 * NT * 4 * 4;              // [C][32][NT*4] cluster partial sums
  p.total = p.c_off + C * 32 * NT * 4 * 4;
  return p;
}

// One cluster of C CTAs per 16 output rows; CTA r of the cluster handles the
// groups [r*GC, min((r+1)*GC, G)) of K and its warps split those groups
// (warp w takes groups w, w + W, ...).  Every thread copies its own 16-byte
// weight slices into shared memory with cp.async at the start, the scales,
// zero-points and activations of the CTA's K range follow asynchronously, so
// a CTA has all of its operands in flight at once and nothing of the stream
// is held in registers.  Partial sums are added across warps through shared
// memory and across the cluster through distributed shared memory into CTA 0,
// always in the same order.
template <int NT>
__global__ void __launch_bounds__(256) w4a16_mma_kernel(const __half* __restrict__ x, int Tc, int N, int K,
                                                       const uint8_t* __restrict__ wq,
                                                       const __half* __restrict__ scales,
                                                       const uint8_t* __restrict__ zeros, int zpitch, int GC,
                                                       int GPW, __half* __restrict__ y, int ldy) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = blockDim.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int G = K / kW4Group;
  const int C = gridDim.x / ((N + 15) / 16) ;  // CTAs per cluster (grid is C x row blocks)
  const uint32_t rank = C > 1 ? cluster_rank() : 0;
  const int gs = rank * GC;
  const int gn = max(0, min(GC, G - gs));      // groups of this CTA
  const W4Smem plan = w4_smem_plan(W, GPW, GC, Tc, NT, C);
  uint4* wbuf = reinterpret_cast<uint4*>(smem + plan.w_off);
  __half* sbuf = reinterpret_cast<__half*>(smem + plan.s_off);
  uint8_t* zbuf = smem + plan.z_off;
  uint4* xbuf = reinterpret_cast<uint4*>(smem + plan.x_off);
  float* red = reinterpret_cast<float*>(smem + plan.r_off);
  float* cred = reinterpret_cast<float*>(smem + plan.c_off);

  const int row0 = (blockIdx.x / C) * 16;
  const int rA = row0 + g, rB = rA + 8;
  // Rows past N read row N-1 (always in bounds); their results are not stored.
  const int rAc = min(rA, N - 1), rBc = min(rB, N - 1);

  // 1. The weight stream: every group of this warp, both rows, in flight.
  {
    const uint8_t* wA = wq + (int64_t)rAc * (K / 2) + gs * (kW4Group / 2) + c * 16;
    const uint8_t* wB = wq + (int64_t)rBc * (K / 2) + gs * (kW4Group / 2) + c * 16;
    uint4* mine = wbuf + (size_t)warp * GPW * 64 + lane;
    for (int i = 0; i < GPW; ++i) {
      const int grp = warp + i * W;
      if (grp < gn) {
        cp_async16(tc::smem_u32(mine + i * 64), wA + grp * (kW4Group / 2));
        cp_async16(tc::smem_u32(mine + i * 64 + 32), wB + grp * (kW4Group / 2));
      }
      cp_async_commit();  // one group per K group, consumed in order below
    }
  }
  // 2. Scales and zero-points of the CTA's rows and groups, into registers
  //    first (all loads issued before any store waits on one).
  //    Thread t covers row t / 16 and groups t % 16, t % 16 + 16 (GC <= 32).
  const int mr = threadIdx.x >> 4, mg = threadIdx.x & 15;
  const bool meta_row = mr < 16;
  __half sv[2];
  uint8_t zv[2];
  if (meta_row) {
    const int64_t row = min(row0 + mr, N - 1);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int grp = mg + 16 * j;
      if (grp < gn) {
        const int ga = gs + grp;
        sv[j] = scales[row * G + ga];
        zv[j] = zeros ? static_cast<uint8_t>((zeros[row * zpitch + (ga >> 1)] >> (4 * (ga & 1))) & 0xF)
                      : static_cast<uint8_t>(8);
      }
    }
  }
  pdl_launch_dependents();
  // 3. Activations (may be produced by the previous kernel in the stream),
  //    loaded to registers and stored in the pair order of the MMA fragments:
  //    (x[8m+j], x[8m+j+4]), j = 0..3.
  pdl_wait();
  const int XC = gn * 16;  // 16-byte chunks per token in this CTA's K range
  for (int tok = 0; tok < Tc; ++tok) {
    const __half* xr = x + (int64_t)tok * K + gs * kW4Group;
    uint4* xs_row = xbuf + (size_t)tok * GC * 16;
    constexpr int kXU = 2;
    for (int m0 = threadIdx.x; m0 < XC; m0 += kXU * blockDim.x) {
      uint4 u[kXU];
#pragma unroll
      for (int j = 0; j < kXU; ++j) {
        const int m = m0 + j * blockDim.x;
        if (m < XC) u[j] = ldg_cg_v4(xr + m * 8);
      }
#pragma unroll
      for (int j = 0; j < kXU; ++j) {
        const int m = m0 + j * blockDim.x;
        if (m < XC) {
          uint32_t q[4];
          pair_x(u[j], q);
          xs_row[m] = make_uint4(q[0], q[1], q[2], q[3]);
        }
      }
    }
  }
  if (meta_row) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int grp = mg + 16 * j;
      if (grp < gn) {
        sbuf[mr * GC + grp] = sv[j];
        zbuf[mr * GC + grp] = zv[j];
      }
    }
  }
  __syncthreads();

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;

  const uint4* mine = wbuf + (size_t)warp * GPW * 64 + lane;
  for (int i = 0; i < GPW; ++i) {
    const int grp = warp + i * W;
    if (grp >= gn) break;
    cp_async_wait_pending(GPW - 1 - i);
    const uint4 qa = mine[i * 64], qb = mine[i * 64 + 32];
    const uint32_t zA = zbuf[g * GC + grp], zB = zbuf[(g + 8) * GC + grp];
    const float sA = __half2float(sbuf[g * GC + grp]);
    const float sB = __half2float(sbuf[(g + 8) * GC + grp]);
    // half2 constants 1024 + z and -(64 + z), built with integer ops
    const uint32_t subA = 0x64006400u | (zA << 16) | zA, addA = 0xD400D400u | (zA << 20) | (zA << 4);
    const uint32_t subB = 0x64006400u | (zB << 16) | zB, addB = 0xD400D400u | (zB << 20) | (zB << 4);

    // A fragments of the 8 MMAs of this group: MMA m uses word m/2 and pairs
    // 2(m%2), 2(m%2)+1.
    uint32_t fa[8][4];
    const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
    const uint32_t wb[4] = {qb.x, qb.y, qb.z, qb.w};
    const UnpackConsts uk = unpack_consts();
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t pa[4], pb[4];
      unpack_word(wa[w], subA, addA, uk, pa);
      unpack_word(wb[w], subB, addB, uk, pb);
      fa[2 * w][0] = pa[0]; fa[2 * w][1] = pb[0]; fa[2 * w][2] = pa[1]; fa[2 * w][3] = pb[1];
      fa[2 * w + 1][0] = pa[2]; fa[2 * w + 1][1] = pb[2]; fa[2 * w + 1][2] = pa[3]; fa[2 * w + 1][3] = pb[3];
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int tok = nt * 8 + g;
      uint4 xp[4];
      if (tok < Tc) {
        const uint4* xr = xbuf + (size_t)tok * GC * 16 + grp * 16 + c * 4;
#pragma unroll
        for (int w = 0; w < 4; ++w) xp[w] = xr[w];
      } else {
#pragma unroll
        for (int w = 0; w < 4; ++w) xp[w] = make_uint4(0u, 0u, 0u, 0u);
      }
      // two independent accumulator chains, added at the end of the group
      float p0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, p1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        mma_16816(p0, fa[2 * w], xp[w].x, xp[w].y);
        mma_16816(p1, fa[2 * w + 1], xp[w].z, xp[w].w);
      }
      acc[nt][0] = fmaf(sA, p0[0] + p1[0], acc[nt][0]);
      acc[nt][1] = fmaf(sA, p0[1] + p1[1], acc[nt][1]);
      acc[nt][2] = fmaf(sB, p0[2] + p1[2], acc[nt][2]);
      acc[nt][3] = fmaf(sB, p0[3] + p1[3], acc[nt][3]);
    }
  }

  // Add the warps' partial sums in a fixed order.
  float* slot = red + ((size_t)warp * 32 + lane) * (NT * 4);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) slot[nt * 4 + i] = acc[nt][i];
  __syncthreads();
  float v[NT][4];
  if (warp == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int i = 0; i < 4; ++i) v[nt][i] = 0.0f;
      for (int wdx = 0; wdx < W; ++wdx) {
        const float* p = red + ((size_t)wdx * 32 + lane) * (NT * 4) + nt * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[nt][i] += p[i];
      }
    }
  }
  if (C > 1) {
    // Send this CTA's sums to CTA 0 of the cluster, then CTA 0 adds them in
    // rank order.
    if (warp == 0) {
      const uint32_t dst = map_to_rank(tc::smem_u32(cred + ((size_t)rank * 32 + lane) * (NT * 4)), 0);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) st_cluster_f32(dst + (nt * 4 + i) * 4, v[nt][i]);
    }
    cluster_sync_all();
    if (rank != 0 || warp != 0) return;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int i = 0; i < 4; ++i) v[nt][i] = 0.0f;
      for (int r = 0; r < C; ++r) {
        const float* p = cred + ((size_t)r * 32 + lane) * (NT * 4) + nt * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[nt][i] += p[i];
      }
    }
  } else if (warp != 0) {
    return;
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    // c0, c1: row g, tokens 2c, 2c+1; c2, c3: row g + 8, same tokens.
    const int t0 = nt * 8 + 2 * c, t1 = t0 + 1;
    if (rA < N) {
      if (t0 < Tc) y[(int64_t)t0 * ldy + rA] = __float2half_rn(v[nt][0]);
      if (t1 < Tc) y[(int64_t)t1 * ldy + rA] = __float2half_rn(v[nt][1]);
    }
    if (rB < N) {
      if (t0 < Tc) y[(int64_t)t0 * ldy + rB] = __float2half_rn(v[nt][2]);
      if (t1 < Tc) y[(int64_t)t1 * ldy + rB] = __float2half_rn(v[nt][3]);
    }
  }
}

// Shared memory a launch may use for staged activations.
constexpr size_t kW4XBudget = 64 * 1024;

template <int NT>
cudaError_t launch_chunk(const __half* x, int Tc, int N, int K, const uint8_t* wq, const __half* scales,
                         const uint8_t* zeros, __half* y, int ldy, cudaStream_t stream) {
  const int G = K / kW4Group;
  const int C = (G + kW4MaxGroupsPerCta - 1) / kW4MaxGroupsPerCta;   // CTAs per cluster
  const int GC = (G + C - 1) / C;                                     // groups per CTA
  const int W = 8;  // the scale / zero-point staging below assumes 256 threads
  const int GPW = (GC + W - 1) / W;
  const W4Smem plan = w4_smem_plan(W, GPW, GC, Tc, NT, C);
  const void* fn = reinterpret_cast<const void*>(w4a16_mma_kernel<NT>);
  cudaError_t e = ensure_max_dynamic_smem(fn);
  if (e != cudaSuccess) return e;
  if (C > 8) {
    // clusters above the portable 8 CTAs: allowed once per device
    static std::once_flag once[64];
    static cudaError_t status[64];
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    } else {
      std::call_once(once[dev], [&] {
        status[dev] = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      });
      e = status[dev];
    }
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C * ((N + 15) / 16));
  cfg.blockDim = dim3(32 * W);
  cfg.dynamicSmemBytes = plan.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, w4a16_mma_kernel<NT>, x, Tc, N, K, wq, scales, zeros, (G + 1) / 2, GC, GPW, y,
                            ldy);
}

// The fallback for shapes without a skinny plan: one launch per chunk of
// tokens that the activation staging budget allows.
cudaError_t launch_w4a16_mma(const void* x, int64_t T, int64_t N, int64_t K, const uint8_t* wq, const void* scales,
                             const uint8_t* zeros, void* y, cudaStream_t stream) {
  const int t = static_cast<int>(T), n = static_cast<int>(N), k = static_cast<int>(K);
  const __half* xh = static_cast<const __half*>(x);
  const __half* sh = static_cast<const __half*>(scales);
  __half* yh = static_cast<__half*>(y);
  // Tokens per launch: as many as the staging budget allows, at most 16.
  const int G = k / kW4Group;
  const int C = (G + kW4MaxGroupsPerCta - 1) / kW4MaxGroupsPerCta;
  const int GC = (G + C - 1) / C;
  int tc_max = static_cast<int>(kW4XBudget / ((size_t)GC * kW4Group * 2));
  tc_max = tc_max < 1 ? 1 : (tc_max > 16 ? 16 : tc_max);
  for (int t0 = 0; t0 < t; t0 += tc_max) {
    const int tc = (t - t0) < tc_max ? (t - t0) : tc_max;
    const __half* xc = xh + (int64_t)t0 * k;
    __half* yc = yh + (int64_t)t0 * n;
    cudaError_t e = (tc <= 8) ? launch_chunk<1>(xc, tc, n, k, wq, sh, zeros, yc, n, stream)
                              : launch_chunk<2>(xc, tc, n, k, wq, sh, zeros, yc, n, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

// Dispatch: one token on the CUDA-core GEMV, up to 16 tokens per launch on
// the streamed tensor-core skinny kernel (more tokens in chunks of 16, each
// chunk one pass over the weights), and the staged kernel above for shapes
// the skinny kernel has no plan for.
// Above this many tokens the tensor-core prefill GEMM runs instead of the
// skinny kernel (16 tokens per launch, the weights read once per launch):
// measured on the Llama-2-7B shapes, one skinny launch wins at 16 tokens, the
// prefill GEMM (128-token tiles, K shared by up to four CTAs) from 17 on
// (17-32 tokens: 12.6 / 25.2 / 22.2 us against 18.1 / 29.9 / 35.7 us for two
// skinny launches on 4096x4096 / 11008x4096 / 4096x11008).
constexpr int64_t kW4a16PrefillMinT = 16;

cudaError_t launch_w4a16_gemm_grouped(const void* x, int64_t T, int64_t K, int count, const int64_t* N,
                                      const uint8_t* const* wq, const void* const* scales,
                                      const uint8_t* const* zeros, void* const* y, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  if (count < 1 || count > QLIN_W4A16_MAX_GROUP) return cudaErrorInvalidValue;
  int64_t total = 0;
  for (int p = 0; p < count; ++p) total += N[p];
  if (total == 0) return cudaSuccess;
  if (w4a16_gemv_supported(T, total, K)) return launch_w4a16_gemv_grouped(x, K, count, N, wq, scales, zeros, y, stream);
  // many tokens: one tensor-core GEMM per matrix, weights dequantized on chip
  if (T > kW4a16PrefillMinT) {
    bool all = true;
    for (int p = 0; p < count; ++p) all = all && (N[p] == 0 || w4a16_prefill_supported(T, N[p], K));
    if (all) {
      for (int p = 0; p < count; ++p) {
        if (N[p] == 0) continue;
        cudaError_t e = launch_w4a16_prefill(x, T, N[p], K, wq[p], scales[p], zeros[p], y[p], stream);
        if (e != cudaSuccess) return e;
      }
      return cudaSuccess;
    }
  }
  constexpr int64_t kChunk = 16;
  const int64_t first = T < kChunk ? T : kChunk, last = T % kChunk;
  if (w4a16_skinny_supported(first, total, K) && (last == 0 || w4a16_skinny_supported(last, total, K))) {
    for (int64_t t0 = 0; t0 < T; t0 += kChunk) {
      const int64_t tc = T - t0 < kChunk ? T - t0 : kChunk;
      void* yc[QLIN_W4A16_MAX_GROUP];
      for (int p = 0; p < count; ++p) yc[p] = static_cast<__half*>(y[p]) + t0 * N[p];
      cudaError_t e = launch_w4a16_skinny_grouped(static_cast<const __half*>(x) + t0 * K, tc, K, count, N, wq, scales,
                                                  zeros, yc, stream);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  for (int p = 0; p < count; ++p) {
    if (N[p] == 0) continue;
    cudaError_t e = launch_w4a16_mma(x, T, N[p], K, wq[p], scales[p], zeros[p], y[p], stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_w4a16_gemm(const void* x, int64_t T, int64_t N, int64_t K, const uint8_t* wq,
                              const void* scales, const uint8_t* zeros, void* y, cudaStream_t stream) {
  if (T == 0 || N == 0) return cudaSuccess;
  return launch_w4a16_gemm_grouped(x, T, K, 1, &N, &wq, &scales, &zeros, &y, stream);
}

}  // namespace qlin
