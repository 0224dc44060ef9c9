// NVFP4 W4A4: block-scaled fp4 GEMM on the tcgen05 tensor cores
//
//   Y[t,n] = g_a . g_b . sum_b sfa[t,b] . sfb[n,b] . sum_{k in b} a[t,k] . b[n,k]
//
// E2M1 elements, one E4M3 scale per 16 elements along K, fp32 accumulation,
// per-tensor fp32 scales applied once in the epilogue ("LLM and AIGC
// quantization: from number formats to W4A4", block-scaled formats: the
// tensor core reads the elements and the block scales and scales each block
// during accumulation; "NVFP4 quantization and ARCQuant", section 2.2: the
// residual channels are extra K columns of the same GEMM).
//
// Kernel structure (one CTA per 128 x 128 output tile, 10 warps):
//   warp 0      TMA producer: packed codes of A and B, 128 rows x 128 bytes
//               (256 elements) per stage, landing in the 128-byte swizzled
//               K-major layout the MMA descriptors describe.
//   warp 1      TMEM allocation and the MMA issuer: per stage, tcgen05.cp of
//               the stage's scale factors from shared memory into TMEM, then
//               4 x tcgen05.mma kind::mxf4nvf4.block_scale.scale_vec::4X
//               (M=128, N=128, K=64).
//   warps 2-5   scale-factor loaders: the row-major E4M3 scales of the
//               stage's 128 A rows and 128 B rows are rearranged into the
//               32-row x 16-byte blocks that tcgen05.cp copies (byte
//               16*(r%32) + 4*(r/32) + j holds row r, K block j of one MMA).
//   warps 6-9   epilogue: the 128 x 128 fp32 accumulator from TMEM, times
//               g_a . g_b, rounded once to bf16 / fp16.
// Every barrier wait is bounded; on expiry the kernel records the site in the
// device error word, stops issuing work, waits (bounded) for copies and MMAs
// already in flight, frees TMEM and exits.
#include <cuda.h>

#include "device_common.cuh"
#include "qlin_internal.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace qlin {
namespace {

constexpr int kBM = 128, kBN = 128;
constexpr int kBKB = 128;                 // bytes of packed codes per row per stage (256 elements)
constexpr int kMmaPerStage = 4;           // K = 64 elements each
constexpr int kStages = 4;
constexpr int kThreads = 320;
constexpr int kAccCols = kBN;
constexpr int kSfColsPerStage = 2 * kMmaPerStage * 4;  // A and B, 4 TMEM columns per MMA
constexpr int kTmemCols = 256;            // accumulator (128) + scale factors (4 stages x 32)

constexpr int kCodeBytes = (kBM + kBN) * kBKB;           // 32 KB per stage
constexpr int kSfBytes = 2 * kMmaPerStage * 512;         // 4 KB per stage
constexpr int kSmemCodes = 0;
constexpr int kSmemSf = kSmemCodes + kStages * kCodeBytes;          // 128 KB
constexpr int kSmemBar = kSmemSf + kStages * kSfBytes;              // +16 KB
constexpr int kNumBars = 2 * kStages + 2;
constexpr int kSmemMisc = kSmemBar + kNumBars * 8;
constexpr int kSmemTotal = kSmemMisc + 16 + 1024;

enum { kSiteEmpty = 1, kSiteFull, kSiteAcc, kSiteDrain };

__global__ void __launch_bounds__(kThreads, 1) nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                                                                 const __grid_constant__ CUtensorMap tmB,
                                                                 const uint8_t* __restrict__ sfa,
                                                                 const uint8_t* __restrict__ sfb, int T, int N,
                                                                 int K, const float* __restrict__ g_a,
                                                                 const float* __restrict__ g_b,
                                                                 void* __restrict__ out, int out_dtype,
                                                                 int32_t* __restrict__ err) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  const int KB = K / 2;                       // packed bytes per row
  const int SFK = K / 16;                     // scale factors per row
  const int num_kb = (KB + kBKB - 1) / kBKB;  // stages

  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t bar0 = sbase + kSmemBar;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  const uint32_t acc_full = bar0 + 8u * (2 * kStages);
  const uint32_t mma_done = bar0 + 8u * (2 * kStages + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemMisc + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(full(s), 1 + 4);  // TMA producer + 4 scale-factor warps
      tc::mbar_init(empty(s), 1);     // MMA commit
    }
    tc::mbar_init(acc_full, 1);
    tc::mbar_init(mma_done, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_sf = tmem + kAccCols;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tc::prefetch_tmap(&tmA);
      tc::prefetch_tmap(&tmB);
      int issued = 0;
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % kStages;
        if (kb >= kStages && !tc::mbar_wait(empty(s), ((kb / kStages) - 1) & 1, err, kSiteEmpty)) {
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        const uint32_t dst = sbase + kSmemCodes + s * kCodeBytes;
        tc::mbar_arrive_expect_tx(full(s), kCodeBytes);
        tc::tma_load_2d(dst, &tmA, kb * kBKB, m0, full(s));
        tc::tma_load_2d(dst + kBM * kBKB, &tmB, kb * kBKB, n0, full(s));
        issued = kb + 1;
      }
      if (*abort_flag) {
        for (int kb = (issued > kStages ? issued - kStages : 0); kb < issued; ++kb)
          tc::mbar_wait(full(kb % kStages), (kb / kStages) & 1, err, kSiteDrain);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_nvf4(kBM, kBN);
      bool issued_any = false;
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % kStages;
        if (!tc::mbar_wait(full(s), (kb / kStages) & 1, err, kSiteFull)) { *abort_flag = 1; break; }
        if (*abort_flag) break;
        tc::tc_fence_after();
        const uint32_t sf_smem = sbase + kSmemSf + s * kSfBytes;
        const uint32_t sf_t = tmem_sf + s * kSfColsPerStage;
        // scale factors of this stage: A blocks then B blocks, 4 columns each
#pragma unroll
        for (int i = 0; i < 2 * kMmaPerStage; ++i) tc::tmem_cp_32x128b_x4(sf_t + 4 * i, tc::plain_desc(sf_smem + 512 * i));
        const uint32_t a_base = sbase + kSmemCodes + s * kCodeBytes;
        const uint32_t b_base = a_base + kBM * kBKB;
        const int kk_valid = min(kMmaPerStage, (KB - kb * kBKB) / 32);
#pragma unroll
        for (int kk = 0; kk < kMmaPerStage; ++kk) {
          if (kk < kk_valid) {
            tc::mma_nvf4(tmem, tc::sw128_kmajor_desc(a_base + 32 * kk), tc::sw128_kmajor_desc(b_base + 32 * kk),
                         idesc, sf_t + 4 * kk, sf_t + 4 * (kMmaPerStage + kk), (kb > 0 || kk > 0) ? 1u : 0u);
          }
        }
        issued_any = true;
        tc::mma_commit(empty(s));
      }
      if (!*abort_flag) {
        tc::mma_commit(acc_full);
      } else if (issued_any) {
        tc::mma_commit(mma_done);
        tc::mbar_wait(mma_done, 0, err, kSiteDrain);
      }
    }
  } else if (warp < 6) {
    // ---------------- scale-factor loaders ----------------
    const int r = threadIdx.x - 64;  // row within the tile, 0..127
    const int ra = m0 + r, rb = n0 + r;
    const uint32_t blk_off = 16u * (r & 31) + 4u * (r >> 5);
    for (int kb = 0; kb < num_kb; ++kb) {
      const int s = kb % kStages;
      bool ok = kb < kStages || tc::mbar_wait(empty(s), ((kb / kStages) - 1) & 1, err, kSiteEmpty);
      ok = __all_sync(0xffffffffu, ok && !*abort_flag);
      if (!ok) { *abort_flag = 1; break; }
      uint32_t va[kMmaPerStage], vb[kMmaPerStage];
#pragma unroll
      for (int kk = 0; kk < kMmaPerStage; ++kk) {
        const int j = kb * (kBKB / 8) + 4 * kk;  // first scale factor of this MMA's K block
        const bool kin = j < SFK;                 // SFK is a multiple of 4
        va[kk] = (kin && ra < T) ? __ldg(reinterpret_cast<const uint32_t*>(sfa + (int64_t)ra * SFK + j)) : 0u;
        vb[kk] = (kin && rb < N) ? __ldg(reinterpret_cast<const uint32_t*>(sfb + (int64_t)rb * SFK + j)) : 0u;
      }
      uint32_t* sf = reinterpret_cast<uint32_t*>(smem + kSmemSf + s * kSfBytes);
#pragma unroll
      for (int kk = 0; kk < kMmaPerStage; ++kk) {
        sf[(512 * kk + blk_off) / 4] = va[kk];
        sf[(512 * (kMmaPerStage + kk) + blk_off) / 4] = vb[kk];
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(full(s));
    }
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;
    const int row = m0 + q * 32 + lane;
    bool ok = tc::mbar_wait(acc_full, 0, err, kSiteAcc);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc::tc_fence_after();
      const float alpha = __ldg(g_a) * __ldg(g_b);
#pragma unroll
      for (int cg = 0; cg < kBN / 32; ++cg) {
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + cg * 32, v);
        tc::tmem_wait_ld();
        if (row < T) {
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            const int col = n0 + cg * 32 + c8 * 8;
            if (col >= N) continue;
            uint4 pk;
            uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float f0 = __uint_as_float(v[c8 * 8 + 2 * i]) * alpha;
              const float f1 = __uint_as_float(v[c8 * 8 + 2 * i + 1]) * alpha;
              if (out_dtype == QLIN_BF16) {
                __nv_bfloat162 h = __floats2bfloat162_rn(f0, f1);
                pw[i] = *reinterpret_cast<uint32_t*>(&h);
              } else {
                __half2 h = __floats2half2_rn(f0, f1);
                pw[i] = *reinterpret_cast<uint32_t*>(&h);
              }
            }
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + (int64_t)row * N + col) = pk;
          }
        }
      }
    } else {
      *abort_flag = 1;
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_nvfp4_gemm(const uint8_t* a, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb,
                              int64_t T, int64_t N, int64_t K, const float* g_a, const float* g_b, void* out,
                              qlin_dtype out_dtype, cudaStream_t stream) {
  if (T == 0 || N == 0) return cudaSuccess;
  CUtensorMap tmA, tmB;
  cudaError_t st = make_tmap_2d_u8(&tmA, a, static_cast<uint64_t>(K / 2), static_cast<uint64_t>(T), kBKB, kBM,
                                   /*swizzle128=*/true);
  if (st != cudaSuccess) return st;
  st = make_tmap_2d_u8(&tmB, b, static_cast<uint64_t>(K / 2), static_cast<uint64_t>(N), kBKB, kBN, true);
  if (st != cudaSuccess) return st;
  st = cudaFuncSetAttribute(nvfp4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTotal);
  if (st != cudaSuccess) return st;
  dim3 grid(static_cast<unsigned>((N + kBN - 1) / kBN), static_cast<unsigned>((T + kBM - 1) / kBM));
  nvfp4_gemm_kernel<<<grid, kThreads, kSmemTotal, stream>>>(tmA, tmB, sfa, sfb, static_cast<int>(T),
                                                            static_cast<int>(N), static_cast<int>(K), g_a, g_b, out,
                                                            static_cast<int>(out_dtype), device_error_word());
  return cudaGetLastError();
}

}  // namespace qlin
