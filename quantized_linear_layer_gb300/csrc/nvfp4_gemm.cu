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
// Persistent kernel: one CTA per SM walks the 128 x 128 output tiles
// (tile = blockIdx.x, + gridDim.x, ...), 7 warps:
//   warp 0      TMA producer: packed codes of A and B, 128 rows x 128 bytes
//               (256 elements) per stage, into the 128-byte swizzled K-major
//               layout the MMA descriptors describe, plus two bulk copies of
//               the stage's E4M3 scales, which are stored in the MMA layout
//               (128-row x 4-block blocks of 512 bytes, byte
//               16*(r%32) + 4*(r/32) + j for row r, K block j) and land exactly
//               as tcgen05.cp reads them.
//   warp 1      TMEM allocation and the MMA issuer: per stage,
//               4 x tcgen05.mma kind::mxf4nvf4.block_scale.scale_vec::4X
//               (M=128, N=128, K=64) into one of two accumulator buffers.
//   warp 6      scale-factor copier: tcgen05.cp of each landed stage's scales
//               into that stage's TMEM slot, handed to the MMA issuer through
//               an mbarrier so the copies run ahead of the MMAs.
//   warps 2-5   epilogue: the fp32 accumulator from TMEM, times g_a . g_b,
//               rounded once to bf16 / fp16; the other accumulator buffer
//               keeps the MMAs of the next tile going meanwhile.
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
constexpr int kStages = 6;
constexpr int kThreads = 224;
constexpr int kAccCols = kBN;
constexpr int kSfColsPerStage = 2 * kMmaPerStage * 4;  // A and B, 4 TMEM columns per MMA
constexpr int kTmemCols = 512;            // 2 accumulators (256) + scale factors (6 stages x 32)

constexpr int kCodeBytes = (kBM + kBN) * kBKB;           // 32 KB per stage
constexpr int kSfBytes = 2 * kMmaPerStage * 512;         // 4 KB per stage
constexpr int kSmemCodes = 0;
constexpr int kSmemSf = kSmemCodes + kStages * kCodeBytes;          // 192 KB
constexpr int kSmemBar = kSmemSf + kStages * kSfBytes;              // +24 KB
constexpr int kNumBars = 3 * kStages + 4 + 2;
constexpr int kSmemMisc = kSmemBar + kNumBars * 8;
constexpr int kSmemTotal = kSmemMisc + 16 + 1024;
static_assert(kSmemTotal <= 227 * 1024, "shared memory budget");
static_assert(2 * kAccCols + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");

enum { kSiteEmpty = 1, kSiteFull, kSiteAccFull, kSiteAccEmpty, kSiteDrain };

// Tile order: groups of 8 M tiles walk all N tiles, so CTAs working at the
// same time share operand tiles in L2.
__device__ __forceinline__ void tile_coords(int tile, int mt_count, int nt_count, int& mt, int& nt) {
  constexpr int kGroup = 8;
  const int per_group = kGroup * nt_count;
  const int grp = tile / per_group;
  const int first_m = grp * kGroup;
  const int rows = min(kGroup, mt_count - first_m);
  const int in = tile - grp * per_group;
  mt = first_m + in % rows;
  nt = in / rows;
}

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
  const int KB = K / 2;                       // packed bytes per row
  const int KG = K / 64;                      // 64-element K blocks (one MMA each)
  const int num_kb = (KB + kBKB - 1) / kBKB;  // stages per tile
  const int mt_count = (T + kBM - 1) / kBM, nt_count = (N + kBN - 1) / kBN;
  const int num_tiles = mt_count * nt_count;
  const int my_tiles = blockIdx.x < num_tiles ? (num_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;

  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t bar0 = sbase + kSmemBar;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto acc_full = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
  const uint32_t mma_done = bar0 + 8u * (2 * kStages + 4);
  auto sf_ready = [&](int s) { return bar0 + 8u * (2 * kStages + 5 + s); };
  const uint32_t cp_done = bar0 + 8u * (3 * kStages + 5);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemMisc + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(full(s), 1);        // TMA producer (codes + scale factors)
      tc::mbar_init(empty(s), 1);       // MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(acc_full(b), 1);
      tc::mbar_init(acc_empty(b), 4);
    }
    tc::mbar_init(mma_done, 1);
    for (int s = 0; s < kStages; ++s) tc::mbar_init(sf_ready(s), 1);  // scale-factor copier commit
    tc::mbar_init(cp_done, 1);
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
  const uint32_t tmem_sf = tmem + 2 * kAccCols;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tc::prefetch_tmap(&tmA);
      tc::prefetch_tmap(&tmB);
      int it = 0, issued = 0;
      for (int ti = 0; ti < my_tiles && !*abort_flag; ++ti) {
        int mt, nt;
        tile_coords(blockIdx.x + ti * gridDim.x, mt_count, nt_count, mt, nt);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % kStages;
          if (it >= kStages && !tc::mbar_wait(empty(s), ((it / kStages) - 1) & 1, err, kSiteEmpty)) {
            *abort_flag = 1;
            break;
          }
          const uint32_t dst = sbase + kSmemCodes + s * kCodeBytes;
          const uint32_t sf_dst = sbase + kSmemSf + s * kSfBytes;
          const int kg0 = kb * kMmaPerStage;                  // first 64-element K block of the stage
          const int nkg = min(kMmaPerStage, KG - kg0);        // blocks of this stage that exist
          tc::mbar_arrive_expect_tx(full(s), kCodeBytes + 2 * nkg * 512);
          tc::tma_load_2d(dst, &tmA, kb * kBKB, mt * kBM, full(s));
          tc::tma_load_2d(dst + kBM * kBKB, &tmB, kb * kBKB, nt * kBN, full(s));
          tc::bulk_load(sf_dst, sfa + ((int64_t)mt * KG + kg0) * 512, nkg * 512, full(s));
          tc::bulk_load(sf_dst + kMmaPerStage * 512, sfb + ((int64_t)nt * KG + kg0) * 512, nkg * 512, full(s));
          issued = it + 1;
        }
      }
      if (*abort_flag) {
        for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
          tc::mbar_wait(full(i % kStages), (i / kStages) & 1, err, kSiteDrain);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_nvf4(kBM, kBN);
      bool issued_any = false;
      int it = 0;
      for (int ti = 0; ti < my_tiles && !*abort_flag; ++ti) {
        const int buf = ti & 1;
        if (ti >= 2 && !tc::mbar_wait(acc_empty(buf), ((ti / 2) - 1) & 1, err, kSiteAccEmpty)) {
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
        const uint32_t d = tmem + buf * kAccCols;
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % kStages;
          // codes landed and scale factors copied into TMEM slot s by the copier warp
          if (!tc::mbar_wait(sf_ready(s), (it / kStages) & 1, err, kSiteFull)) { *abort_flag = 1; break; }
          tc::tc_fence_after();
          const uint32_t sf_t = tmem_sf + s * kSfColsPerStage;
          const uint32_t a_base = sbase + kSmemCodes + s * kCodeBytes;
          const uint32_t b_base = a_base + kBM * kBKB;
          const int kk_valid = min(kMmaPerStage, (KB - kb * kBKB) / 32);
#pragma unroll
          for (int kk = 0; kk < kMmaPerStage; ++kk) {
            if (kk < kk_valid) {
              tc::mma_nvf4(d, tc::sw128_kmajor_desc(a_base + 32 * kk), tc::sw128_kmajor_desc(b_base + 32 * kk),
                           idesc, sf_t + 4 * kk, sf_t + 4 * (kMmaPerStage + kk), (kb > 0 || kk > 0) ? 1u : 0u);
            }
          }
          issued_any = true;
          tc::mma_commit(empty(s));
        }
        if (*abort_flag) break;
        tc::mma_commit(acc_full(buf));
      }
      if (*abort_flag && issued_any) {
        tc::mma_commit(mma_done);
        tc::mbar_wait(mma_done, 0, err, kSiteDrain);
      }
    }
  } else if (warp == 6) {
    // ---------------- scale-factor copier ----------------
    // Copies each stage's scale factors from shared memory into the stage's
    // TMEM slot as soon as the stage has landed, ahead of the MMA issuer.
    if (lane == 0) {
      int it = 0;
      for (int ti = 0; ti < my_tiles && !*abort_flag; ++ti) {
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % kStages;
          if (!tc::mbar_wait(full(s), (it / kStages) & 1, err, kSiteFull)) { *abort_flag = 1; break; }
          tc::tc_fence_after();
          const uint32_t sf_smem = sbase + kSmemSf + s * kSfBytes;
          const uint32_t sf_t = tmem_sf + s * kSfColsPerStage;
#pragma unroll
          for (int i = 0; i < 2 * kMmaPerStage; ++i)
            tc::tmem_cp_32x128b_x4(sf_t + 4 * i, tc::plain_desc(sf_smem + 512 * i));
          tc::mma_commit(sf_ready(s));
        }
      }
      if (*abort_flag && it > 0) {
        // copies still in flight must land before TMEM is freed
        tc::mma_commit(cp_done);
        tc::mbar_wait(cp_done, 0, err, kSiteDrain);
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;  // warps 2-5: TMEM lane quadrants 2, 3, 0, 1
    const float alpha = __ldg(g_a) * __ldg(g_b);
    for (int ti = 0; ti < my_tiles; ++ti) {
      const int buf = ti & 1;
      bool ok = tc::mbar_wait(acc_full(buf), (ti / 2) & 1, err, kSiteAccFull);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) { *abort_flag = 1; break; }
      tc::tc_fence_after();
      int mt, nt;
      tile_coords(blockIdx.x + ti * gridDim.x, mt_count, nt_count, mt, nt);
      const int row = mt * kBM + q * 32 + lane;
      const int n0 = nt * kBN;
#pragma unroll
      for (int cg = 0; cg < kBN / 32; ++cg) {
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * kAccCols + cg * 32, v);
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
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(acc_empty(buf));
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
                                   /*swizzle_bytes=*/128);
  if (st != cudaSuccess) return st;
  st = make_tmap_2d_u8(&tmB, b, static_cast<uint64_t>(K / 2), static_cast<uint64_t>(N), kBKB, kBN, 128);
  if (st != cudaSuccess) return st;
  st = cudaFuncSetAttribute(nvfp4_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTotal);
  if (st != cudaSuccess) return st;
  const int64_t tiles = ((T + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
  const int grid = static_cast<int>(tiles < sm_count() ? tiles : sm_count());
  nvfp4_gemm_kernel<<<grid, kThreads, kSmemTotal, stream>>>(tmA, tmB, sfa, sfb, static_cast<int>(T),
                                                            static_cast<int>(N), static_cast<int>(K), g_a, g_b, out,
                                                            static_cast<int>(out_dtype), device_error_word());
  return cudaGetLastError();
}

}  // namespace qlin
