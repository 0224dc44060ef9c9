// FP8 W8A8: E4M3 x E4M3 GEMM on the tcgen05 tensor cores (kind::f8f6f4)
//
//   out[t,n] = s_a[t] . s_b[n] . sum_k dec(a[t,k]) . dec(b[n,k]) + bias[n]
//
// ("LLM and AIGC quantization: from number formats to W4A4", "W4A4, FP8 and
// block-scaled formats": x / s is converted to E4M3, the FP8 tensor core
// multiplies with FP32 accumulation, and the epilogue multiplies by the two
// scales; activations per token, weights per channel.)
//
// Persistent kernel: one CTA per SM walks the 128 x 256 output tiles
// (tile = blockIdx.x, + gridDim.x, ...), 10 warps:
//   warp 0      TMA producer: E4M3 codes of A (128 rows) and B (256 rows),
//               128 bytes (128 elements) per row per stage, into the 128-byte
//               swizzled K-major layout the MMA descriptors describe, in a
//               4-stage ring.
//   warp 1      TMEM allocation and the MMA issuer: per stage 4 x tcgen05.mma
//               kind::f8f6f4 (M=128, N=256, K=32, E4M3 operands, fp32
//               accumulator) into the 256-column accumulator.
//   warps 2-9   epilogue: warp w reads TMEM lane quadrant w%4, columns
//               128*((w-2)/4) .. +127, of the finished accumulator, applies
//               s_a[row] . (acc . s_b[col]) + bias[col] in float32, packs to
//               bf16 / fp16 pairs, releases the accumulator before it stores
//               (so the next tile's MMAs start meanwhile), and stores 128-byte
//               row segments after an 8 x 8 shuffle transpose.
// The same skeleton as the block-scaled fp4 GEMM without the scale factors:
// one 8-bit element is one byte, so a 128-byte stage row holds 128 elements
// and each K = 32 MMA reads 32 bytes of every row, the step the descriptors
// take inside the swizzle atom.  The products of two E4M3 values are exact
// in fp32 and the tensor core accumulates in fp32.
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

constexpr int kBM = 128, kBN = 256;
constexpr int kBK = 128;                  // bytes (= E4M3 elements) per row per stage
constexpr int kMmaK = 32;                 // K of one kind::f8f6f4 MMA for 8-bit operands
constexpr int kMmaPerStage = kBK / kMmaK;
constexpr int kStages = 4;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kTmemCols = kBN;            // the fp32 accumulator

constexpr int kCodeBytes = (kBM + kBN) * kBK;              // 48 KB per stage
constexpr int kSmemCodes = 0;
constexpr int kParBytes = 2 * 128 * 4;                     // one epilogue warp's s_b and bias of 128 columns
constexpr int kSmemPar = kSmemCodes + kStages * kCodeBytes;
constexpr int kSmemBar = kSmemPar + kEpiWarps * kParBytes;
constexpr int kNumBars = 2 * kStages + 3;
constexpr int kSmemMisc = kSmemBar + kNumBars * 8;
constexpr int kSmemTotal = kSmemMisc + 16 + 1024;
static_assert(kSmemTotal <= 227 * 1024, "shared memory budget");

enum { kSiteEmpty = 1, kSiteFull, kSiteAccFull, kSiteAccEmpty, kSiteDrain };

// Instruction descriptor, kind::f8f6f4: fp32 accumulator (bits 4-5 = 1), A and
// B formats in bits 7-9 and 10-12 (E4M3 = 0), both K-major, N / 8 in bits
// 17-22, M / 16 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f8_e4m3(int m, int n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

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

__device__ __forceinline__ float bias_at(const void* bias, int dtype, int i) {
  if (dtype == QLIN_F16) return __half2float(static_cast<const __half*>(bias)[i]);
  if (dtype == QLIN_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(bias)[i]);
  return static_cast<const float*>(bias)[i];
}

__global__ void __launch_bounds__(kThreads, 1) fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                                                              const __grid_constant__ CUtensorMap tmB, int T, int N,
                                                              int K, const float* __restrict__ scale_a,
                                                              const float* __restrict__ scale_b,
                                                              const void* __restrict__ bias, int bias_dtype,
                                                              void* __restrict__ out, int out_dtype,
                                                              int32_t* __restrict__ err) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_kb = (K + kBK - 1) / kBK;     // stages per tile
  const int mt_count = (T + kBM - 1) / kBM, nt_count = (N + kBN - 1) / kBN;
  const int num_tiles = mt_count * nt_count;
  const int my_tiles = blockIdx.x < num_tiles ? (num_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;

  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t bar0 = sbase + kSmemBar;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  const uint32_t acc_full = bar0 + 8u * (2 * kStages);
  const uint32_t acc_empty = bar0 + 8u * (2 * kStages + 1);
  const uint32_t mma_done = bar0 + 8u * (2 * kStages + 2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemMisc + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(full(s), 1);    // TMA producer
      tc::mbar_init(empty(s), 1);   // MMA commit
    }
    tc::mbar_init(acc_full, 1);
    tc::mbar_init(acc_empty, kEpiWarps);
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

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tc::prefetch_tmap(&tmA);
      tc::prefetch_tmap(&tmB);
      // the operands may come from the previous kernel in the stream
      // (programmatic dependent launch: this grid may start before it ends)
      pdl_wait();
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
          // K bytes past the end of the rows arrive as zeros (code 0 = +0)
          tc::mbar_arrive_expect_tx(full(s), kCodeBytes);
          tc::tma_load_2d(dst, &tmA, kb * kBK, mt * kBM, full(s));
          tc::tma_load_2d(dst + kBM * kBK, &tmB, kb * kBK, nt * kBN, full(s));
          issued = it + 1;
        }
      }
      // the last copies must have landed before the CTA exits
      for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
        tc::mbar_wait(full(i % kStages), (i / kStages) & 1, err, kSiteDrain);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_f8_e4m3(kBM, kBN);
      bool issued_any = false;
      int it = 0;
      for (int ti = 0; ti < my_tiles && !*abort_flag; ++ti) {
        // the epilogue has taken the previous tile's accumulator into registers
        if (ti >= 1 && !tc::mbar_wait(acc_empty, (ti - 1) & 1, err, kSiteAccEmpty)) {
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % kStages;
          if (!tc::mbar_wait(full(s), (it / kStages) & 1, err, kSiteFull)) {
            *abort_flag = 1;
            break;
          }
          tc::tc_fence_after();
          const uint32_t a_base = sbase + kSmemCodes + s * kCodeBytes;
          const uint32_t b_base = a_base + kBM * kBK;
          // MMAs that cover at least one real K element of the stage
          const int kk_valid = min(kMmaPerStage, (K - kb * kBK + kMmaK - 1) / kMmaK);
#pragma unroll
          for (int kk = 0; kk < kMmaPerStage; ++kk) {
            if (kk < kk_valid)
              mma_f8(tmem, tc::sw128_kmajor_desc(a_base + kMmaK * kk), tc::sw128_kmajor_desc(b_base + kMmaK * kk),
                     idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          issued_any = true;
          tc::mma_commit(empty(s));
        }
        if (*abort_flag) break;
        tc::mma_commit(acc_full);
      }
      if (*abort_flag && issued_any) {
        // MMAs still in flight must finish before TMEM is freed
        tc::mma_commit(mma_done);
        tc::mbar_wait(mma_done, 0, err, kSiteDrain);
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;                      // TMEM lane quadrant this warp may access
    const int half = (warp - 2) / 4;             // column half of the 256-column tile
    float* par_sb = reinterpret_cast<float*>(smem + kSmemPar + (warp - 2) * kParBytes);
    float* par_bias = par_sb + 128;
    pdl_wait();  // the scales and the bias may come from the previous kernel
    for (int ti = 0; ti < my_tiles; ++ti) {
      int mt, nt;
      tile_coords(blockIdx.x + ti * gridDim.x, mt_count, nt_count, mt, nt);
      const int c0 = nt * kBN + half * 128;      // first output column of this warp
      // this warp's column parameters (a private copy: no other warp's
      // progress matters), loaded before the accumulator is ready
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int col = lane + 32 * j, n = c0 + col;
        par_sb[col] = n < N ? scale_b[n] : 0.0f;
        par_bias[col] = (n < N && bias != nullptr) ? bias_at(bias, bias_dtype, n) : 0.0f;
      }
      const int row = mt * kBM + q * 32 + lane;
      const float sa = row < T ? scale_a[row] : 0.0f;
      __syncwarp();
      bool ok = tc::mbar_wait(acc_full, ti & 1, err, kSiteAccFull);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) { *abort_flag = 1; break; }
      tc::tc_fence_after();
      uint32_t pk[64];                           // 128 outputs of this lane's row, two per word
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + half * 128;
#pragma unroll
      for (int cg = 0; cg < 4; ++cg) {
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(taddr + cg * 32, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int col = cg * 32 + 2 * i;
          const float f0 = fmaf(sa, __uint_as_float(v[2 * i]) * par_sb[col], par_bias[col]);
          const float f1 = fmaf(sa, __uint_as_float(v[2 * i + 1]) * par_sb[col + 1], par_bias[col + 1]);
          if (out_dtype == QLIN_BF16) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f0, f1);
            pk[16 * cg + i] = *reinterpret_cast<uint32_t*>(&h);
          } else {
            __half2 h = __floats2half2_rn(f0, f1);
            pk[16 * cg + i] = *reinterpret_cast<uint32_t*>(&h);
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(acc_empty);  // accumulator free for the next tile
      // 8 x 8 transpose of 16-byte chunks inside each group of 8 lanes
      // (three xor-butterfly steps): afterwards lane 8g+j holds, in slot e of
      // column block b, chunk 8b+j of row 8g+e, so each store below writes 128
      // contiguous bytes of four rows instead of 16 bytes of 32 rows.
#pragma unroll
      for (int st = 0; st < 3; ++st) {
        const bool up = (lane >> st) & 1;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
#pragma unroll
          for (int e0 = 0; e0 < 8; ++e0) {
            if (e0 & (1 << st)) continue;
            const int e1 = e0 | (1 << st);
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              uint32_t& x0 = pk[4 * (8 * b + e0) + w];
              uint32_t& x1 = pk[4 * (8 * b + e1) + w];
              const uint32_t got = __shfl_xor_sync(0xffffffffu, up ? x0 : x1, 1 << st);
              if (up) x0 = got; else x1 = got;
            }
          }
        }
      }
      const int j = lane & 7;
      const int row0 = mt * kBM + q * 32 + 8 * (lane >> 3);
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const int col = c0 + 8 * (8 * b + j);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int r = row0 + e;
          if (r < T && col < N)
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + (int64_t)r * N + col) =
                make_uint4(pk[4 * (8 * b + e)], pk[4 * (8 * b + e) + 1], pk[4 * (8 * b + e) + 2],
                           pk[4 * (8 * b + e) + 3]);
        }
      }
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

cudaError_t launch_fp8_gemm(const uint8_t* a, const uint8_t* b, int64_t T, int64_t N, int64_t K, const float* scale_a,
                            const float* scale_b, const void* bias, qlin_dtype bias_dtype, void* out,
                            qlin_dtype out_dtype, cudaStream_t stream) {
  if (T == 0 || N == 0) return cudaSuccess;
  CUtensorMap tmA, tmB;
  cudaError_t st = make_tmap_2d_u8(&tmA, a, static_cast<uint64_t>(K), static_cast<uint64_t>(T), kBK, kBM,
                                   /*swizzle_bytes=*/128);
  if (st != cudaSuccess) return st;
  st = make_tmap_2d_u8(&tmB, b, static_cast<uint64_t>(K), static_cast<uint64_t>(N), kBK, kBN, 128);
  if (st != cudaSuccess) return st;
  st = ensure_max_dynamic_smem(reinterpret_cast<const void*>(fp8_gemm_kernel));
  if (st != cudaSuccess) return st;
  const int64_t tiles = ((T + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
  const int grid = static_cast<int>(tiles < sm_count() ? tiles : sm_count());
  // programmatic dependent launch: the prologue (barriers, TMEM, tensor maps)
  // overlaps the end of the previous kernel (the activation quantizer)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemTotal;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fp8_gemm_kernel, tmA, tmB, static_cast<int>(T), static_cast<int>(N),
                            static_cast<int>(K), scale_a, scale_b, bias, static_cast<int>(bias_dtype), out,
                            static_cast<int>(out_dtype), device_error_word());
}

}  // namespace qlin
