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
// Persistent kernel: one CTA per SM walks the 128 x 256 output tiles
// (tile = blockIdx.x, + gridDim.x, ...), 14 warps:
//   warp 0      TMA producer: packed codes of A (128 rows) and B (256 rows),
//               128 bytes (256 elements) per row per stage, into the 128-byte
//               swizzled K-major layout the MMA descriptors describe, plus bulk
//               copies of the stage's E4M3 scales, which are stored in the MMA
//               layout (128-row x 4-block blocks of 512 bytes, byte
//               16*(r%32) + 4*(r/32) + j for row r, K block j); B's 256 rows
//               are two such blocks.
//   warps 10-13 scale-factor writers, one per TMEM lane quadrant: lane l of
//               a block holds, in 16 bytes, the scales of rows l, l+32, l+64,
//               l+96, which is what every quadrant of the scale TMEM slot holds
//               at lane l (4 columns per 128 rows).  Each warp reads its 16-byte
//               pieces of the landed stage with ld.shared and writes the
//               stage's 48 columns (A: 4 per MMA, B: 8 per MMA, rows 128-255
//               in the upper 4) into its own quadrant with tcgen05.st.  Written
//               from registers, the scales stay off the tensor pipe, where
//               tcgen05.cp copies of the same bytes queue behind the MMAs and
//               take longer than the MMAs themselves.
//   warp 1      TMEM allocation and the MMA issuer: per stage, once the four
//               writers have arrived, 4 x tcgen05.mma
//               kind::mxf4nvf4.block_scale.scale_vec::4X (M=128, N=256, K=64)
//               into the 256-column accumulator.  The wide N reads each A tile
//               once for 256 output columns, which keeps the shared-memory
//               bytes per multiply-add (TMA writes plus MMA reads) a quarter
//               below those of a 128 x 128 tile.
//   warps 2-9   epilogue: warp w reads TMEM lane quadrant w%4, columns
//               128*((w-2)/4) .. +127, of the finished accumulator, packs them
//               to bf16 / fp16 pairs in registers (times g_a . g_b, one
//               rounding) and releases the accumulator before it stores, so
//               the next tile's MMAs start meanwhile.
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
constexpr int kBKB = 128;                 // bytes of packed codes per row per stage (256 elements)
constexpr int kMmaPerStage = 4;           // K = 64 elements each
constexpr int kStages = 4;
constexpr int kEpiWarps = 8;
constexpr int kSfWarp0 = 2 + kEpiWarps;   // first of the 4 scale-factor writer warps
constexpr int kThreads = 32 * (kSfWarp0 + 4);
constexpr int kAccCols = kBN;
constexpr int kSfaCols = 4;               // TMEM columns of one MMA's A scales (128 rows)
constexpr int kSfbCols = 4 * kBN / 128;   // TMEM columns of one MMA's B scales (256 rows)
constexpr int kSfColsPerStage = kMmaPerStage * (kSfaCols + kSfbCols);
constexpr int kTmemCols = 512;            // accumulator (256) + scale factors (4 stages x 48)

constexpr int kSfBlock = 512;                               // one 128-row x 4-block scale block
constexpr int kCodeBytes = (kBM + kBN) * kBKB;              // 48 KB per stage
constexpr int kSfBytes = kMmaPerStage * (1 + kBN / 128) * kSfBlock;  // 6 KB per stage
constexpr int kSmemCodes = 0;
constexpr int kSmemSf = kSmemCodes + kStages * kCodeBytes;          // 192 KB
constexpr int kSmemBar = kSmemSf + kStages * kSfBytes;              // +24 KB
constexpr int kNumBars = 4 * kStages + 3;
constexpr int kSmemMisc = kSmemBar + kNumBars * 8;
constexpr int kSmemTotal = kSmemMisc + 16 + 1024;
static_assert(kSmemTotal <= 227 * 1024, "shared memory budget");
static_assert(kAccCols + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
static_assert(kBN % 128 == 0 && kBN <= 256, "B tile is whole 128-row scale blocks");

enum { kSiteEmpty = 1, kSiteFull, kSiteAccFull, kSiteAccEmpty, kSiteDrain };

// The block-scaled formats of this kernel.  A stage always holds 128 code
// bytes per row (4 MMAs of 32 bytes along K), and a 512-byte scale block holds
// 4 scales per row for 128 rows; one scale block covers 1 MMA (NVFP4, 4
// scales of 16 elements per K = 64), 2 MMAs (MXFP4, 2 scales of 32 per
// K = 64) or 4 MMAs (MXFP8, 1 scale of 32 per K = 32).  The MMA's scale-data
// ID (instruction descriptor bits 4-5 for B, 29-30 for A) selects the bytes
// of the 32-bit TMEM word that belong to it.
enum { kFmtNvf4 = 0, kFmtMxf4 = 1, kFmtMxf8 = 2 };

template <int F>
struct BsFormat {
  static constexpr int kElemsPerByte = F == kFmtMxf8 ? 1 : 2;
  static constexpr int kScaleK = F == kFmtNvf4 ? 16 : 32;             // elements per scale
  static constexpr int kMmaPerSfBlock = F == kFmtNvf4 ? 1 : (F == kFmtMxf4 ? 2 : 4);
  static constexpr int kSfBlocksPerStage = kMmaPerStage / kMmaPerSfBlock;
};

// Instruction descriptor: E2M1 x E2M1 with E4M3 scales (NVFP4), E2M1 x E2M1
// with E8M0 scales (MXFP4), E4M3 x E4M3 with E8M0 scales (MXFP8), fp32
// accumulator, K-major A and B, M = 128, N = n.
template <int F>
__host__ __device__ constexpr uint32_t idesc_bs(int m, int n, uint32_t sf_id) {
  const uint32_t elems = F == kFmtMxf8 ? 0u : (1u << 7) | (1u << 10);
  const uint32_t e8m0 = F == kFmtNvf4 ? 0u : (1u << 23);
  return elems | e8m0 | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24) |
         (sf_id << 4) | (sf_id << 29);
}

template <int F>
__device__ __forceinline__ void mma_bs(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  if constexpr (F == kFmtNvf4) {
    tc::mma_nvf4(d_tmem, a_desc, b_desc, idesc, sfa_tmem, sfb_tmem, accumulate);
  } else if constexpr (F == kFmtMxf4) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p; }" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
  } else {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p; }" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
  }
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

template <int F>
__global__ void __launch_bounds__(kThreads, 1) block_scaled_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
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
  using Fmt = BsFormat<F>;
  const int KB = K / Fmt::kElemsPerByte;      // code bytes per row
  const int KG = (K / Fmt::kScaleK + 3) / 4;  // 4-scale groups per row (512-byte scale blocks per 128 rows)
  const int num_kb = (KB + kBKB - 1) / kBKB;  // stages per tile
  const int mt_count = (T + kBM - 1) / kBM, nt_count = (N + kBN - 1) / kBN;
  const int num_tiles = mt_count * nt_count;
  const int my_tiles = blockIdx.x < num_tiles ? (num_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;

  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t bar0 = sbase + kSmemBar;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto sf_ready = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
  auto sf_full = [&](int s) { return bar0 + 8u * (3 * kStages + s); };
  const uint32_t acc_full = bar0 + 8u * (4 * kStages);
  const uint32_t acc_empty = bar0 + 8u * (4 * kStages + 1);
  const uint32_t mma_done = bar0 + 8u * (4 * kStages + 2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemMisc + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(full(s), 1);        // TMA producer: codes
      tc::mbar_init(sf_full(s), 1);     // TMA producer: scale factors
      tc::mbar_init(empty(s), 1);       // MMA commit
      tc::mbar_init(sf_ready(s), 4);    // the four scale-factor writer warps
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
  const uint32_t tmem_sf = tmem + kAccCols;
  const int n128_count = (N + 127) / 128;  // 128-row scale blocks of B

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
        const int nb0 = nt * (kBN / 128);                     // first 128-row scale block of the B tile
        const int nbs = min(kBN / 128, n128_count - nb0);     // scale blocks of the B tile that exist
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % kStages;
          if (it >= kStages && !tc::mbar_wait(empty(s), ((it / kStages) - 1) & 1, err, kSiteEmpty)) {
            *abort_flag = 1;
            break;
          }
          const uint32_t dst = sbase + kSmemCodes + s * kCodeBytes;
          const uint32_t sf_dst = sbase + kSmemSf + s * kSfBytes;
          const int kg0 = kb * Fmt::kSfBlocksPerStage;        // first scale group of the stage
          const int nkg = min(Fmt::kSfBlocksPerStage, KG - kg0);  // groups of this stage that exist
          // scales first, on their own barrier: the writer warps put them into
          // TMEM while the codes are still in flight
          tc::mbar_arrive_expect_tx(sf_full(s), (1 + nbs) * nkg * kSfBlock);
          tc::bulk_load(sf_dst, sfa + ((int64_t)mt * KG + kg0) * kSfBlock, nkg * kSfBlock, sf_full(s));
          for (int h = 0; h < nbs; ++h)
            tc::bulk_load(sf_dst + (1 + h) * kMmaPerStage * kSfBlock,
                          sfb + ((int64_t)(nb0 + h) * KG + kg0) * kSfBlock, nkg * kSfBlock, sf_full(s));
          tc::mbar_arrive_expect_tx(full(s), kCodeBytes);
          tc::tma_load_2d(dst, &tmA, kb * kBKB, mt * kBM, full(s));
          tc::tma_load_2d(dst + kBM * kBKB, &tmB, kb * kBKB, nt * kBN, full(s));
          issued = it + 1;
        }
      }
      if (*abort_flag) {
        for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i) {
          tc::mbar_wait(sf_full(i % kStages), (i / kStages) & 1, err, kSiteDrain);
          tc::mbar_wait(full(i % kStages), (i / kStages) & 1, err, kSiteDrain);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
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
          // scales written into TMEM slot s by the writer warps, codes landed
          if (!tc::mbar_wait(sf_ready(s), (it / kStages) & 1, err, kSiteFull) ||
              !tc::mbar_wait(full(s), (it / kStages) & 1, err, kSiteFull)) {
            *abort_flag = 1;
            break;
          }
          tc::tc_fence_after();
          const uint32_t sf_t = tmem_sf + s * kSfColsPerStage;
          const uint32_t a_base = sbase + kSmemCodes + s * kCodeBytes;
          const uint32_t b_base = a_base + kBM * kBKB;
          const int kk_valid = min(kMmaPerStage, (KB - kb * kBKB) / 32);
#pragma unroll
          for (int kk = 0; kk < kMmaPerStage; ++kk) {
            if (kk < kk_valid) {
              constexpr int mpb = Fmt::kMmaPerSfBlock;
              const int blk = kk / mpb;                       // the stage's scale block of this MMA
              const uint32_t sf_id = static_cast<uint32_t>((kk % mpb) * (4 / mpb));
              mma_bs<F>(tmem, tc::sw128_kmajor_desc(a_base + 32 * kk), tc::sw128_kmajor_desc(b_base + 32 * kk),
                        idesc_bs<F>(kBM, kBN, sf_id), sf_t + kSfaCols * blk,
                        sf_t + kMmaPerStage * kSfaCols + kSfbCols * blk, (kb > 0 || kk > 0) ? 1u : 0u);
            }
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
  } else if (warp >= kSfWarp0) {
    // ---------------- scale-factor writers ----------------
    // Slot layout: A scale block j in columns 4j..4j+3, then B scale block j
    // in columns 16+8j..16+8j+7 (rows 0-127, then rows 128-255).  The MX
    // formats use the first 2 (MXFP4) or 1 (MXFP8) blocks; the rest are zero.
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int it = 0;
    for (int ti = 0; ti < my_tiles && !*abort_flag; ++ti) {
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const int s = it % kStages;
        ok = tc::mbar_wait(sf_full(s), (it / kStages) & 1, err, kSiteFull);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) { *abort_flag = 1; break; }
        tc::tc_fence_after();
        const uint32_t src = sbase + kSmemSf + s * kSfBytes + 16 * lane;
        uint32_t v[kSfColsPerStage];
#pragma unroll
        for (int kk = 0; kk < kMmaPerStage; ++kk) {
          if (kk >= BsFormat<F>::kSfBlocksPerStage) {
#pragma unroll
            for (int c = 0; c < 4; ++c) v[4 * kk + c] = 0u;
#pragma unroll
            for (int c = 0; c < 4 * (kBN / 128); ++c) v[kMmaPerStage * kSfaCols + kSfbCols * kk + c] = 0u;
            continue;
          }
          const uint4 w = tc::lds128(src + kSfBlock * kk);
          v[4 * kk] = w.x; v[4 * kk + 1] = w.y; v[4 * kk + 2] = w.z; v[4 * kk + 3] = w.w;
#pragma unroll
          for (int h = 0; h < kBN / 128; ++h) {
            const uint4 u = tc::lds128(src + ((1 + h) * kMmaPerStage + kk) * kSfBlock);
            const int c = kMmaPerStage * kSfaCols + kSfbCols * kk + 4 * h;
            v[c] = u.x; v[c + 1] = u.y; v[c + 2] = u.z; v[c + 3] = u.w;
          }
        }
        const uint32_t dst = tmem + lane_base + kAccCols + s * kSfColsPerStage;
        tc::tmem_st_32x32b_x32(dst, v);
        tc::tmem_st_32x32b_x16(dst + 32, v + 32);
        tc::tmem_wait_st();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(sf_ready(s));
      }
      if (!ok) break;
    }
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;                      // TMEM lane quadrant this warp may access
    const int half = (warp - 2) / 4;             // column half of the 256-column tile
    pdl_wait();  // the global scales may come from the previous kernel
    const float alpha = g_a != nullptr ? __ldg(g_a) * __ldg(g_b) : 1.0f;  // MX formats: no per-tensor scales
    for (int ti = 0; ti < my_tiles; ++ti) {
      bool ok = tc::mbar_wait(acc_full, ti & 1, err, kSiteAccFull);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) { *abort_flag = 1; break; }
      tc::tc_fence_after();
      int mt, nt;
      tile_coords(blockIdx.x + ti * gridDim.x, mt_count, nt_count, mt, nt);
      const int c0 = nt * kBN + half * 128;      // first output column of this warp
      uint32_t pk[64];                           // 128 outputs, two per word
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + half * 128;
#pragma unroll
      for (int cg = 0; cg < 4; ++cg) {
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(taddr + cg * 32, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float f0 = __uint_as_float(v[2 * i]) * alpha;
          const float f1 = __uint_as_float(v[2 * i + 1]) * alpha;
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

template <int F>
cudaError_t launch_block_scaled_gemm(const uint8_t* a, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb,
                                     int64_t T, int64_t N, int64_t K, const float* g_a, const float* g_b, void* out,
                                     qlin_dtype out_dtype, cudaStream_t stream) {
  if (T == 0 || N == 0) return cudaSuccess;
  const uint64_t row_bytes = static_cast<uint64_t>(K / BsFormat<F>::kElemsPerByte);
  CUtensorMap tmA, tmB;
  cudaError_t st = make_tmap_2d_u8(&tmA, a, row_bytes, static_cast<uint64_t>(T), kBKB, kBM, /*swizzle_bytes=*/128);
  if (st != cudaSuccess) return st;
  st = make_tmap_2d_u8(&tmB, b, row_bytes, static_cast<uint64_t>(N), kBKB, kBN, 128);
  if (st != cudaSuccess) return st;
  st = ensure_max_dynamic_smem(reinterpret_cast<const void*>(block_scaled_gemm_kernel<F>));
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
  return cudaLaunchKernelEx(&cfg, block_scaled_gemm_kernel<F>, tmA, tmB, sfa, sfb, static_cast<int>(T),
                            static_cast<int>(N), static_cast<int>(K), g_a, g_b, out, static_cast<int>(out_dtype),
                            device_error_word());
}

}  // namespace

cudaError_t launch_nvfp4_gemm(const uint8_t* a, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb,
                              int64_t T, int64_t N, int64_t K, const float* g_a, const float* g_b, void* out,
                              qlin_dtype out_dtype, cudaStream_t stream) {
  return launch_block_scaled_gemm<kFmtNvf4>(a, sfa, b, sfb, T, N, K, g_a, g_b, out, out_dtype, stream);
}

cudaError_t launch_mx_gemm(const uint8_t* a, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb, int64_t T,
                           int64_t N, int64_t K, qlin_mx_fmt fmt, void* out, qlin_dtype out_dtype,
                           cudaStream_t stream) {
  if (fmt == QLIN_MX_FP8_E4M3)
    return launch_block_scaled_gemm<kFmtMxf8>(a, sfa, b, sfb, T, N, K, nullptr, nullptr, out, out_dtype, stream);
  return launch_block_scaled_gemm<kFmtMxf4>(a, sfa, b, sfb, T, N, K, nullptr, nullptr, out, out_dtype, stream);
}

}  // namespace qlin
