// W8A8 with both operands given as exact fp16 codes: the int8 GEMM with the
// exact int32 accumulator and the fused epilogue, nothing widened on chip
//
//   D^  = A^ . B^^T                                   (int32, exact)
//   out = s_a[t] . s_b[n] . (D^ - azp[t] . azp_adj[n]) + bias[n]
//
// ("LLM and AIGC quantization: from number formats to W4A4", W8A8 section:
// INT8 products, INT32 accumulation, the two scales applied as an outer
// product in the epilogue; "vLLM W8A8 quantized GEMM: CUTLASS epilogue
// design", sections 2.1-2.4 for the four epilogues and section 3 for the
// evaluation order scale_a . (scale_b . acc) + bias.)
//
// Every code, of the activations and of the weights, is an integer of
// magnitude <= 128 and is stored as the fp16 number of the same value: the
// activation quantizer writes its codes in that form and the weights are
// converted once at load time.  The 16-bit tensor cores then read both tiles
// where TMA puts them.  Exactness is that of the int8-operand kernel: every
// product is exact in fp32, K runs in chunks of 1024 so that every partial sum
// of a chunk stays within 1024 . 128 . 128 = 2^24, and each chunk's fp32
// result is converted to int32 and added in int32, which gives D^ bit for bit.
//
// Persistent kernel: one CTA per SM walks 128 x BN output tiles (groups of 8
// row tiles share column tiles for L2 reuse), BN = 256, or 224 where that
// gives fewer rounds of tiles on the SMs (2048 x 4096: 304 tiles of 224
// columns are two full rounds on 152 SMs, where 256 tiles of 256 columns took
// two rounds with the second a third empty), 10 warps:
//   warp 0     TMA producer: 64 K elements (128 bytes of fp16) of the tile's
//              128 A rows and BN B rows per stage, in the 128-byte swizzled
//              K-major layout the MMA descriptors describe, 4-stage ring of
//              48 (44) KB stages.
//   warp 1     TMEM allocation and the MMA issuer: per stage 4 x tcgen05.mma
//              kind::f16 (M=128, N=BN, K=16, both operands in shared memory)
//              into one of two BN-column chunk accumulators, which alternate
//              chunk by chunk (and across tiles).
//   warps 2-9  epilogue: lane l of the warp with TMEM lane quadrant q owns row
//              32q + l and columns h BN / 2 .. (h + 1) BN / 2 - 1 of the tile,
//              h = (warp - 2) / 4.  It reads each finished chunk, adds it in
//              int32 to BN / 2 running totals held in registers and releases the
//              accumulator at once, so the MMAs of the chunk after next never
//              wait for more than one read.  After the tile's last chunk it
//              applies the epilogue from the registers and stores 128-byte
//              row segments, while the next tile's MMAs run.
// Every barrier wait is bounded; on expiry the kernel records the site in the
// device error word, stops issuing work, waits (bounded) for copies and MMAs
// already in flight, frees TMEM and exits.
#include <cuda.h>

#include <mutex>

#include "device_common.cuh"
#include "qlin_internal.h"
#include "tc_common.cuh"
#include "tmap.h"

namespace qlin {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;                        // K elements per stage: 128 bytes of fp16 per row
constexpr int kRowBytes = 2 * kBK;
constexpr int kMmaPerStage = kBK / 16;
constexpr int kStages = 4;
constexpr int kChunkK = 1024;                  // exact fp32 accumulation span
constexpr int kKbPerChunk = kChunkK / kBK;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kTmemCols = 512;                 // two chunk accumulators of BN columns

// The plan of a tile width BN.
template <int BN>
struct F16Cfg {
  static constexpr int kCols = BN / 2;                       // columns of the tile one epilogue warp owns
  static constexpr int kStageBytes = (kBM + BN) * kRowBytes;  // 48 or 44 KB
  static constexpr int kSmemPar = kStages * kStageBytes;
  static constexpr int kParBytes = 3 * kCols * 4;            // one epilogue warp's s_b, azp_adj and bias
  static constexpr int kSmemBar = kSmemPar + kEpiWarps * kParBytes;
  static constexpr int kNumBars = 2 * kStages + 2 + 2 + 1;
  static constexpr int kSmemMisc = kSmemBar + kNumBars * 8;
  static constexpr int kSmemTotal = kSmemMisc + 16 + 1024;   // + alignment slack
  static_assert(BN == 256 || BN == 224, "tile widths");
  static_assert(2 * BN <= kTmemCols, "TMEM budget");
  static_assert(kSmemTotal <= 227 * 1024, "shared memory budget");
  static_assert(kStageBytes % 1024 == 0 && (kBM * kRowBytes) % 1024 == 0,
                "stages and the B tile keep the 1024-byte alignment of the swizzled atoms");
  static_assert(kCols % 16 == 0, "the epilogue reads TMEM 16 columns at a time");
};

enum { kSiteEmpty = 1, kSiteFull, kSiteAccEmpty, kSiteAccFull, kSiteDrain };

struct EpiArgs {
  const float* scale_a;
  const float* scale_b;
  const int32_t* azp;
  const int32_t* azp_adj;
  const void* bias;
  int scale_a_per_row, scale_b_per_col, bias_dtype, out_dtype;
};

__device__ __forceinline__ float load_as_float(const void* p, int dtype, int i) {
  if (dtype == QLIN_F16) return __half2float(static_cast<const __half*>(p)[i]);
  if (dtype == QLIN_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  return static_cast<const float*>(p)[i];
}

// Output tile `tile` in the persistent order: groups of 8 row tiles walk the
// column tiles together, so the B tiles of a column are reused from L2.
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

template <int BN>
__global__ void __launch_bounds__(kThreads, 1) w8a8_f16_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                                                                   const __grid_constant__ CUtensorMap tmB, int T,
                                                                   int N, int K, EpiArgs epi, void* __restrict__ out,
                                                                   int32_t* __restrict__ err) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  using Cfg = F16Cfg<BN>;
  constexpr int kCols = Cfg::kCols, kStageBytes = Cfg::kStageBytes, kSmemPar = Cfg::kSmemPar;
  constexpr int kParBytes = Cfg::kParBytes, kSmemBar = Cfg::kSmemBar, kSmemMisc = Cfg::kSmemMisc;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt_count = (T + kBM - 1) / kBM, nt_count = (N + BN - 1) / BN;
  const int tiles = mt_count * nt_count;
  const int my_tiles = blockIdx.x < tiles ? (tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int num_kb = (K + kBK - 1) / kBK;
  const int num_chunks = (num_kb + kKbPerChunk - 1) / kKbPerChunk;

  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t bar0 = sbase + kSmemBar;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto acc_full = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
  const uint32_t mma_done = bar0 + 8u * (2 * kStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemMisc + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(full(s), 1);   // TMA producer
      tc::mbar_init(empty(s), 1);  // MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(acc_full(b), 1);
      tc::mbar_init(acc_empty(b), kEpiWarps);
    }
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
      // the codes may come from the previous kernel in the stream
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
          const uint32_t dst = sbase + s * kStageBytes;
          // K elements past the end of the rows, and rows past T or N, arrive
          // as zeros (fp16 +0)
          tc::mbar_arrive_expect_tx(full(s), kStageBytes);
          tc::tma_load_2d(dst, &tmA, kb * kRowBytes, mt * kBM, full(s));
          tc::tma_load_2d(dst + kBM * kRowBytes, &tmB, kb * kRowBytes, nt * BN, full(s));
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
      const uint32_t idesc = tc::idesc_f16(kBM, BN, 0);  // fp16 x fp16 -> fp32
      bool issued_any = false;
      int it = 0, g = 0;  // stage and chunk counters across tiles
      for (int ti = 0; ti < my_tiles && !*abort_flag; ++ti) {
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int kin = kb % kKbPerChunk;
          const int buf = g & 1;
          // the epilogue has read the accumulator's previous chunk
          if (kin == 0 && g >= 2 && !tc::mbar_wait(acc_empty(buf), ((g >> 1) - 1) & 1, err, kSiteAccEmpty)) {
            *abort_flag = 1;
            break;
          }
          const int s = it % kStages;
          if (!tc::mbar_wait(full(s), (it / kStages) & 1, err, kSiteFull)) {
            *abort_flag = 1;
            break;
          }
          tc::tc_fence_after();
          const uint32_t a_base = sbase + s * kStageBytes;
          const uint32_t b_base = a_base + kBM * kRowBytes;
          const uint32_t d = tmem + buf * BN;
          // MMAs that cover at least one real K element of the stage
          const int kk_valid = min(kMmaPerStage, (K - kb * kBK + 15) / 16);
#pragma unroll
          for (int kk = 0; kk < kMmaPerStage; ++kk) {
            if (kk < kk_valid)
              tc::mma_f16(d, tc::sw128_kmajor_desc(a_base + 32 * kk), tc::sw128_kmajor_desc(b_base + 32 * kk), idesc,
                          (kin > 0 || kk > 0) ? 1u : 0u);
          }
          issued_any = true;
          tc::mma_commit(empty(s));
          if (kin == kKbPerChunk - 1 || kb == num_kb - 1) {
            tc::mma_commit(acc_full(buf));
            ++g;
          }
        }
      }
      if (*abort_flag && issued_any) {
        // MMAs still in flight must finish before TMEM is freed
        tc::mma_commit(mma_done);
        tc::mbar_wait(mma_done, 0, err, kSiteDrain);
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;             // TMEM lane quadrant this warp may access
    const int ew = warp - 2;
    const int col0 = (ew >> 2) * kCols;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    float* par_sb = reinterpret_cast<float*>(smem + kSmemPar + ew * kParBytes);
    int32_t* par_adj = reinterpret_cast<int32_t*>(par_sb + kCols);
    float* par_bias = par_sb + 2 * kCols;
    pdl_wait();  // the scales and zero-points may come from the previous kernel
    const bool raw = epi.out_dtype == QLIN_I32;
    const bool per_tensor_adj = epi.azp == nullptr && epi.azp_adj != nullptr;
    int g = 0;
    bool ok = true;
    for (int ti = 0; ti < my_tiles && ok; ++ti) {
      int mt, nt;
      tile_coords(blockIdx.x + ti * gridDim.x, mt_count, nt_count, mt, nt);
      const int c0 = nt * BN + col0;  // first output column of this warp
      // Column parameters of this tile, in a copy private to this warp (so no
      // other warp's progress matters), loaded while the MMAs run.
      __syncwarp();
      if (!raw) {
#pragma unroll
        for (int j = 0; j < (kCols + 31) / 32; ++j) {
          const int col = lane + 32 * j, n = c0 + col;
          if (col >= kCols) break;
          const bool inb = n < N;
          par_sb[col] = inb ? (epi.scale_b_per_col ? epi.scale_b[n] : epi.scale_b[0]) : 0.0f;
          par_adj[col] = (inb && epi.azp_adj != nullptr) ? epi.azp_adj[n] : 0;
          par_bias[col] = (inb && epi.bias != nullptr) ? load_as_float(epi.bias, epi.bias_dtype, n) : 0.0f;
        }
      }
      __syncwarp();
      const int row = mt * kBM + q * 32 + lane;
      float sa = 0.0f;
      int32_t za = 0;
      if (!raw && row < T) {
        sa = epi.scale_a_per_row ? epi.scale_a[row] : epi.scale_a[0];
        za = epi.azp != nullptr ? epi.azp[row] : 0;
      }

      int32_t tot[kCols];  // D^ of this lane's row, columns c0 .. c0 + 127
#pragma unroll
      for (int i = 0; i < kCols; ++i) tot[i] = 0;
      for (int c = 0; c < num_chunks; ++c, ++g) {
        const int buf = g & 1;
        ok = tc::mbar_wait(acc_full(buf), (g >> 1) & 1, err, kSiteAccFull);
        ok = __all_sync(0xffffffffu, ok);  // lanes agree and reconverge before tcgen05.ld
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
        const uint32_t ta = lane_base + buf * BN + col0;
#pragma unroll
        for (int cg = 0; cg < kCols / 16; ++cg) {
          uint32_t v[16];
          tc::tmem_ld_32x32b_x16(ta + cg * 16, v);
          tc::tmem_wait_ld();
          // every chunk sum is an integer below 2^24 in magnitude: exact in
          // fp32 and converted exactly
#pragma unroll
          for (int i = 0; i < 16; ++i) tot[cg * 16 + i] += __float2int_rn(__uint_as_float(v[i]));
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(acc_empty(buf));  // accumulator free for the chunk after next
      }
      if (!ok) break;

      if (raw) {
        // test hook: D^ itself, 16 bytes per store
        if (row < T) {
          int32_t* o = static_cast<int32_t*>(out) + (int64_t)row * N + c0;
#pragma unroll
          for (int c4 = 0; c4 < kCols / 4; ++c4)
            if (c0 + 4 * c4 < N)
              *reinterpret_cast<int4*>(o + 4 * c4) =
                  make_int4(tot[4 * c4], tot[4 * c4 + 1], tot[4 * c4 + 2], tot[4 * c4 + 3]);
        }
        continue;
      }

      // out = s_a . ((D^ - azp . azp_adj) . s_b) + bias: the correction in
      // int32, one conversion to float, then the scales and the bias in fp32.
      // Blocks of 64 columns (the last one partial when BN / 2 = 112), each
      // packed, transposed and stored in turn.
      const int j = lane & 7;
      const int row0 = mt * kBM + q * 32 + 8 * (lane >> 3);
#pragma unroll
      for (int b = 0; b < (kCols + 63) / 64; ++b) {
        uint32_t pk[32];  // this row's columns 64b .. 64b + 63, two per word
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float f[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col = 64 * b + 2 * i + h;
            if (col >= kCols) {
              f[h] = 0.0f;
              continue;
            }
            const int32_t corr = per_tensor_adj ? par_adj[col] : za * par_adj[col];
            const float d = __int2float_rn(tot[col] - corr);
            f[h] = fmaf(sa, d * par_sb[col], par_bias[col]);
          }
          if (epi.out_dtype == QLIN_BF16) {
            __nv_bfloat162 p2 = __floats2bfloat162_rn(f[0], f[1]);
            pk[i] = *reinterpret_cast<uint32_t*>(&p2);
          } else {
            __half2 p2 = __floats2half2_rn(f[0], f[1]);
            pk[i] = *reinterpret_cast<uint32_t*>(&p2);
          }
        }
        // 8 x 8 transpose of 16-byte chunks inside each group of 8 lanes
        // (three xor-butterfly steps): afterwards lane 8g + j holds, in slot
        // e, chunk j of row 8g + e, so each store writes 128 contiguous bytes
        // of four rows instead of 16 bytes of 32 rows.
#pragma unroll
        for (int st = 0; st < 3; ++st) {
          const bool up = (lane >> st) & 1;
#pragma unroll
          for (int e0 = 0; e0 < 8; ++e0) {
            if (e0 & (1 << st)) continue;
            const int e1 = e0 | (1 << st);
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              uint32_t& x0 = pk[4 * e0 + w];
              uint32_t& x1 = pk[4 * e1 + w];
              const uint32_t got = __shfl_xor_sync(0xffffffffu, up ? x0 : x1, 1 << st);
              if (up) x0 = got; else x1 = got;
            }
          }
        }
        const int col = c0 + 64 * b + 8 * j;
        const bool in_tile = 64 * b + 8 * j < kCols;  // the 16-byte chunk is this warp's
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int r = row0 + e;
          if (r < T && col < N && in_tile)
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + (int64_t)r * N + col) =
                make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
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

template <int BN>
cudaError_t launch_f16_bn(const CUtensorMap& tmA, const CUtensorMap& tmB, int64_t T, int64_t N, int64_t K,
                          const EpiArgs& epi, void* out, int64_t tiles, cudaStream_t stream) {
  // the shared-memory attribute, set once per device
  static std::once_flag once[64];
  static cudaError_t attr[64];
  int dev = 0;
  cudaError_t st = cudaGetDevice(&dev);
  if (st != cudaSuccess) return st;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [&] {
    attr[dev] = cudaFuncSetAttribute(w8a8_f16_gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     F16Cfg<BN>::kSmemTotal);
  });
  if (attr[dev] != cudaSuccess) return attr[dev];
  const int grid = static_cast<int>(tiles < sm_count() ? tiles : sm_count());
  // programmatic dependent launch: the prologue (barriers, TMEM, tensor maps)
  // overlaps the end of the previous kernel (the activation quantizer)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = F16Cfg<BN>::kSmemTotal;
  cfg.stream = stream;
  cudaLaunchAttribute la[1];
  la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  la[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = la;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, w8a8_f16_gemm_kernel<BN>, tmA, tmB, static_cast<int>(T), static_cast<int>(N),
                            static_cast<int>(K), epi, out, device_error_word());
}

cudaError_t launch_w8a8_gemm_f16(const void* a16, const void* b16, int64_t T, int64_t N, int64_t K,
                                 const W8A8Epilogue& e, void* out, cudaStream_t stream) {
  if (T == 0 || N == 0) return cudaSuccess;
  // the tile width with the least (rounds of tiles on the SMs) x width
  const int64_t sms = sm_count(), mt = (T + kBM - 1) / kBM;
  auto cost = [&](int64_t bn) { return (mt * ((N + bn - 1) / bn) + sms - 1) / sms * bn; };
  const int bn = cost(224) < cost(256) ? 224 : 256;
  const int64_t tiles = mt * ((N + bn - 1) / bn);
  CUtensorMap tmA, tmB;
  cudaError_t st = make_tmap_2d_u8(&tmA, a16, static_cast<uint64_t>(K) * 2, static_cast<uint64_t>(T), kRowBytes, kBM,
                                   /*swizzle_bytes=*/128);
  if (st != cudaSuccess) return st;
  st = make_tmap_2d_u8(&tmB, b16, static_cast<uint64_t>(K) * 2, static_cast<uint64_t>(N), kRowBytes, bn, 128);
  if (st != cudaSuccess) return st;
  EpiArgs epi;
  epi.scale_a = e.scale_a;
  epi.scale_b = e.scale_b;
  epi.azp = e.azp;
  epi.azp_adj = e.azp_adj;
  epi.bias = e.bias;
  epi.scale_a_per_row = e.scale_a_per_row ? 1 : 0;
  epi.scale_b_per_col = e.scale_b_per_col ? 1 : 0;
  epi.bias_dtype = e.bias_dtype;
  epi.out_dtype = e.out_dtype;
  if (bn == 224) return launch_f16_bn<224>(tmA, tmB, T, N, K, epi, out, tiles, stream);
  return launch_f16_bn<256>(tmA, tmB, T, N, K, epi, out, tiles, stream);
}

}  // namespace qlin
