// W8A8: int8 GEMM with an exact int32 accumulator and the fused epilogue
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
// GB300 has no int8 tensor-core MMA (tcgen05 kind::i8 does not exist for
// sm_103a).  The contraction therefore runs on the 16-bit tensor cores on
// exact fp16 copies of the int8 codes: every code is an integer of magnitude
// <= 128, exact in fp16, every product is exact in fp32, and K is processed in
// chunks of 1024 so that every partial sum of a chunk stays within
// 1024 . 128 . 128 = 2^24, where fp32 holds every integer exactly.  Each
// chunk's fp32 accumulator is converted to int32 and added in int32, which
// gives D^ bit for bit.
//
// Kernel structure (one CTA per 128 x 128 output tile, 10 warps):
//   warp 0      TMA producer: int8 tiles of A and B (128 x 64 bytes each)
//               into a 4-stage staging ring.
//   warp 1      TMEM allocation and the MMA issuer: 4 x tcgen05.mma
//               (M=128, N=128, K=16, fp16 -> fp32) per 64-wide K stage into
//               one of two 128-column TMEM accumulators (one per K chunk,
//               double buffered).
//   warps 2-5   converters: int8 staging -> fp16 operand ring in the 128-byte
//               swizzled K-major layout the MMA descriptors describe.  The
//               conversion is a byte permute into the low mantissa of fp16
//               1024 and one half2 subtract per two codes.
//   warps 6-9   epilogue: drain each finished chunk accumulator into int32
//               registers (one output row per thread), then apply the
//               epilogue and store.
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

constexpr int kBM = 128, kBN = 128, kBK = 64;
constexpr int kStg = 4;             // int8 staging stages
constexpr int kOps = 4;             // fp16 operand stages
constexpr int kChunkK = 1024;       // exact fp32 accumulation span
constexpr int kKbPerChunk = kChunkK / kBK;
constexpr int kTmemCols = 2 * kBN;  // two accumulator buffers
constexpr int kThreads = 320;

constexpr int kStgBytes = (kBM + kBN) * kBK;            // 16 KB (A then B)
constexpr int kOpBytes = (kBM + kBN) * kBK * 2;         // 32 KB (A then B, fp16)
constexpr int kSmemStg = 0;
constexpr int kSmemOps = kSmemStg + kStg * kStgBytes;                 // 64 KB
constexpr int kSmemPar = kSmemOps + kOps * kOpBytes;                  // 192 KB
constexpr int kSmemBar = kSmemPar + 3 * kBN * 4;                      // +1.5 KB
constexpr int kNumBars = 2 * kStg + 2 * kOps + 2 + 2 + 1;
constexpr int kSmemMisc = kSmemBar + kNumBars * 8;
constexpr int kSmemTotal = kSmemMisc + 16 + 1024;                     // + alignment slack

// Sites recorded in the device error word when a wait expires.
enum { kSiteStgEmpty = 1, kSiteStgFull, kSiteOpEmpty, kSiteOpFull, kSiteAccEmpty, kSiteAccFull, kSiteDrain };

struct EpiArgs {
  const float* scale_a;
  const float* scale_b;
  const int32_t* azp;
  const int32_t* azp_adj;
  const void* bias;
  int scale_a_per_row, scale_b_per_col, bias_dtype, out_dtype;
};

__device__ __forceinline__ uint32_t h2_sub_u32(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// 16 int8 codes -> 16 exact fp16 values (two 16-byte chunks).
__device__ __forceinline__ void int8x16_to_f16(uint4 v, uint4& h0, uint4& h1) {
  const uint32_t kBias = 0x64806480u;  // fp16 (1152, 1152) = 1024 + 128
  uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // fp16 with exponent of 1024 and the offset code (code + 128) in the low
    // mantissa bits is exactly 1024 + code + 128.
    o[2 * i] = h2_sub_u32(__byte_perm(w[i], 0x64646464u, 0x4140), kBias);
    o[2 * i + 1] = h2_sub_u32(__byte_perm(w[i], 0x64646464u, 0x4342), kBias);
  }
  h0 = make_uint4(o[0], o[1], o[2], o[3]);
  h1 = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ float load_as_float(const void* p, int dtype, int i) {
  if (dtype == QLIN_F16) return __half2float(static_cast<const __half*>(p)[i]);
  if (dtype == QLIN_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  return static_cast<const float*>(p)[i];
}

__global__ void __launch_bounds__(kThreads, 1) w8a8_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                                                                const __grid_constant__ CUtensorMap tmB, int T,
                                                                int N, int K, EpiArgs epi, void* __restrict__ out,
                                                                int32_t* __restrict__ err) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  const int num_kb = (K + kBK - 1) / kBK;
  const int num_chunks = (num_kb + kKbPerChunk - 1) / kKbPerChunk;

  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t bar0 = sbase + kSmemBar;
  auto stg_full = [&](int s) { return bar0 + 8u * s; };
  auto stg_empty = [&](int s) { return bar0 + 8u * (kStg + s); };
  auto op_full = [&](int o) { return bar0 + 8u * (2 * kStg + o); };
  auto op_empty = [&](int o) { return bar0 + 8u * (2 * kStg + kOps + o); };
  auto acc_full = [&](int b) { return bar0 + 8u * (2 * kStg + 2 * kOps + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (2 * kStg + 2 * kOps + 2 + b); };
  const uint32_t mma_done = bar0 + 8u * (2 * kStg + 2 * kOps + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemMisc + 4);
  float* par_sb = reinterpret_cast<float*>(smem + kSmemPar);
  int32_t* par_adj = reinterpret_cast<int32_t*>(smem + kSmemPar + kBN * 4);
  float* par_bias = reinterpret_cast<float*>(smem + kSmemPar + 2 * kBN * 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStg; ++s) { tc::mbar_init(stg_full(s), 1); tc::mbar_init(stg_empty(s), 4); }
    for (int o = 0; o < kOps; ++o) { tc::mbar_init(op_full(o), 4); tc::mbar_init(op_empty(o), 1); }
    for (int b = 0; b < 2; ++b) { tc::mbar_init(acc_full(b), 1); tc::mbar_init(acc_empty(b), 4); }
    tc::mbar_init(mma_done, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  if (warp >= 6) {
    // Per-column epilogue parameters of this tile.
    const int col = threadIdx.x - 192;  // 0..127
    const int n = n0 + col;
    const bool inb = n < N;
    if (epi.out_dtype != QLIN_I32) {
      par_sb[col] = inb ? (epi.scale_b_per_col ? epi.scale_b[n] : epi.scale_b[0]) : 0.0f;
      par_adj[col] = (inb && epi.azp_adj != nullptr) ? epi.azp_adj[n] : 0;
      par_bias[col] = (inb && epi.bias != nullptr) ? load_as_float(epi.bias, epi.bias_dtype, n) : 0.0f;
    }
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
      int issued = 0;
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % kStg;
        if (kb >= kStg && !tc::mbar_wait(stg_empty(s), ((kb / kStg) - 1) & 1, err, kSiteStgEmpty)) {
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        const uint32_t dst = sbase + kSmemStg + s * kStgBytes;
        tc::mbar_arrive_expect_tx(stg_full(s), kStgBytes);
        tc::tma_load_2d(dst, &tmA, kb * kBK, m0, stg_full(s));
        tc::tma_load_2d(dst + kBM * kBK, &tmB, kb * kBK, n0, stg_full(s));
        issued = kb + 1;
      }
      if (*abort_flag) {
        // Let the copies already issued land before the CTA can exit.
        for (int kb = (issued > kStg ? issued - kStg : 0); kb < issued; ++kb)
          tc::mbar_wait(stg_full(kb % kStg), (kb / kStg) & 1, err, kSiteDrain);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_f16(kBM, kBN, 0);  // fp16 x fp16 -> fp32
      bool issued_any = false;
      for (int kb = 0; kb < num_kb; ++kb) {
        const int o = kb % kOps;
        const int chunk = kb / kKbPerChunk, kin = kb % kKbPerChunk;
        const int buf = chunk & 1;
        if (kin == 0 && chunk >= 2 &&
            !tc::mbar_wait(acc_empty(buf), ((chunk / 2) - 1) & 1, err, kSiteAccEmpty)) {
          *abort_flag = 1;
          break;
        }
        if (!tc::mbar_wait(op_full(o), (kb / kOps) & 1, err, kSiteOpFull)) {
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        tc::tc_fence_after();
        const uint32_t a_base = sbase + kSmemOps + o * kOpBytes;
        const uint32_t b_base = a_base + kBM * kBK * 2;
        const uint32_t d = tmem + buf * kBN;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          tc::mma_f16(d, tc::sw128_kmajor_desc(a_base + 32 * k), tc::sw128_kmajor_desc(b_base + 32 * k), idesc,
                      (kin > 0 || k > 0) ? 1u : 0u);
        }
        issued_any = true;
        tc::mma_commit(op_empty(o));
        if (kin == kKbPerChunk - 1 || kb == num_kb - 1) tc::mma_commit(acc_full(buf));
      }
      if (*abort_flag && issued_any) {
        tc::mma_commit(mma_done);
        tc::mbar_wait(mma_done, 0, err, kSiteDrain);
      }
    }
  } else if (warp < 6) {
    // ---------------- converters ----------------
    const int ct = threadIdx.x - 64;  // 0..127
    for (int kb = 0; kb < num_kb; ++kb) {
      const int s = kb % kStg, o = kb % kOps;
      bool ok = tc::mbar_wait(stg_full(s), (kb / kStg) & 1, err, kSiteStgFull);
      if (ok && kb >= kOps) ok = tc::mbar_wait(op_empty(o), ((kb / kOps) - 1) & 1, err, kSiteOpEmpty);
      ok = __all_sync(0xffffffffu, ok && !*abort_flag);  // lanes agree and reconverge
      if (!ok) { *abort_flag = 1; break; }
      const uint32_t src = sbase + kSmemStg + s * kStgBytes;
      const uint32_t dst = sbase + kSmemOps + o * kOpBytes;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int item = ct + 128 * j;          // 1024 16-byte chunks: A rows then B rows
        const int op = item >> 9;               // 0 = A, 1 = B
        const int r = (item >> 2) & 127;        // row within the tile
        const int cc = item & 3;                // 16-byte chunk within the 64-byte row
        const uint4 v = lds128(src + op * (kBM * kBK) + r * kBK + cc * 16);
        uint4 h0, h1;
        int8x16_to_f16(v, h0, h1);
        const uint32_t rowb = dst + op * (kBM * kBK * 2) + (r >> 3) * 1024 + (r & 7) * 128;
        sts128(rowb + (((2 * cc) ^ (r & 7)) << 4), h0);
        sts128(rowb + (((2 * cc + 1) ^ (r & 7)) << 4), h1);
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(op_full(o));
        tc::mbar_arrive(stg_empty(s));
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = m0 + q * 32 + lane;
    int32_t acc[kBN];
#pragma unroll
    for (int i = 0; i < kBN; ++i) acc[i] = 0;
    bool ok = true;
    for (int chunk = 0; chunk < num_chunks; ++chunk) {
      const int buf = chunk & 1;
      ok = tc::mbar_wait(acc_full(buf), (chunk / 2) & 1, err, kSiteAccFull);
      ok = __all_sync(0xffffffffu, ok);  // lanes agree and reconverge before tcgen05.ld
      if (!ok) { *abort_flag = 1; break; }
      tc::tc_fence_after();
#pragma unroll
      for (int cg = 0; cg < kBN / 32; ++cg) {
        uint32_t v[32];
        tc::tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * kBN + cg * 32, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[cg * 32 + i] += __float2int_rn(__uint_as_float(v[i]));
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(acc_empty(buf));
    }
    if (ok && row < T) {
      if (epi.out_dtype == QLIN_I32) {
        int32_t* o = static_cast<int32_t*>(out) + (int64_t)row * N + n0;
#pragma unroll
        for (int c4 = 0; c4 < kBN / 4; ++c4) {
          if (n0 + c4 * 4 < N)
            *reinterpret_cast<int4*>(o + c4 * 4) = make_int4(acc[4 * c4], acc[4 * c4 + 1], acc[4 * c4 + 2],
                                                              acc[4 * c4 + 3]);
        }
      } else {
        const float sa = epi.scale_a_per_row ? epi.scale_a[row] : epi.scale_a[0];
        const int32_t za = epi.azp != nullptr ? epi.azp[row] : 0;
        const bool per_tensor_adj = epi.azp == nullptr && epi.azp_adj != nullptr;
        __half* oh = static_cast<__half*>(out) + (int64_t)row * N + n0;
        __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out) + (int64_t)row * N + n0;
#pragma unroll
        for (int c8 = 0; c8 < kBN / 8; ++c8) {
          if (n0 + c8 * 8 >= N) continue;
          float f[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int col = c8 * 8 + i;
            // D^ - azp . azp_adj in int32, then one conversion to float
            const int32_t corr = per_tensor_adj ? par_adj[col] : za * par_adj[col];
            const float d = __int2float_rn(acc[col] - corr);
            f[i] = fmaf(sa, d * par_sb[col], par_bias[col]);
          }
          if (epi.out_dtype == QLIN_BF16) {
            __nv_bfloat162 p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            *reinterpret_cast<uint4*>(ob + c8 * 8) = *reinterpret_cast<uint4*>(p);
          } else {
            __half2 p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) p[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
            *reinterpret_cast<uint4*>(oh + c8 * 8) = *reinterpret_cast<uint4*>(p);
          }
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

cudaError_t launch_w8a8_gemm(const int8_t* a, const int8_t* b, int64_t T, int64_t N, int64_t K,
                             const W8A8Epilogue& e, void* out, cudaStream_t stream) {
  if (T == 0 || N == 0) return cudaSuccess;
  CUtensorMap tmA, tmB;
  cudaError_t st = make_tmap_2d_u8(&tmA, a, static_cast<uint64_t>(K), static_cast<uint64_t>(T), kBK, kBM);
  if (st != cudaSuccess) return st;
  st = make_tmap_2d_u8(&tmB, b, static_cast<uint64_t>(K), static_cast<uint64_t>(N), kBK, kBN);
  if (st != cudaSuccess) return st;
  st = cudaFuncSetAttribute(w8a8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTotal);
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
  dim3 grid(static_cast<unsigned>((N + kBN - 1) / kBN), static_cast<unsigned>((T + kBM - 1) / kBM));
  w8a8_gemm_kernel<<<grid, kThreads, kSmemTotal, stream>>>(tmA, tmB, static_cast<int>(T), static_cast<int>(N),
                                                           static_cast<int>(K), epi, out, device_error_word());
  return cudaGetLastError();
}

}  // namespace qlin
