// Online Hadamard rotation of activation rows before 4-bit quantization.
//
// The operation: every group of n consecutive elements of a row times the
// normalized Hadamard matrix H_n / sqrt(n), then times signs[k] (+-1 per
// column, QuaRot's diag(+-1)) if given, rounded once to the output type.
//   Sylvester H_n ("LLM and AIGC quantization", QuaRot section): computed
//     by the fast Walsh-Hadamard transform, log2(n) butterfly stages, stage
//     h mapping the pair (a, b) at distance h to (a + b, a - b);
//   regular H_n, n = 4^k (ConvRot section: the Kronecker power of
//     H4 = [[1,1,1,-1],[1,1,-1,1],[1,-1,1,1],[-1,1,1,1]]): computed by
//     radix-4 stages at strides 1, 4, 16, ..., each quad (x0, x1, x2, x3)
//     becoming y_i = s - 2 x_(3-i) with s = (x0 + x1) + (x2 + x3) (H4 is the
//     all-ones matrix minus twice the anti-diagonal).
// fp32 rows, and other group sizes, run the stages in float32 on the CUDA
// cores, then one multiply by c = float32(1/sqrt(n)) and the signs; the
// result is within float32 rounding of the exact rotation.  Each thread holds
// 8 consecutive elements; stages inside them run in registers, stages across
// lanes by shuffles (Sylvester up to n = 256, the regular transform up to
// 256), and Sylvester stages beyond 256 elements through shared memory, one
// CTA of n/8 threads per group.  That form is bound by its shuffle and
// add instructions (0.43-0.57 of HBM at n <= 256, 0.2 at n = 4096).
//
// fp16 and bf16 rows with n = 256 (both matrices) or a Sylvester n = 4096 run
// on the warp-level tensor cores instead, as the dense products of ConvRot's
// formulation cut into Kronecker factors of order 16 (kernels below): the
// arithmetic leaves the issue slots and the kernels stream at HBM speed.
// There the intermediates are kept to 16 significant bits (a bf16 pair), so
// the result is within about 2^-16 of the exact rotation's magnitude before
// the final rounding, and the same on every run.
//
// The kernels do not trigger a programmatic dependent launch: the quantizers
// that read the rotated rows are launched without it and read x at their
// start.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <type_traits>

#include "device_common.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace {

constexpr int kHdThreads = 256;

// Eight elements as float32 through the coherent path (not the read-only
// one: the rotation may run in place).
template <int DT>
__device__ __forceinline__ void load8(const void* p, float* v) {
  if constexpr (DT == 2) {
    const float4 a = static_cast<const float4*>(p)[0], b = static_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 u = *static_cast<const uint4*>(p);
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

template <int DT>
__device__ __forceinline__ void store8(void* p, const float* v) {
  if constexpr (DT == 2) {
    float4* q = static_cast<float4*>(p);
    q[0] = make_float4(v[0], v[1], v[2], v[3]);
    q[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (DT == 0) {
        __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&h);
      } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&h);
      }
    }
    *static_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Sylvester stages h = 1, 2, 4 (inside the thread's 8 elements), up to n/2.
__device__ __forceinline__ void fwht_in_thread(float* v, int n) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
    if (h >= n) break;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i & h) continue;
      const float a = v[i], b = v[i + h];
      v[i] = __fadd_rn(a, b);
      v[i + h] = __fsub_rn(a, b);
    }
  }
}

// Sylvester stages h = 8 m for lane bits m = 1 .. 16 while h < min(n, 256).
__device__ __forceinline__ void fwht_across_lanes(float* v, int n, int lane) {
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    if (8 * m >= n) break;
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
      v[i] = upper ? __fsub_rn(o, v[i]) : __fadd_rn(v[i], o);  // (a + b, a - b), a the lower index
    }
  }
}

__device__ __forceinline__ float quad_out(float q0, float q1, float q2, float q3, int pos) {
  const float s = __fadd_rn(__fadd_rn(q0, q1), __fadd_rn(q2, q3));
  const float x = pos == 0 ? q3 : pos == 1 ? q2 : pos == 2 ? q1 : q0;  // x_(3 - pos)
  return __fsub_rn(s, 2.0f * x);
}

// Regular-Hadamard radix-4 stages at strides 1, 4, 16, 64 while the stride is < n.
__device__ __forceinline__ void regular_stages(float* v, int n, int lane) {
  // stride 1: quads (0..3) and (4..7) of the thread
  {
    float y[8];
#pragma unroll
    for (int b = 0; b < 8; b += 4)
#pragma unroll
      for (int p = 0; p < 4; ++p) y[b + p] = quad_out(v[b], v[b + 1], v[b + 2], v[b + 3], p);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = y[i];
  }
  if (n <= 4) return;
  // stride 4: quad (r, r + 4, r + 8, r + 12) of a 16-element block = this
  // lane's elements r, r + 4 and the neighbour lane's (lane ^ 1)
  {
    const bool odd = (lane & 1) != 0;
    float y[8];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float o0 = __shfl_xor_sync(0xffffffffu, v[r], 1);
      const float o1 = __shfl_xor_sync(0xffffffffu, v[r + 4], 1);
      const float q0 = odd ? o0 : v[r], q1 = odd ? o1 : v[r + 4];
      const float q2 = odd ? v[r] : o0, q3 = odd ? v[r + 4] : o1;
      y[r] = quad_out(q0, q1, q2, q3, odd ? 2 : 0);
      y[r + 4] = quad_out(q0, q1, q2, q3, odd ? 3 : 1);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = y[i];
  }
  // strides 16 and 64: the quad's members are the lanes that differ in two
  // lane bits (1-2, then 3-4), same element index.  Three shuffles give the
  // pair sum (q0 + q1 or q2 + q3), then s, then x_(3 - pos), the lane whose
  // position is pos ^ 3; float addition is commutative, so every lane of the
  // quad holds the same s = (q0 + q1) + (q2 + q3).
#pragma unroll
  for (int shift = 1; shift <= 3; shift += 2) {
    if ((8 << shift) >= n) break;  // stride 8 . 2^shift
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float pair = __fadd_rn(v[i], __shfl_xor_sync(0xffffffffu, v[i], 1 << shift));
      const float sum = __fadd_rn(pair, __shfl_xor_sync(0xffffffffu, pair, 2 << shift));
      const float mirror = __shfl_xor_sync(0xffffffffu, v[i], 3 << shift);
      v[i] = __fsub_rn(sum, 2.0f * mirror);
    }
  }
}

__device__ __forceinline__ void scale_and_sign(float* v, float c, const int8_t* __restrict__ signs, int64_t col0) {
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], c);
  if (signs != nullptr) {
    const uint2 sg = __ldg(reinterpret_cast<const uint2*>(signs + col0));
    const uint32_t w[2] = {sg.x, sg.y};
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (static_cast<int8_t>((w[i >> 2] >> (8 * (i & 3))) & 0xFF) < 0) v[i] = -v[i];
  }
}

// Groups of n <= 256: one warp walks 256 consecutive elements (all its groups),
// grid-stride over the rows' 8-element vectors; every lane of a warp runs the
// same iterations (the shuffles need the whole warp), and a group is all in
// range or all out (K is a multiple of n).
template <int DT, int KIND>
__global__ void __launch_bounds__(kHdThreads) hadamard_warp_kernel(const void* x, int64_t nvec, int K,
                                                                  int n, float c, const int8_t* __restrict__ signs,
                                                                  void* y) {
  // x and y may be the same rows (in place): every element is read by the
  // thread that later writes it, before the write
  constexpr int EB = DT == 2 ? 4 : 2;
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kHdThreads;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kHdThreads + (threadIdx.x & ~31); base < nvec;
       base += stride) {
    const int64_t vi = base + lane;
    const bool active = vi < nvec;
    float v[8];
    if (active) {
      load8<DT>(static_cast<const char*>(x) + vi * 8 * EB, v);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    }
    if constexpr (KIND == 0) {
      fwht_in_thread(v, n);
      fwht_across_lanes(v, n, lane);
    } else {
      regular_stages(v, n, lane);
    }
    if (!active) continue;
    scale_and_sign(v, c, signs, (vi * 8) % K);
    store8<DT>(static_cast<char*>(y) + vi * 8 * EB, v);
  }
}

// Sylvester groups of 512 .. 8192: one CTA of n / 8 threads per group, the
// stages h >= 256 through shared memory (each thread keeps its own 8 values
// in registers and reads the 8 partners).
template <int DT>
__global__ void __launch_bounds__(1024) hadamard_cta_kernel(const void* x, int64_t groups, int K, int n,
                                                            float c, const int8_t* __restrict__ signs,
                                                            void* y, int64_t e_base = 0) {
  // x and y point at element e_base of the rows (the signs' column is taken from it)
  extern __shared__ __align__(16) float buf[];
  constexpr int EB = DT == 2 ? 4 : 2;
  const int tid = threadIdx.x, lane = tid & 31;
  for (int64_t g = blockIdx.x; g < groups; g += gridDim.x) {
    const int64_t e0 = g * n + 8 * tid;  // first element of this thread
    float v[8];
    load8<DT>(static_cast<const char*>(x) + e0 * EB, v);
    fwht_in_thread(v, n);
    fwht_across_lanes(v, n, lane);
    for (int h = 256; h < n; h <<= 1) {
      // 32-byte rows per thread, written and read as two 16-byte pieces
      float4* mine = reinterpret_cast<float4*>(buf + 8 * tid);
      mine[0] = make_float4(v[0], v[1], v[2], v[3]);
      mine[1] = make_float4(v[4], v[5], v[6], v[7]);
      __syncthreads();
      const int j0 = 8 * tid;  // the 8 elements share bit h (h >= 256 > 7)
      const bool upper = (j0 & h) != 0;
      const float4* other = reinterpret_cast<const float4*>(buf + (j0 ^ h));
      const float4 o0 = other[0], o1 = other[1];
      const float o[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = upper ? __fsub_rn(o[i], v[i]) : __fadd_rn(v[i], o[i]);
      __syncthreads();
    }
    scale_and_sign(v, c, signs, (e_base + e0) % K);
    store8<DT>(static_cast<char*>(y) + e0 * EB, v);
  }
}

// ---- groups of 256 on the tensor cores (fp16 / bf16 rows) ----------------
//
// A group of 256 elements is a 16 x 16 matrix M (element 16 a + b at row a,
// column b), and both Hadamard matrices of order 256 are Kronecker squares of
// a symmetric 16 x 16 factor F (Sylvester: H16; regular: H4 (x) H4, ConvRot's
// construction), so the rotated group is x . (F (x) F) = F . M . F, two
// 16 x 16 products per group on the warp-level tensor cores:
//   stage 1: Q = F . M      (A = F, constant; B = M, read with ldmatrix.trans
//                            from the warp's shared-memory copy of the group)
//   stage 2: Y = Q . F      (A = Q: the m16n8k16 accumulator of stage 1 has
//                            the layout of the next A operand; B = F)
// Products of +-1 with the fp16 / bf16 inputs are exact and the tensor core
// accumulates in fp32.  Q enters stage 2 as a pair of bf16 values (hi and the
// remainder Q - hi), 16 significant bits with fp32's range, so Y is within
// about 2^-16 |Y| of the exact product before the one rounding to the output
// type.  Per group a warp issues ~65 instructions (one 16-byte load and store
// per lane, 6 MMAs), against several hundred for the shuffle butterflies.

constexpr int kHmWarps = 8;           // warps per CTA
constexpr int kHmBatch = 4;           // groups in flight per warp
constexpr int kHmGroupBytes = 512;    // 256 elements of 2 bytes

// F[i][j] of the 16 x 16 factor: Sylvester (-1)^popcount(i & j); regular the
// product of H4 entries over the two base-4 digits (H4[r][c] = -1 exactly when
// r + c == 3).
__device__ __forceinline__ float hm_factor(int kind, int i, int j) {
  if (kind == 0) return (__popc(i & j) & 1) ? -1.0f : 1.0f;
  const bool neg = (((i >> 2) + (j >> 2)) == 3) != (((i & 3) + (j & 3)) == 3);
  return neg ? -1.0f : 1.0f;
}

template <int DT>
__device__ __forceinline__ uint32_t hm_pack(float lo, float hi) {
  if constexpr (DT == 0) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// D = A . B + D, m16n8k16, fp32 accumulation; DT 0: fp16 operands, 1: bf16.
template <int DT>
__device__ __forceinline__ void hm_mma(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
  if constexpr (DT == 0)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (hi, lo) bf16 pairs of two floats: hi = bf16(v), lo = bf16(v - hi).
__device__ __forceinline__ void hm_split(float v0, float v1, uint32_t& hi, uint32_t& lo) {
  hi = hm_pack<1>(v0, v1);
  const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xFFFF0000u);
  lo = hm_pack<1>(__fsub_rn(v0, h0), __fsub_rn(v1, h1));
}

// Byte offset of the 16-byte half `h` of row r of a group's 16 x 32-byte
// tile: the halves of rows 4-7 and 12-15 are swapped, so that the eight rows
// an ldmatrix phase reads fall in distinct banks.
__device__ __forceinline__ uint32_t hm_off(int r, int h) { return r * 32 + ((h ^ ((r >> 2) & 1)) << 4); }

template <int DT, int KIND>
__global__ void __launch_bounds__(kHmWarps * 32) hadamard256_mma_kernel(const void* x, int64_t groups, int K,
                                                                        const int8_t* __restrict__ signs, void* y) {
  __shared__ __align__(128) unsigned char tile[kHmWarps][kHmBatch][kHmGroupBytes];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  // F as the A operand (rows g, g + 8; columns 2c, 2c + 1, 2c + 8, 2c + 9)
  // in the input type for stage 1, and in bf16 for stage 2's B operand (F is
  // symmetric, so the same four words serve as the B fragments of both
  // column tiles: b0/b1 of tile 0 = a0/a2, of tile 1 = a1/a3)
  uint32_t fa[4], fb[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int r = g + 8 * (q & 1), k = 2 * c + 8 * (q >> 1);
    const float f0 = hm_factor(KIND, r, k), f1 = hm_factor(KIND, r, k + 1);
    fa[q] = hm_pack<DT>(f0, f1);
    fb[q] = hm_pack<1>(f0, f1);
  }
  const float scale = 1.0f / 16.0f;  // 1 / sqrt(256), exact
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kHmWarps;
  const char* xb = static_cast<const char*>(x);
  char* yb = static_cast<char*>(y);
  const uint32_t tbase = static_cast<uint32_t>(__cvta_generic_to_shared(&tile[warp][0][0]));
  // ldmatrix.x4.trans row addresses: matrix i = lane / 8 covers rows
  // 8 (i & 1) .. + 7 and column half i >> 1; this lane gives row (lane % 8)
  const int lm_row = (lane & 7) + 8 * ((lane >> 3) & 1), lm_half = lane >> 4;
  for (int64_t g0 = (static_cast<int64_t>(blockIdx.x) * kHmWarps + warp) * kHmBatch; g0 < groups;
       g0 += nwarps * kHmBatch) {
    uint4 in[kHmBatch];
#pragma unroll
    for (int b = 0; b < kHmBatch; ++b)
      if (g0 + b < groups) in[b] = *reinterpret_cast<const uint4*>(xb + (g0 + b) * kHmGroupBytes + lane * 16);
    __syncwarp();  // the previous batch's output reads of the tile are done
#pragma unroll
    for (int b = 0; b < kHmBatch; ++b)
      if (g0 + b < groups) {
        const uint32_t a = tbase + b * kHmGroupBytes + hm_off(lane >> 1, lane & 1);
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(in[b].x), "r"(in[b].y), "r"(in[b].z),
                     "r"(in[b].w)
                     : "memory");
      }
    __syncwarp();
#pragma unroll
    for (int b = 0; b < kHmBatch; ++b) {
      if (g0 + b >= groups) break;
      const uint32_t tb = tbase + b * kHmGroupBytes;
      uint32_t m0, m1, m2, m3;  // B fragments of M: (rows 0-7 | 8-15) x (columns 0-7 | 8-15)
      asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                   : "=r"(m0), "=r"(m1), "=r"(m2), "=r"(m3)
                   : "r"(tb + hm_off(lm_row, lm_half)));
      // stage 1: Q = F . M, column tiles 0-7 and 8-15
      float q0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, q1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      hm_mma<DT>(q0, fa[0], fa[1], fa[2], fa[3], m0, m1);
      hm_mma<DT>(q1, fa[0], fa[1], fa[2], fa[3], m2, m3);
      // stage 2: Y = Q . F with Q as A fragments (rows g, g + 8; columns
      // 2c.. of tile 0, then of tile 1), hi and lo parts
      uint32_t ah[4], al[4];
      hm_split(q0[0], q0[1], ah[0], al[0]);
      hm_split(q0[2], q0[3], ah[1], al[1]);
      hm_split(q1[0], q1[1], ah[2], al[2]);
      hm_split(q1[2], q1[3], ah[3], al[3]);
      float y0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, y1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      hm_mma<1>(y0, al[0], al[1], al[2], al[3], fb[0], fb[2]);
      hm_mma<1>(y0, ah[0], ah[1], ah[2], ah[3], fb[0], fb[2]);
      hm_mma<1>(y1, al[0], al[1], al[2], al[3], fb[1], fb[3]);
      hm_mma<1>(y1, ah[0], ah[1], ah[2], ah[3], fb[1], fb[3]);
      // Y[g][2c..], Y[g+8][2c..] of each column tile back into the tile,
      // scaled and rounded (the column signs come after the transpose)
      const uint32_t o00 = hm_pack<DT>(y0[0] * scale, y0[1] * scale), o01 = hm_pack<DT>(y0[2] * scale, y0[3] * scale);
      const uint32_t o10 = hm_pack<DT>(y1[0] * scale, y1[1] * scale), o11 = hm_pack<DT>(y1[2] * scale, y1[3] * scale);
      __syncwarp();  // every lane's ldmatrix of this group is done
      asm volatile("st.shared.u32 [%0], %1;" ::"r"(tb + hm_off(g, 0) + 4 * c), "r"(o00) : "memory");
      asm volatile("st.shared.u32 [%0], %1;" ::"r"(tb + hm_off(g + 8, 0) + 4 * c), "r"(o01) : "memory");
      asm volatile("st.shared.u32 [%0], %1;" ::"r"(tb + hm_off(g, 1) + 4 * c), "r"(o10) : "memory");
      asm volatile("st.shared.u32 [%0], %1;" ::"r"(tb + hm_off(g + 8, 1) + 4 * c), "r"(o11) : "memory");
    }
    __syncwarp();
#pragma unroll
    for (int b = 0; b < kHmBatch; ++b) {
      if (g0 + b >= groups) break;
      uint4 o;
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(o.x), "=r"(o.y), "=r"(o.z), "=r"(o.w)
                   : "r"(tbase + b * kHmGroupBytes + hm_off(lane >> 1, lane & 1))
                   : "memory");
      const int64_t e0 = (g0 + b) * 256 + lane * 8;  // first element of this lane's 8
      if (signs != nullptr) {
        // a -1 sign flips the sign bit of the element (exact)
        const uint2 sg = __ldg(reinterpret_cast<const uint2*>(signs + e0 % K));
        uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t sb = (i < 4 ? sg.x : sg.y) >> (8 * (i & 3));
          if (sb & 0x80u) w[i >> 1] ^= 0x8000u << (16 * (i & 1));
        }
        o = make_uint4(w[0], w[1], w[2], w[3]);
      }
      *reinterpret_cast<uint4*>(yb + e0 * 2) = o;
    }
  }
}

// ---- Sylvester groups of 512 .. 4096 on the tensor cores (fp16 / bf16 rows) --
//
// H_n = H_m (x) H_256 with m = n / 256: with a group cut into m sub-blocks
// x_a of 256,
//   y[256 c + j] = sum_a H_m[a][c] . Z_a[j],   Z_a = x_a . H_256 = F . M_a . F.
// A CTA takes 4096 consecutive elements at a time (16 sub-blocks: 16 / m
// whole groups): each warp rotates two sub-blocks exactly as above
// (unnormalized), the CTA collects Z (16 x 256, as bf16 hi and lo parts) in
// shared memory, and a third 16 x 16 product Y = B . Z combines the
// sub-blocks of each group, B = diag(H_m, ..., H_m) (for n = 4096, B = F),
// each warp 32 of the 256 columns; then one multiply by float32(1/sqrt(n))
// (exact for n = 1024 and 4096).  The next 4096 elements are loaded while the
// current ones are rotated.  The kernel takes whole blocks of 4096 only (a
// bounds check per load cost 15% here); the groups after the last whole block
// (fewer than 4096 elements, m < 16) run through the float32 butterflies.

constexpr int kH4Warps = 8;

// Byte offset of element (row r, column j) of a 16 x 256 bf16 / fp16 matrix
// (512-byte rows) with its 16-byte chunks permuted by (r & 7), so that eight
// rows of one chunk column fall in distinct banks.
__device__ __forceinline__ uint32_t h4_off(int r, int j) {
  return r * 512 + ((((j >> 3) ^ (r & 7))) << 4) + (j & 7) * 2;
}

template <int DT, int m>
__global__ void __launch_bounds__(kH4Warps * 32) hadamard4096_mma_kernel(const void* x, int64_t passes, float scale_rt,
                                                                         int K, const int8_t* __restrict__ signs,
                                                                         void* y) {
  // 1 / sqrt(256 m): exact for m = 4 and 16, float32-rounded (scale_rt) otherwise
  const float scale = m == 16 ? 1.0f / 64.0f : m == 4 ? 1.0f / 32.0f : scale_rt;
  // passes: blocks of 4096 consecutive elements (16 sub-blocks of 256)
  const int64_t groups = passes;
  __shared__ __align__(128) unsigned char stage[kH4Warps][2][kHmGroupBytes];  // inputs, then the output rows
  __shared__ __align__(128) unsigned char zbuf[2][16 * 512];                 // Z as bf16: hi, lo
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  // F (= H16) for the sub-block rotations; B = diag(H_m, ..., H_m) (rows c,
  // columns a: H_m[c % m][a % m] when c / m == a / m, else 0) to combine them.
  // On a diagonal block H16[c][a] = (-1)^popcount(c / m) H_m[c % m][a % m]
  // (the bits above log2 m are equal), so B is F masked and sign-flipped.
  // F is kept once, as bf16 (fb); the fp16 copy for stage 1 is rebuilt from
  // its sign bits where it is used (+-1: 0x3C00 in fp16, 0x3F80 in bf16),
  // which keeps the fp16 build within 64 registers (4 CTAs per SM)
  uint32_t fb[4], fc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int r = g + 8 * (q & 1), k = 2 * c + 8 * (q >> 1);
    const float f0 = hm_factor(0, r, k), f1 = hm_factor(0, r, k + 1);
    fb[q] = hm_pack<1>(f0, f1);
    // k is even and m >= 2, so k and k + 1 lie in the same block
    fc[q] = m == 16 ? fb[q] : r / m != k / m ? 0u : fb[q] ^ ((__popc(r / m) & 1) ? 0x80008000u : 0u);
  }
  const char* xb = static_cast<const char*>(x);
  char* yb = static_cast<char*>(y);
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(&stage[warp][0][0]));
  const uint32_t sall = static_cast<uint32_t>(__cvta_generic_to_shared(&stage[0][0][0]));
  const uint32_t zb = static_cast<uint32_t>(__cvta_generic_to_shared(&zbuf[0][0]));
  const int lm_row = (lane & 7) + 8 * ((lane >> 3) & 1), lm_half = lane >> 4;
  int64_t gi = blockIdx.x;
  uint4 in[2];
  if (gi < groups) {
#pragma unroll
    for (int sb = 0; sb < 2; ++sb)
      in[sb] = *reinterpret_cast<const uint4*>(xb + gi * 8192 + (2 * warp + sb) * kHmGroupBytes + lane * 16);
  }
  for (; gi < groups; gi += gridDim.x) {
    // this warp's two sub-blocks into its staging tiles; the next group's load in flight
#pragma unroll
    for (int sb = 0; sb < 2; ++sb) {
      const uint32_t a = sbase + sb * kHmGroupBytes + hm_off(lane >> 1, lane & 1);
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(in[sb].x), "r"(in[sb].y), "r"(in[sb].z),
                   "r"(in[sb].w)
                   : "memory");
    }
    const int64_t gn = gi + gridDim.x;
    if (gn < groups) {
#pragma unroll
      for (int sb = 0; sb < 2; ++sb)
        in[sb] = *reinterpret_cast<const uint4*>(xb + gn * 8192 + (2 * warp + sb) * kHmGroupBytes + lane * 16);
    }
    __syncwarp();
#pragma unroll
    for (int sb = 0; sb < 2; ++sb) {
      const int a = 2 * warp + sb;
      uint32_t m0, m1, m2, m3;
      asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                   : "=r"(m0), "=r"(m1), "=r"(m2), "=r"(m3)
                   : "r"(sbase + sb * kHmGroupBytes + hm_off(lm_row, lm_half)));
      float q0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, q1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      uint32_t fa[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if constexpr (DT == 0)
          asm volatile("lop3.b32 %0, %1, 0x80008000, 0x3C003C00, 0xEA;" : "=r"(fa[q]) : "r"(fb[q]));
        else
          fa[q] = fb[q];
      }
      hm_mma<DT>(q0, fa[0], fa[1], fa[2], fa[3], m0, m1);
      hm_mma<DT>(q1, fa[0], fa[1], fa[2], fa[3], m2, m3);
      uint32_t ah[4], al[4];
      hm_split(q0[0], q0[1], ah[0], al[0]);
      hm_split(q0[2], q0[3], ah[1], al[1]);
      hm_split(q1[0], q1[1], ah[2], al[2]);
      hm_split(q1[2], q1[3], ah[3], al[3]);
      float y0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, y1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      hm_mma<1>(y0, al[0], al[1], al[2], al[3], fb[0], fb[2]);
      hm_mma<1>(y0, ah[0], ah[1], ah[2], ah[3], fb[0], fb[2]);
      hm_mma<1>(y1, al[0], al[1], al[2], al[3], fb[1], fb[3]);
      hm_mma<1>(y1, ah[0], ah[1], ah[2], ah[3], fb[1], fb[3]);
      // Z_a[j] for j = 16 g + 2c (+1), 16 (g + 8) + 2c, then 8 columns on
      const float zv[4][2] = {{y0[0], y0[1]}, {y0[2], y0[3]}, {y1[0], y1[1]}, {y1[2], y1[3]}};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int j = 16 * (g + 8 * (p & 1)) + 8 * (p >> 1) + 2 * c;
        uint32_t hi, lo;
        hm_split(zv[p][0], zv[p][1], hi, lo);
        const uint32_t o = h4_off(a, j);
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(zb + o), "r"(hi) : "memory");
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(zb + 16 * 512 + o), "r"(lo) : "memory");
      }
    }
    __syncthreads();  // Z complete; every warp's staging tiles free
    // Y = B . Z on this warp's columns 32 w .. 32 w + 31 (four column tiles)
#pragma unroll
    for (int t = 0; t < 4; t += 2) {
      const int j0 = 32 * warp + 8 * t;
      // matrices: rows 0-7 | 8-15 of columns j0.. and j0 + 8..
      const int r = (lane & 7) + 8 * ((lane >> 3) & 1), jj = j0 + 8 * (lane >> 4);
      uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
      asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                   : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
                   : "r"(zb + h4_off(r, jj)));
      asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                   : "=r"(l0), "=r"(l1), "=r"(l2), "=r"(l3)
                   : "r"(zb + 16 * 512 + h4_off(r, jj)));
      float d0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, d1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      hm_mma<1>(d0, fc[0], fc[1], fc[2], fc[3], l0, l1);
      hm_mma<1>(d0, fc[0], fc[1], fc[2], fc[3], h0, h1);
      hm_mma<1>(d1, fc[0], fc[1], fc[2], fc[3], l2, l3);
      hm_mma<1>(d1, fc[0], fc[1], fc[2], fc[3], h2, h3);
      // y[256 c_out + j], c_out = g, g + 8, j = j0 (+8) + 2c: scaled, rounded,
      // into the output rows (the staging area, 16 rows of 512 bytes)
      const float dv[4][2] = {{d0[0], d0[1]}, {d0[2], d0[3]}, {d1[0], d1[1]}, {d1[2], d1[3]}};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int co = g + 8 * (p & 1), j = j0 + 8 * (p >> 1) + 2 * c;
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(sall + h4_off(co, j)),
                     "r"(hm_pack<DT>(dv[p][0] * scale, dv[p][1] * scale))
                     : "memory");
      }
    }
    __syncthreads();  // the output rows are complete; Z may be overwritten
    // this warp writes output rows 2w and 2w + 1 (1 KB, 16 bytes per lane per row)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = 2 * warp + rr;
      uint4 o;
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(o.x), "=r"(o.y), "=r"(o.z), "=r"(o.w)
                   : "r"(sall + h4_off(row, 8 * lane))
                   : "memory");
      const int64_t e0 = gi * 4096 + row * 256 + 8 * lane;
      if (signs != nullptr) {
        const uint2 sg = __ldg(reinterpret_cast<const uint2*>(signs + e0 % K));
        uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t sb = (i < 4 ? sg.x : sg.y) >> (8 * (i & 3));
          if (sb & 0x80u) w[i >> 1] ^= 0x8000u << (16 * (i & 1));
        }
        o = make_uint4(w[0], w[1], w[2], w[3]);
      }
      *reinterpret_cast<uint4*>(yb + e0 * 2) = o;
    }
    __syncthreads();  // the output rows are read before the next group's inputs land there
  }
}

}  // namespace

cudaError_t launch_hadamard(const void* x, qlin_dtype dtype, int64_t rows, int64_t K, qlin_hadamard_kind kind,
                            int64_t n, const int8_t* signs, void* y, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const float c = static_cast<float>(1.0 / std::sqrt(static_cast<double>(n)));
  const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
  auto go = [&](auto dt) -> cudaError_t {
    constexpr int DT = decltype(dt)::value;
    if constexpr (DT != 2) {
      if (n == 256) {
        // tensor cores: 4 CTAs of 8 warps per SM, each warp 4 groups at a time
        const int64_t groups = rows * (K / 256);
        const int64_t want = (groups + kHmWarps * kHmBatch - 1) / (kHmWarps * kHmBatch);
        const int64_t cap4 = static_cast<int64_t>(sm_count()) * 4;
        const unsigned grid = static_cast<unsigned>(want < cap4 ? want : cap4);
        if (kind == QLIN_HADAMARD_SYLVESTER)
          hadamard256_mma_kernel<DT, 0><<<grid, kHmWarps * 32, 0, stream>>>(x, groups, static_cast<int>(K), signs, y);
        else
          hadamard256_mma_kernel<DT, 1><<<grid, kHmWarps * 32, 0, stream>>>(x, groups, static_cast<int>(K), signs, y);
        return cudaGetLastError();
      }
      if (n >= 512 && n <= 4096 && kind == QLIN_HADAMARD_SYLVESTER) {
        const int64_t total = rows * K, passes = total / 4096;
        const int Ki = static_cast<int>(K);
        if (passes > 0) {
          const int64_t cap4 = static_cast<int64_t>(sm_count()) * 4;
          const unsigned grid = static_cast<unsigned>(passes < cap4 ? passes : cap4);
          switch (n) {
            case 512: hadamard4096_mma_kernel<DT, 2><<<grid, kH4Warps * 32, 0, stream>>>(x, passes, c, Ki, signs, y); break;
            case 1024: hadamard4096_mma_kernel<DT, 4><<<grid, kH4Warps * 32, 0, stream>>>(x, passes, c, Ki, signs, y); break;
            case 2048: hadamard4096_mma_kernel<DT, 8><<<grid, kH4Warps * 32, 0, stream>>>(x, passes, c, Ki, signs, y); break;
            default: hadamard4096_mma_kernel<DT, 16><<<grid, kH4Warps * 32, 0, stream>>>(x, passes, c, Ki, signs, y); break;
          }
          cudaError_t e = cudaGetLastError();
          if (e != cudaSuccess) return e;
        }
        // whole groups after the last block of 4096 elements: the butterflies
        const int64_t done = passes * 4096, tail_groups = (total - done) / n;
        if (tail_groups == 0) return cudaSuccess;
        constexpr int EB = DT == 2 ? 4 : 2;
        const size_t smem = static_cast<size_t>(n) * sizeof(float);
        hadamard_cta_kernel<DT><<<static_cast<unsigned>(tail_groups), static_cast<unsigned>(n / 8), smem, stream>>>(
            static_cast<const char*>(x) + done * EB, tail_groups, Ki, static_cast<int>(n), c, signs,
            static_cast<char*>(y) + done * EB, done);
        return cudaGetLastError();
      }
    }
    if (n <= 256) {
      const int64_t nvec = rows * (K / 8);
      const int64_t want = (nvec + kHdThreads - 1) / kHdThreads;
      const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
      if (kind == QLIN_HADAMARD_SYLVESTER)
        hadamard_warp_kernel<DT, 0><<<grid, kHdThreads, 0, stream>>>(x, nvec, static_cast<int>(K),
                                                                       static_cast<int>(n), c, signs, y);
      else
        hadamard_warp_kernel<DT, 1><<<grid, kHdThreads, 0, stream>>>(x, nvec, static_cast<int>(K),
                                                                       static_cast<int>(n), c, signs, y);
      return cudaGetLastError();
    }
    const int64_t groups = rows * (K / n);
    const unsigned grid = static_cast<unsigned>(groups < cap ? groups : cap);
    const size_t smem = static_cast<size_t>(n) * sizeof(float);
    if (smem > 48 * 1024) {
      cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(hadamard_cta_kernel<DT>));
      if (e != cudaSuccess) return e;
    }
    hadamard_cta_kernel<DT><<<grid, static_cast<unsigned>(n / 8), smem, stream>>>(x, groups, static_cast<int>(K),
                                                                                static_cast<int>(n), c, signs, y);
    return cudaGetLastError();
  };
  switch (dtype) {
    case QLIN_F16: return go(std::integral_constant<int, 0>{});
    case QLIN_BF16: return go(std::integral_constant<int, 1>{});
    default: return go(std::integral_constant<int, 2>{});
  }
}

}  // namespace qlin
