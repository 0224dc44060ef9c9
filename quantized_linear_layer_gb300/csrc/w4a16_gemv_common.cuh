// Shared device code of the W4A16 decode GEMV kernels (one launch per linear,
// and the persistent sequence of linears): the integer dot products of one
// 32-code chunk, the fixed-point activation planes, and the cross-lane sum
// of a batch of rows.  The arithmetic is stated in w4a16_gemv.cu.
#pragma once

#include <cuda_fp16.h>

#include "device_common.cuh"

namespace qlin {
namespace gv {

// d = c + sum_i a.byte[i] . b.byte[i], a unsigned bytes, b signed bytes.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// sum_k (n[k] - z) . x_fix[k] over one 32-code chunk (16 bytes).
// xp[p][2w] / xp[p][2w + 1] hold byte plane p of the even / odd codes of
// word w.  The even codes are masked to bytes in place (w & 0x0F0F0F0F); the
// odd ones stay in the high nibble of their byte (w & 0xF0F0F0F0 = 16 n) and
// get their own accumulators (multiples of 16, shifted back exactly).  Every
// partial sum is an exact integer below 2^20, and the zero-point term
// z . sum(plane) is subtracted per plane in int32, so the result is
// sum (n - z) . x_fix exactly until the one conversion to fp32 per plane.
__device__ __forceinline__ float gv_chunk(uint4 q, const uint32_t (*xp)[8], const int* xsum, int z) {
  int he = 0, ho = 0, me = 0, mo = 0, le = 0, lo = 0;
  const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint32_t ev = wd[w] & 0x0F0F0F0Fu, od = wd[w] & 0xF0F0F0F0u;
    he = dp4a_us(ev, xp[0][2 * w], he);
    ho = dp4a_us(od, xp[0][2 * w + 1], ho);
    me = dp4a_us(ev, xp[1][2 * w], me);
    mo = dp4a_us(od, xp[1][2 * w + 1], mo);
    le = dp4a_us(ev, xp[2][2 * w], le);
    lo = dp4a_us(od, xp[2][2 * w + 1], lo);
  }
  const int h = he + (ho >> 4) - z * xsum[0];
  const int m = me + (mo >> 4) - z * xsum[1];
  const int l = le + (lo >> 4) - z * xsum[2];
  return fmaf(static_cast<float>(h), 65536.0f, fmaf(static_cast<float>(m), 256.0f, static_cast<float>(l)));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Rows rg, rg + RG, rg + 2 RG, rg + 3 RG of one stage: the thread's partial
// sums.  Row indices past the stage are clamped to its last row (their sums
// are never stored), so the four chunks run without branches and interleave;
// idle lanes have zero activations and contribute 0.  Addresses are 32-bit
// shared-window offsets: cbase = the thread's chunk in the stage, sbase = its
// group's packed {scale, zero} of the stage's first row (fp16 scale bits in
// the low half, the zero-point in the high half).
template <int B>
__device__ __forceinline__ void gv_batch(uint32_t cbase, uint32_t sbase, int rows_i, int RG, int rg, int row_bytes,
                                         int G, const uint32_t (*xp)[8], const int* xsum, float sx, float* p) {
  uint4 q[B];
  uint32_t m[B];
#pragma unroll
  for (int b = 0; b < B; ++b) {
    const int rrc = min(rg + RG * b, rows_i - 1);
    q[b] = lds128(cbase + rrc * row_bytes);
    m[b] = lds32(sbase + rrc * G * 4);
  }
#pragma unroll
  for (int b = 0; b < B; ++b) {
    const float sg = __half2float(__ushort_as_half(static_cast<unsigned short>(m[b] & 0xFFFFu)));
    p[b] = (sg * sx) * gv_chunk(q[b], xp, xsum, static_cast<int>(m[b] >> 16));
  }
}

// A thread's activation chunk as fixed-point byte planes.
struct GvX {
  uint32_t xp[3][8];  // byte planes hi, mid, lo
  int xsum[3];        // plane sums over the chunk
  float sx;           // x = x_fix . sx
};

// Builds the planes of a chunk from its 32 activations xf (when act):
// x_fix = round(x / sx) with sx = max|x| / (127 . 2^15), so that
// |x - x_fix . sx| <= 0.75 sx (the rounded quotient, 2^-22.4 of the chunk's
// largest |x|: finer than fp16 for every element above max|x| . 2^-11), in
// three signed base-256 digits.
__device__ __forceinline__ void gv_build_planes(const float* xf, bool act, GvX& X) {
  uint32_t (&xp)[3][8] = X.xp;
  int (&xsum)[3] = X.xsum;
  xsum[0] = xsum[1] = xsum[2] = 0;
  float sx = 1.0f;
  if (act) {
    // four partial maxima (short dependency chains)
    float pm[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int t = 0; t < 32; ++t) pm[t & 3] = fmaxf(pm[t & 3], fabsf(xf[t]));
    const float amax = fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]));
    sx = amax > 0.0f ? amax * (1.0f / 4161536.0f) : 1.0f;   // 4161536 = 127 . 2^15
    const float inv = 1.0f / sx;
    // x_fix + 0x8080: byte 0 ^ 0x80 = lo, byte 1 ^ 0x80 = mid, byte 2 = hi.
    // x . inv + 1.5 . 2^23 rounds x . inv to an integer (|x . inv| < 2^22).
    uint32_t vb[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) vb[t] = __float_as_uint(fmaf(xf[t], inv, 12582912.0f)) - 0x4B400000u + 0x8080u;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
#pragma unroll
      for (int par = 0; par < 2; ++par) {
        const int e = 8 * w + par;  // elements e, e + 2, e + 4, e + 6
        const uint32_t hi01 = __byte_perm(vb[e], vb[e + 2], 0x0062), hi23 = __byte_perm(vb[e + 4], vb[e + 6], 0x0062);
        const uint32_t md01 = __byte_perm(vb[e], vb[e + 2], 0x0051), md23 = __byte_perm(vb[e + 4], vb[e + 6], 0x0051);
        const uint32_t lo01 = __byte_perm(vb[e], vb[e + 2], 0x0040), lo23 = __byte_perm(vb[e + 4], vb[e + 6], 0x0040);
        xp[0][2 * w + par] = __byte_perm(hi01, hi23, 0x5410);
        xp[1][2 * w + par] = __byte_perm(md01, md23, 0x5410) ^ 0x80808080u;
        xp[2][2 * w + par] = __byte_perm(lo01, lo23, 0x5410) ^ 0x80808080u;
      }
    }
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      xsum[0] = dp4a_us(0x01010101u, xp[0][w], xsum[0]);
      xsum[1] = dp4a_us(0x01010101u, xp[1][w], xsum[1]);
      xsum[2] = dp4a_us(0x01010101u, xp[2][w], xsum[2]);
    }
  } else {
#pragma unroll
    for (int w = 0; w < 8; ++w) xp[0][w] = xp[1][w] = xp[2][w] = 0u;
  }
  X.sx = sx;
}

// 32 fp16 activations as floats from four 16-byte words.
__device__ __forceinline__ void gv_unpack_x(const uint4* u, float* xf) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const __half2* h = reinterpret_cast<const __half2*>(&u[w]);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 f = __half22float2(h[t]);
      xf[8 * w + 2 * t] = f.x;
      xf[8 * w + 2 * t + 1] = f.y;
    }
  }
}

// Chunk j of x (when act) read through L2 only, then its planes.
__device__ __forceinline__ void gv_load_x(const __half* x, int j, bool act, GvX& X) {
  float xf[32];
  if (act) {
    const uint4* xg = reinterpret_cast<const uint4*>(x + j * 32);
    uint4 u[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) u[w] = ldg_cg_v4(xg + w);
    gv_unpack_x(u, xf);
  }
  gv_build_planes(xf, act, X);
}

// Chunk j of an x staged in shared memory at xs (when act), then its planes.
__device__ __forceinline__ void gv_load_x_smem(uint32_t xs, int j, bool act, GvX& X) {
  float xf[32];
  if (act) {
    uint4 u[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) u[w] = lds128(xs + j * 64 + w * 16);
    gv_unpack_x(u, xf);
  }
  gv_build_planes(xf, act, X);
}

// Sum over the 32 lanes of each of B row values v[0..B) (B a power of two),
// as a butterfly: at the step with lane mask m = 1, 2, 4, ... a lane keeps
// the half of its values selected by its bit and adds the partner's copy of
// that half; after log2(B) steps lane l holds row bitrev(l mod B) summed
// over its lane group, and the remaining xor steps sum over all 32 lanes.
// Every row's total is the same tree of additions whatever its position in
// the batch.  Returns the row whose total lane `lane` holds in k.
template <int B>
__device__ __forceinline__ int gv_reduce_batch(const float* v, int lane, float& k) {
  float w[B];
#pragma unroll
  for (int b = 0; b < B; ++b) w[b] = v[b];
  int row_sel = 0;
#pragma unroll
  for (int half = B / 2, m = 1; half >= 1; half >>= 1, m <<= 1) {
    const bool hi = (lane & m) != 0;
    row_sel = (row_sel << 1) | (hi ? 1 : 0);
#pragma unroll
    for (int j = 0; j < half; ++j) {
      const float keep = hi ? w[j + half] : w[j];
      const float send = hi ? w[j] : w[j + half];
      w[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  k = w[0];
#pragma unroll
  for (int m = B; m < 32; m <<= 1) k += __shfl_xor_sync(0xffffffffu, k, m);
  return row_sel;
}

}  // namespace gv
}  // namespace qlin
