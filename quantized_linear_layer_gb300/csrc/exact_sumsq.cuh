// Exact sum of squares of one row, rounded once to float32, computed by a CTA.
//
// The fused RMSNorm needs sum_k x_k^2.  No page fixes an order for that sum,
// and float32 additions in different orders round differently, so the sum is
// taken exactly and rounded once (to nearest, ties to even): one result,
// whatever the number of threads or the order in which they add.
//
// Every finite float32 x is m * 2^(max(E,1) - 150), with E its exponent field
// and m < 2^24 an integer (the significand with its implicit bit), so
//   x^2 = m^2 * 2^(pos - 298),   pos = 2 max(E,1) - 2 in [0, 506],
// with m^2 < 2^48.  A square occupies the bit positions [pos, pos + 48) of
// one long integer N whose value is N * 2^-298, and the row's sum is N.
//
// N is built in 32-bit windows of positions: window w holds positions
// [low + 32 w, low + 32 w + 32), where no square of the row has a set bit
// below low.  Each thread adds the window's slice of each of its
// squares into a 64-bit integer; the CTA adds the threads' totals (at most
// 2^31 terms below 2^32 each, so no total overflows); then one warp, a lane
// per window, carries from the lowest window upwards and rounds the integer
// to float32.  Integer
// additions are associative, so the result does not depend on the order.
// A NaN element gives NaN, an infinite one +inf.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

namespace qlin {

constexpr int kExactSqMaxWindows = 18;  // positions 0 .. 554 (the highest bit of a square)

template <int WARPS>
struct ExactSqScratch {
  int top[WARPS];                                        // per warp: largest |x| bit pattern
  int low[WARPS];                                        // per warp: smallest nonzero |x| pattern / 2
  unsigned special[WARPS];                               // per warp (fp16 path): 1 an inf, 2 a NaN
  unsigned long long win[kExactSqMaxWindows][WARPS];     // window totals, per warp
  float result;
};

// m^2 (as hi:lo) and pos of one float32; m == 0 for zeros; special for inf / NaN.
__device__ __forceinline__ void exact_sq_term(float x, uint32_t& m, uint64_t& m2, int& pos, unsigned& special) {
  const uint32_t bits = __float_as_uint(x);
  const uint32_t E = (bits >> 23) & 0xffu, man = bits & 0x7fffffu;
  if (E == 0xffu) {
    special |= man ? 2u : 1u;
    m = 0;
  } else {
    m = E ? (man | 0x800000u) : man;
  }
  m2 = static_cast<uint64_t>(m) * m;
  pos = 2 * static_cast<int>(E > 1u ? E : 1u) - 2;
}

// Bits [L, L + 32) of m2 * 2^pos.
__device__ __forceinline__ uint32_t exact_sq_slice(uint64_t m2, int pos, int L) {
  const int d = pos - L;
  if (d >= 0) return d < 32 ? static_cast<uint32_t>(m2) << d : 0u;
  const int r = -d;  // 1 .. 554
  return r < 64 ? static_cast<uint32_t>(m2 >> r) : 0u;
}

// Warp-level finish: lane w holds window w's total t_w (0 for w >= nw).
// N = sum_w t_w 2^(32 w) is put into 32-bit digits D_w with one carry-
// lookahead step across the lanes, then rounded to float32 (nearest, ties to
// even).  Every lane returns the result.  nw <= 18, so the digits (up to
// nw + 1 of them) fit in the warp.
__device__ __forceinline__ float exact_sq_finish_warp(unsigned long long t, int low) {
  const unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const uint32_t lo = static_cast<uint32_t>(t), hi = static_cast<uint32_t>(t >> 32);
  uint32_t hi_prev = __shfl_up_sync(FULL, hi, 1);
  if (lane == 0) hi_prev = 0;
  const unsigned long long s = static_cast<unsigned long long>(lo) + hi_prev;  // < 2^33
  const uint32_t d = static_cast<uint32_t>(s);
  // carry generated out of lane w (s >= 2^32: then d <= 2^32 - 2, so it does not
  // also propagate), and lanes a carry passes through (d = 2^32 - 1).  With these
  // as bit masks, the carries into every lane are the carries of the binary sum
  // G + (G | P): a G bit always carries out, a P bit passes an incoming carry
  // on, any other bit stops it.
  const unsigned G = __ballot_sync(FULL, (s >> 32) != 0ull);
  const unsigned B = G | __ballot_sync(FULL, d == 0xffffffffu);
  const unsigned C = (G + B) ^ G ^ B;  // bit w: carry into lane w
  const uint32_t D = d + ((C >> lane) & 1u);
  const unsigned nz = __ballot_sync(FULL, D != 0u);
  if (nz == 0u) return 0.0f;
  const int tl = 31 - __clz(static_cast<int>(nz));                // leading digit
  const uint32_t Dt = __shfl_sync(FULL, D, tl);
  const int lead = low + 32 * tl + 31 - __clz(static_cast<int>(Dt));  // absolute position of the leading bit
  const int ulp = max(lead - 23, 149);      // float32 keeps 24 bits, and nothing below 2^-149
  if (lead < ulp - 1) return 0.0f;          // below half the smallest subnormal
  uint32_t q;
  if (ulp <= low) {
    // every bit is at or above the last kept position: exact (N < 2^24)
    q = __shfl_sync(FULL, D, 0) << (low - ulp);
  } else {
    const int rp = ulp - 1 - low;           // relative position of the round bit, >= 0
    const int j0 = rp >> 5, sh = rp & 31;   // j0 <= tl < 32
    const uint32_t d0 = __shfl_sync(FULL, D, j0);
    const uint32_t d1 = __shfl_sync(FULL, D, min(j0 + 1, 31));
    const unsigned long long w = ((static_cast<unsigned long long>(j0 + 1 <= tl ? d1 : 0u) << 32) | d0) >> sh;
    q = static_cast<uint32_t>(w >> 1);      // bits [ulp, lead]: nothing above lead is set
    const bool round_bit = (w & 1ull) != 0ull;
    const bool sticky = (__ballot_sync(FULL, lane < j0 && D != 0u) != 0u) ||
                        (sh != 0 && (d0 & ((1u << sh) - 1u)) != 0u);
    if (round_bit && (sticky || (q & 1u))) ++q;
  }
  // q * 2^(ulp - 298): the float32 with exponent field ulp - 148 and q's low 23
  // bits (q < 2^23 only on the subnormal grid, ulp = 149; q = 2^24 after
  // rounding carries into the exponent field by itself)
  const uint32_t bits = (static_cast<uint32_t>(ulp - 149) << 23) + q;
  return bits >= 0x7f800000u ? __uint_as_float(0x7f800000u) : __uint_as_float(bits);
}

// The exact sum of squares of the elements that for_each(f) passes to f, over
// all WARPS * 32 threads of the CTA (every thread must call this, and the
// call contains block-wide barriers).  Returns the float32 result to every
// thread.  TZ is a number of low bits known to be zero in every m^2: 32 for
// bf16 inputs (8-bit significands), 26 for fp16 inputs, 0 for float32.
//
// The window range comes from the largest and the smallest nonzero |x|
// (their bit patterns order like the values): the largest square ends below
// position pos(max) + 48, and no square has a set bit below pos(min) + TZ.
template <int WARPS, int TZ, class ForEach>
__device__ float exact_sum_squares_cta(ForEach for_each, ExactSqScratch<WARPS>& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t amax = 0, amin = 0xffffffffu;
  for_each([&](float x) {
    const uint32_t a = __float_as_uint(x) & 0x7fffffffu;
    amax = max(amax, a);
    amin = min(amin, a == 0u ? 0xffffffffu : a);
  });
  amax = __reduce_max_sync(0xffffffffu, amax);
  amin = __reduce_min_sync(0xffffffffu, amin);
  if (lane == 0) {
    sh.top[warp] = static_cast<int>(amax);
    sh.low[warp] = static_cast<int>(amin >> 1);  // as a non-negative int (the order is kept)
  }
  __syncthreads();
  amax = static_cast<uint32_t>(sh.top[0]);
  uint32_t amin2 = static_cast<uint32_t>(sh.low[0]);
#pragma unroll
  for (int w = 1; w < WARPS; ++w) {
    amax = max(amax, static_cast<uint32_t>(sh.top[w]));
    amin2 = min(amin2, static_cast<uint32_t>(sh.low[w]));
  }
  amin = amin2 << 1;
  // NaN above the infinity pattern, infinity equal to it
  const unsigned special = amax > 0x7f800000u ? 2u : (amax == 0x7f800000u ? 1u : 0u);
  const auto pos_of = [](uint32_t a) {
    const int E = static_cast<int>(a >> 23);
    return 2 * (E > 1 ? E : 1) - 2;
  };
  const int top = amax == 0u ? -1 : pos_of(amax) + 48;
  const int low = amax == 0u ? 0 : pos_of(amin) + TZ;
  const int nw = (top < 0 || special) ? 0 : (top - low + 31) >> 5;  // uniform over the CTA
  for (int w = 0; w < nw; ++w) {
    const int L = low + 32 * w;
    unsigned long long acc = 0;
    for_each([&](float x) {
      uint32_t m;
      uint64_t m2;
      int pos;
      unsigned sp = 0;
      exact_sq_term(x, m, m2, pos, sp);
      acc += exact_sq_slice(m2, pos, L);
    });
#pragma unroll
    for (int h = 16; h >= 1; h >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, h);
    if (lane == 0) sh.win[w][warp] = acc;
  }
  __syncthreads();
  if (warp == 0) {
    unsigned long long t = 0;
    if (lane < nw) {
#pragma unroll
      for (int i = 0; i < WARPS; ++i) t += sh.win[lane][i];
    }
    float r = exact_sq_finish_warp(t, low);
    if (special & 1u) r = __uint_as_float(0x7f800000u);
    if (special & 2u) r = __uint_as_float(0x7fc00000u);
    if (lane == 0) sh.result = r;
  }
  __syncthreads();
  return sh.result;
}

// The same sum for elements that are fp16 values (converted to float32
// exactly), in one pass and without the range statistics: every fp16 x is
// m * 2^(max(e,1) - 25) with e its 5-bit exponent field and m < 2^11, so
// x^2 = m^2 * 2^(p - 48) with p = 2 max(e,1) - 2 in [0, 58] and m^2 < 2^22:
// all squares are integers times 2^-48 below 2^80, three 32-bit digits.
// Each thread adds each square's two 32-bit pieces into 64-bit digit sums
// (below 2^32 per element, so any row length is exact); the CTA adds the
// threads' digits and one warp finishes as above (position 250 is 2^-48).
// Returns the same float32 as exact_sum_squares_cta.
template <int WARPS, class ForEach>
__device__ float exact_sum_squares_f16_cta(ForEach for_each, ExactSqScratch<WARPS>& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long d[3] = {0, 0, 0};
  unsigned special = 0;
  for_each([&](float x) {
    const uint32_t h = __half_as_ushort(__float2half_rn(x));  // exact: x is an fp16 value
    const uint32_t e = (h >> 10) & 31u, man = h & 1023u;
    if (e == 31u) special |= man ? 2u : 1u;
    const uint32_t m = e == 31u ? 0u : (e ? (man | 1024u) : man);
    const uint32_t p = e > 1u ? 2u * e - 2u : 0u;
    const unsigned long long v = static_cast<unsigned long long>(m * m) << (p & 31u);
    const uint32_t vlo = static_cast<uint32_t>(v), vhi = static_cast<uint32_t>(v >> 32);
    if (p < 32u) {
      d[0] += vlo;
      d[1] += vhi;
    } else {
      d[1] += vlo;
      d[2] += vhi;
    }
  });
#pragma unroll
  for (int i = 0; i < 3; ++i) {
#pragma unroll
    for (int h = 16; h >= 1; h >>= 1) d[i] += __shfl_xor_sync(0xffffffffu, d[i], h);
  }
  special = __reduce_or_sync(0xffffffffu, special);
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < 3; ++i) sh.win[i][warp] = d[i];
    sh.special[warp] = special;
  }
  __syncthreads();
  if (warp == 0) {
    unsigned long long t = 0;
    unsigned sp = 0;
#pragma unroll
    for (int i = 0; i < WARPS; ++i) sp |= sh.special[i];
    if (lane < 3) {
#pragma unroll
      for (int i = 0; i < WARPS; ++i) t += sh.win[lane][i];
    }
    float r = exact_sq_finish_warp(t, 250);
    if (sp & 1u) r = __uint_as_float(0x7f800000u);
    if (sp & 2u) r = __uint_as_float(0x7fc00000u);
    if (lane == 0) sh.result = r;
  }
  __syncthreads();
  return sh.result;
}

}  // namespace qlin
