// Shared device code of the W4A16 tensor-core kernels (a few tokens): the
// exact int4 -> fp16 (q - z) unpack into m16n8k16 A fragments, the matching
// activation pairs for the B fragments, the warp-level MMA, and the cluster
// primitives the split-K reduction uses.
//
// Fragment mapping.  Thread (g, c) = (lane / 4, lane % 4) loads 16 bytes (32
// codes) of rows g and g + 8 at K offset 32c within a 128-code group.  Each
// 32-bit word holds eight consecutive codes k .. k+7; the unpack yields the
// half2 pairs (k, k+4), (k+1, k+5), (k+2, k+6), (k+3, k+7).  These pairs are
// assigned to the MMA's logical K slots (2c, 2c+1) and (2c+8, 2c+9); the
// activation fragment of the same thread is built with exactly the same
// assignment, so the product over a group covers every K index once.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace qlin {
namespace w4mma {

__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b),
                      *reinterpret_cast<__half2*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}

// A pure register operation (not volatile), so that the compiler may
// interleave independent MMAs with each other and with the unpack.
__device__ __forceinline__ void mma_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// half2 constants for the unpack of zero-point z: sub = (1024 + z, 1024 + z)
// and add = (-(64 + z), -(64 + z)), built with integer operations.
__device__ __forceinline__ uint32_t zp_sub(uint32_t z) { return 0x64006400u | (z << 16) | z; }
__device__ __forceinline__ uint32_t zp_add(uint32_t z) { return 0xD400D400u | (z << 20) | (z << 4); }

// (a & b) | c in one three-input logic operation (lookup table 0xEA).  The
// mask and the fp16 exponent are passed in registers: with two immediates
// the compiler splits the operation in two.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// The unpack constants, kept in registers by the caller across a loop.
struct UnpackConsts {
  uint32_t lo, hi, ex;
};
__device__ __forceinline__ UnpackConsts unpack_consts() {
  UnpackConsts k;
  // opaque to constant folding, so that each stays one register
  asm("mov.b32 %0, 0x000F000F;" : "=r"(k.lo));
  asm("mov.b32 %0, 0x00F000F0;" : "=r"(k.hi));
  asm("mov.b32 %0, 0x64006400;" : "=r"(k.ex));
  return k;
}

// Exact fp16 (q - z) pairs from one word of eight codes.
//   out[0] = (k, k+4), out[1] = (k+1, k+5), out[2] = (k+2, k+6), out[3] = (k+3, k+7)
// 0x6400 is fp16 1024: OR-ing a nibble n into its low mantissa bits gives
// 1024 + n, and 1024 + 16n for the nibble one position higher.
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t sub, uint32_t add, const UnpackConsts& k,
                                            uint32_t* out) {
  const uint32_t kSixteenth = 0x2C002C00u;
  out[0] = h2_sub(and_or(w, k.lo, k.ex), sub);                // (1024 + n) - (1024 + z)
  out[1] = h2_fma(and_or(w, k.hi, k.ex), kSixteenth, add);    // (1024 + 16n) / 16 - (64 + z)
  const uint32_t w8 = w >> 8;
  out[2] = h2_sub(and_or(w8, k.lo, k.ex), sub);
  out[3] = h2_fma(and_or(w8, k.hi, k.ex), kSixteenth, add);
}

// Activation pairs (x[k+j], x[k+j+4]) for j = 0..3 from eight consecutive fp16.
__device__ __forceinline__ void pair_x(uint4 u, uint32_t* out) {
  out[0] = __byte_perm(u.x, u.z, 0x5410);
  out[1] = __byte_perm(u.x, u.z, 0x7632);
  out[2] = __byte_perm(u.y, u.w, 0x5410);
  out[3] = __byte_perm(u.y, u.w, 0x7632);
}

// The eight MMAs of one 128-code group for rows g and g + 8 (codes qa, qb
// with zero-point constants), accumulated into two chains p0, p1 per token
// tile; xb[nt][w] holds the activation pairs of word w for token tile nt.
template <int NT>
__device__ __forceinline__ void group_mma(uint4 qa, uint4 qb, uint32_t subA, uint32_t addA, uint32_t subB,
                                          uint32_t addB, const uint4 (*xb)[4], float (*p0)[4], float (*p1)[4],
                                          const UnpackConsts& k) {
  const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
  const uint32_t wb[4] = {qb.x, qb.y, qb.z, qb.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t pa[4], pb[4];
    unpack_word(wa[w], subA, addA, k, pa);
    unpack_word(wb[w], subB, addB, k, pb);
    const uint32_t f0[4] = {pa[0], pb[0], pa[1], pb[1]};
    const uint32_t f1[4] = {pa[2], pb[2], pa[3], pb[3]};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mma_16816(p0[nt], f0, xb[nt][w].x, xb[nt][w].y);
      mma_16816(p1[nt], f1, xb[nt][w].z, xb[nt][w].w);
    }
  }
}

// ---- clusters ----------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// Arrive (release, cluster scope) on an mbarrier given by its shared::cluster
// address, which may belong to another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// One poll (acquire, cluster scope) of a local mbarrier's phase.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

}  // namespace w4mma
}  // namespace qlin
