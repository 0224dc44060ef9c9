// W4A16 with act-order (g_idx): column k of the weights belongs to group
// g_idx[k] ("LLM and AIGC quantization: from number formats to W4A4", GPTQ
// engineering details: desc_act quantizes the columns in descending diag(H)
// order, so the groups no longer follow the column order and the scale reads
// become scattered).
//
// GB300 design: the scattered scale reads are removed once, offline.  The
// columns are put in group order (a stable sort by g_idx, perm), the packed
// codes are rewritten in that order, and the scales and zero-points keep
// their [N][G] layout, now contiguous per group.  At run time only the
// activations are gathered, x'[t][j] = x[t][perm[j]], and the ordinary g128
// kernels run on (x', sorted codes):
//   sum_j x[t, perm[j]] . w[n, perm[j]] = sum_k x[t, k] . w[n, k].
// The gather is HBM-bound (2TK bytes read and written).
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "qlin_internal.h"

namespace qlin {
namespace {

constexpr int kAoThreads = 256;

// One thread per group: the group's columns in ascending order (the stable
// sort).  A group that does not hold exactly `group` columns (g_idx out of
// range or uneven) is recorded in the device error word; its unfilled
// positions are left as they were.
__global__ void act_order_perm_kernel(const int32_t* __restrict__ g_idx, int K, int group, int G,
                                      int32_t* __restrict__ perm, int32_t* __restrict__ err) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= G) return;
  int cnt = 0;
  for (int k = 0; k < K; ++k) {
    if (__ldg(g_idx + k) == g) {
      if (cnt < group) perm[g * group + cnt] = k;
      ++cnt;
    }
  }
  if (cnt != group) record_device_error(err, kDevErrBadIndex);
}

__device__ __forceinline__ uint32_t checked_col(int32_t c, int K, int32_t* err) {
  if (static_cast<uint32_t>(c) >= static_cast<uint32_t>(K)) {
    record_device_error(err, kDevErrBadIndex);
    return static_cast<uint32_t>(K - 1);  // keep the gather in bounds
  }
  return static_cast<uint32_t>(c);
}

// out[n] codes in column order perm: output byte b of row n holds the codes of
// source columns perm[2b] (low nibble) and perm[2b + 1].
__global__ void w4_permute_k_kernel(const uint8_t* __restrict__ wq, int64_t nbytes, int K,
                                    const int32_t* __restrict__ perm, uint8_t* __restrict__ out,
                                    int32_t* __restrict__ err) {
  const int half = K / 2;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nbytes;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = i / half;
    const int b = static_cast<int>(i - n * half);
    const uint8_t* row = wq + n * half;
    const uint32_t k0 = checked_col(__ldg(perm + 2 * b), K, err);
    const uint32_t k1 = checked_col(__ldg(perm + 2 * b + 1), K, err);
    const uint32_t c0 = (__ldg(row + (k0 >> 1)) >> (4 * (k0 & 1))) & 0xFu;
    const uint32_t c1 = (__ldg(row + (k1 >> 1)) >> (4 * (k1 & 1))) & 0xFu;
    out[i] = static_cast<uint8_t>(c0 | (c1 << 4));
  }
}

// x'[t][j] = x[t][perm[j]]: one CTA per row at a time; the row is copied into
// shared memory with 16-byte loads (coalesced), then each thread gathers
// eight elements from it and writes them with one 16-byte store.
__global__ void __launch_bounds__(kAoThreads) x_permute_kernel(const __half* __restrict__ x, int64_t T, int K,
                                                                const int32_t* __restrict__ perm,
                                                                __half* __restrict__ out, int32_t* __restrict__ err) {
  extern __shared__ __align__(16) unsigned short row[];
  // the GEMM that follows may start streaming its weights meanwhile (it waits
  // for this grid before it reads the gathered activations)
  pdl_launch_dependents();
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(x + t * K);
    for (int i = threadIdx.x; i < K / 8; i += kAoThreads) reinterpret_cast<uint4*>(row)[i] = __ldg(src + i);
    __syncthreads();
    for (int j0 = threadIdx.x * 8; j0 < K; j0 += kAoThreads * 8) {
      const int4 p0 = __ldg(reinterpret_cast<const int4*>(perm + j0));
      const int4 p1 = __ldg(reinterpret_cast<const int4*>(perm + j0 + 4));
      const int32_t cols[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = static_cast<uint32_t>(row[checked_col(cols[2 * i], K, err)]) |
               (static_cast<uint32_t>(row[checked_col(cols[2 * i + 1], K, err)]) << 16);
      *reinterpret_cast<uint4*>(out + t * K + j0) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();  // the row buffer is refilled for the next row
  }
}

unsigned grid_for(int64_t items) {
  const int64_t want = (items + kAoThreads - 1) / kAoThreads;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
  return static_cast<unsigned>(want < cap ? want : cap);
}

}  // namespace

cudaError_t launch_w4a16_act_order_prepare(const int32_t* g_idx, int64_t K, int64_t group, const uint8_t* wq,
                                           int64_t N, int32_t* perm, uint8_t* wq_sorted, cudaStream_t stream) {
  const int G = static_cast<int>(K / group);
  act_order_perm_kernel<<<(G + kAoThreads - 1) / kAoThreads, kAoThreads, 0, stream>>>(
      g_idx, static_cast<int>(K), static_cast<int>(group), G, perm, device_error_word());
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || N == 0) return e;
  const int64_t nbytes = N * (K / 2);
  w4_permute_k_kernel<<<grid_for(nbytes), kAoThreads, 0, stream>>>(wq, nbytes, static_cast<int>(K), perm, wq_sorted,
                                                                   device_error_word());
  return cudaGetLastError();
}

cudaError_t launch_x_permute(const void* x, int64_t T, int64_t K, const int32_t* perm, void* out,
                             cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(K) * 2;
  if (smem > 48 * 1024) {
    cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(x_permute_kernel));
    if (e != cudaSuccess) return e;
  }
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  const unsigned grid = static_cast<unsigned>(T < cap ? T : cap);
  x_permute_kernel<<<grid, kAoThreads, smem, stream>>>(static_cast<const __half*>(x), T, static_cast<int>(K), perm,
                                                       static_cast<__half*>(out), device_error_word());
  return cudaGetLastError();
}

}  // namespace qlin
