// W4A16 decode GEMV (one token) on the CUDA cores.
//
//   y[n] = sum_g s[n,g] . sum_{k in g} x[k] . (q[n,k] - z[n,g])
//
// ("Chapter 9 - Quantization kernels", 9.5 dequantize right before the
// multiply, weights stay 4-bit in HBM and shared memory; 9.6 the magic-number
// unpack; "LLM and AIGC quantization", W4A16 section.)
//
// Why not the tensor core at T = 1.  A warp-level m16n8k16 MMA with the
// token as the N side spends 7/8 of its work on padding; on this GPU that
// caps a decode GEMV below the HBM rate.  One token needs one multiply-add
// per weight, which the CUDA cores' 4-way byte dot product (dp4a) does with
// far fewer instructions per code than any float unpack.
//
// Integer dot products.  Each thread rounds its 32 activations once to fixed
// point with a per-chunk scale s_x = max|x| / (127 . 2^15) and writes the
// result in base-256 signed digits, x_fix = 2^16 hi + 2^8 mid + lo, as three
// byte planes.  Two AND masks turn a word of eight codes into the bytes of its
// even and odd codes, and one dp4a per plane and parity gives
// sum (n - z) . plane exactly in int32 (the zero-point enters once per chunk
// as z . sum(plane)).  The plane sums are combined and scaled by s_g . s_x in
// fp32.  Every x is represented within 0.75 s_x = 2^-22.4 of its chunk's
// largest |x|, finer than fp16 itself for every element above
// max|x| . 2^-11, however the magnitudes within the chunk are spread.
//
// Data path for GB300.  One CTA per SM owns a contiguous band of weight rows;
// the band is contiguous in HBM, so a single elected thread streams it into a
// ring of shared-memory stages with 1-D bulk copies (no per-thread load
// instructions).  The ring is filled before the kernel waits on the previous
// kernel in the stream (programmatic dependent launch): the weights do not
// depend on it, so one layer's weights stream in while the previous layer is
// still finishing, and HBM sees no gap at the layer boundary.  The CTA uses
// less than half of an SM, so the next layer's CTA fits beside it.
//
// Work split.  Thread j of a row owns the 32-code chunk j of every row (its
// 32 activations live in registers for the whole kernel); a row's chunks are
// spread over the warps of one row group, the CTA's rows over its row groups.
// Per row a warp adds its lanes' partial sums with shuffles; the warps' sums
// meet in shared memory and are added in a fixed order at the end.
//
// Grouped launch.  Several weight matrices applied to the same activations
// (the q, k and v projections of a decoder block, or gate and up) run as one
// launch over their concatenated rows: the bands simply continue from one
// matrix into the next, a stage that straddles a boundary is filled by one
// bulk copy per matrix, and the matrices share a single wait on the kernel
// that produced the activations.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "device_common.cuh"
#include "qlin_internal.h"
#include "tc_common.cuh"
#include "w4a16_gemv_common.cuh"

namespace qlin {
namespace {

using namespace gv;

constexpr int kGvMaxWarpsPerRow = 12;       // K <= 12 * 32 * 32 = 12288
constexpr int kGvMaxComputeWarps = 12;
constexpr int kGvThreadsMax = (kGvMaxComputeWarps + 1) * 32;
constexpr int kGvCtaBytes = 112 * 1024;     // two CTAs (this layer, the next) fit on one SM
constexpr int kGvMaxRegs = 72;              // registers per thread (fixed: the launch plan counts them)
constexpr int kGvL2Ahead = 2;               // stages of L2 prefetch ahead of the copy into the ring
constexpr int kGvMinStages = 2;
constexpr int kGvMaxStages = 8;
constexpr int kGvSiteFull = 1, kGvSiteEmpty = 2, kGvSiteDrain = 3;
constexpr int kGvMaxGroup = QLIN_W4A16_MAX_GROUP;
constexpr int64_t kMaxGemvRows = int64_t(1) << 30;  // launch rows are ints

struct GvArgs {
  const __half* x;
  // matrix p covers rows [row_end[p-1], row_end[p]) of the launch
  const uint8_t* wq[kGvMaxGroup];
  const __half* scales[kGvMaxGroup];
  const uint8_t* zeros[kGvMaxGroup];
  __half* y[kGvMaxGroup];
  int row_end[kGvMaxGroup];
  int np;
  int32_t* err;
  int N, K, zpitch;
  int WPR, RG;                 // warps per row, row groups
  int R, S, stage_bytes;       // rows per stage, stages
  int off_sz, off_red, off_raw_s, off_raw_z, off_bar;
};

// Matrix of launch row r, and the first launch row of that matrix.
__device__ __forceinline__ int gv_matrix(const GvArgs& a, int r, int& first) {
  int p = 0;
#pragma unroll
  for (int i = 0; i < kGvMaxGroup - 1; ++i)
    if (i < a.np - 1 && r >= a.row_end[i]) p = i + 1;
  first = p > 0 ? a.row_end[p - 1] : 0;
  return p;
}

// The band's scales and zero-points are staged raw in shared memory, one
// bulk copy per matrix segment and array.  A copy starts at the 16-byte
// boundary below its first byte and ends at the one above its last (the
// copied window never leaves the 16-byte blocks holding the segment), and
// each segment's window starts 16-byte aligned in the staging area.
struct GvSeg {
  int row0, rows;         // band rows [row0, row0 + rows) (relative to the band)
  int sc_off, z_off;      // staging offsets of the segment's first scale / zero byte
  const char* sc_lo;      // copy windows (16-byte aligned)
  uint32_t sc_bytes;
  const char* z_lo;
  uint32_t z_bytes;
};

// Segment `k` of the band [r0, r0 + nrows), in band order; false past the last.
__device__ __forceinline__ bool gv_segment(const GvArgs& a, int r0, int nrows, int G, int k, GvSeg& sg) {
  int done = 0, sc_off = 0, z_off = 0;
  for (int i = 0; done < nrows; ++i) {
    const int r = r0 + done;
    int first;
    const int p = gv_matrix(a, r, first);
    const int seg = min(nrows - done, a.row_end[p] - r);
    const char* sc = reinterpret_cast<const char*>(a.scales[p] + static_cast<int64_t>(r - first) * G);
    const char* sc_lo = reinterpret_cast<const char*>(reinterpret_cast<uintptr_t>(sc) & ~uintptr_t(15));
    const uint32_t sc_bytes = static_cast<uint32_t>(
        ((reinterpret_cast<uintptr_t>(sc) + static_cast<uintptr_t>(seg) * G * 2 + 15) & ~uintptr_t(15)) -
        reinterpret_cast<uintptr_t>(sc_lo));
    const char* z_lo = nullptr;
    uint32_t z_bytes = 0;
    int z_delta = 0;
    if (a.zeros[p]) {
      const char* z = reinterpret_cast<const char*>(a.zeros[p] + static_cast<int64_t>(r - first) * a.zpitch);
      z_lo = reinterpret_cast<const char*>(reinterpret_cast<uintptr_t>(z) & ~uintptr_t(15));
      z_bytes = static_cast<uint32_t>(
          ((reinterpret_cast<uintptr_t>(z) + static_cast<uintptr_t>(seg) * a.zpitch + 15) & ~uintptr_t(15)) -
          reinterpret_cast<uintptr_t>(z_lo));
      z_delta = static_cast<int>(z - z_lo);
    }
    if (i == k) {
      sg.row0 = done;
      sg.rows = seg;
      sg.sc_off = sc_off + static_cast<int>(sc - sc_lo);
      sg.z_off = a.zeros[p] ? z_off + z_delta : -1;
      sg.sc_lo = sc_lo;
      sg.sc_bytes = sc_bytes;
      sg.z_lo = z_lo;
      sg.z_bytes = z_bytes;
      return true;
    }
    sc_off += static_cast<int>(sc_bytes);
    z_off += static_cast<int>(z_bytes);
    done += seg;
  }
  return false;
}


// B rows of each stage per warp and row group (a power of two).  Warps past
// the producer (ballast of the alternate launch shape) leave at once.
template <int B>
__global__ void __maxnreg__(kGvMaxRegs) w4a16_gemv_kernel(const GvArgs a) {
  constexpr int kGvRowsPerBatch = B;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ncw = a.RG * a.WPR;  // compute warps; warp ncw is the producer
  const int G = a.K >> 7, KC = a.K >> 5, row_bytes = a.K >> 1;
  const int base = a.N / gridDim.x, extra = a.N % gridDim.x;
  const int r0 = blockIdx.x * base + min(static_cast<int>(blockIdx.x), extra);
  const int nrows = base + (static_cast<int>(blockIdx.x) < extra ? 1 : 0);
  const int nloads = (nrows + a.R - 1) / a.R;
  const int S = a.S;
  uint32_t* sz = reinterpret_cast<uint32_t*>(smem + a.off_sz);  // per (row, group): fp16 s | z << 16
  float* red = reinterpret_cast<float*>(smem + a.off_red);
  const uint32_t ring = tc::smem_u32(smem);
  const uint32_t bar0 = tc::smem_u32(smem + a.off_bar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + a.off_bar + 16 * S);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (S + s); };
  const uint32_t meta_full = bar0 + 16u * S + 8u;  // the band's raw scales and zero-points

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(full(s), 1);
      tc::mbar_init(empty(s), ncw);
    }
    tc::mbar_init(meta_full, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  if (warp > ncw) return;

  if (warp == ncw) {
    // ---------------- producer: the CTA's band of weight rows ----------------
    if (lane == 0) {
      const uint64_t policy = tc::l2_policy_evict_first();
      // scales and zero-points first: the compute warps convert them while
      // the weight rows stream
      {
        uint32_t meta_bytes = 0;
        GvSeg sg;
        for (int k = 0; gv_segment(a, r0, nrows, G, k, sg); ++k) meta_bytes += sg.sc_bytes + sg.z_bytes;
        tc::mbar_arrive_expect_tx(meta_full, meta_bytes);
        const uint32_t raw_s = tc::smem_u32(smem + a.off_raw_s), raw_z = tc::smem_u32(smem + a.off_raw_z);
        uint32_t so = 0, zo = 0;
        for (int k = 0; gv_segment(a, r0, nrows, G, k, sg); ++k) {
          tc::bulk_load(raw_s + so, sg.sc_lo, sg.sc_bytes, meta_full);
          so += sg.sc_bytes;
          if (sg.z_bytes) tc::bulk_load(raw_z + zo, sg.z_lo, sg.z_bytes, meta_full);
          zo += sg.z_bytes;
        }
      }
      int i = 0;
      for (; i < nloads; ++i) {
        const int s = i % S;
        if (i >= S && !tc::mbar_wait_sleep(empty(s), ((i / S) - 1) & 1, a.err, kGvSiteEmpty, 128)) {
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        const int rows_i = min(a.R, nrows - i * a.R);
        // the rows kGvL2Ahead stages ahead, into L2 only: more bytes in
        // flight than the ring holds, so the copy into the ring later hits L2
        const int ia = i + kGvL2Ahead;
        if (ia < nloads) {
          const int rl = r0 + ia * a.R, nl = min(a.R, nrows - ia * a.R);
          for (int done = 0; done < nl;) {
            int first;
            const int p = gv_matrix(a, rl + done, first);
            const int seg = min(nl - done, a.row_end[p] - (rl + done));
            tc::bulk_prefetch_l2(a.wq[p] + static_cast<int64_t>(rl + done - first) * row_bytes,
                                 static_cast<uint32_t>(seg * row_bytes));
            done += seg;
          }
        }
        tc::mbar_arrive_expect_tx(full(s), static_cast<uint32_t>(rows_i * row_bytes));
        // one bulk copy per matrix the stage's rows fall in
        for (int done = 0; done < rows_i;) {
          const int r = r0 + i * a.R + done;
          int first;
          const int p = gv_matrix(a, r, first);
          const int seg = min(rows_i - done, a.row_end[p] - r);
          tc::bulk_load_policy(ring + s * a.stage_bytes + done * row_bytes,
                               a.wq[p] + static_cast<int64_t>(r - first) * row_bytes,
                               static_cast<uint32_t>(seg * row_bytes), full(s), policy);
          done += seg;
        }
      }
      // The last copy into each stage must have landed before the CTA exits.
      for (int j = max(0, i - S); j < i; ++j) tc::mbar_wait(full(j % S), (j / S) & 1, a.err, kGvSiteDrain);
      tc::mbar_wait(meta_full, 0, a.err, kGvSiteDrain);
    }
    return;
  }

  // ---------------- compute warps ----------------
  const int nct = ncw * 32;
  // Scales and zero-points of the band (weights, so converted before waiting
  // on the previous kernel) from their raw staging copies into packed pairs.
  {
    bool ok = tc::mbar_wait(meta_full, 0, a.err, kGvSiteFull);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) *abort_flag = 1;
    const unsigned char* raw_s = smem + a.off_raw_s;
    const unsigned char* raw_z = smem + a.off_raw_z;
    GvSeg sg;
    for (int k = 0; ok && gv_segment(a, r0, nrows, G, k, sg); ++k) {
      const int ne = sg.rows * G;
      for (int e = threadIdx.x; e < ne; e += nct) {
        const int r = e / G, g = e - r * G;
        const uint32_t sv = *reinterpret_cast<const unsigned short*>(raw_s + sg.sc_off + 2 * e);
        const uint32_t zv = sg.z_off >= 0 ? (raw_z[sg.z_off + r * a.zpitch + (g >> 1)] >> ((g & 1) * 4)) & 0xFu : 8u;
        sz[(sg.row0 + r) * G + g] = sv | (zv << 16);
      }
    }
  }
  const int rg = warp / a.WPR, wr = warp - rg * a.WPR;
  const int j = wr * 32 + lane;  // this thread's chunk
  const bool act = j < KC;
  const int jc = min(j, KC - 1);  // in-bounds chunk for the idle lanes of the last warp

  // The activations may come from the previous kernel: one warp waits for it,
  // the others block on the named barrier (which also publishes the scales
  // and zero-points) instead of polling.  They are read through L2 only: an
  // L1 line filled while the previous kernel was still running could be stale.
  if (warp == 0) pdl_wait();
  named_sync(1, nct);
  GvX X;
  gv_load_x(a.x, j, act, X);
  const uint32_t (*xp)[8] = X.xp;
  const int* xsum = X.xsum;
  const float sx = X.sx;

  const uint32_t sz_base = tc::smem_u32(sz + (jc >> 2));  // this thread's group column
  {
    // The reduction of one batch runs in the same block as the dot products
    // of the next, so that the shuffles' latency overlaps the dp4a work.
    float prev[kGvRowsPerBatch];
#pragma unroll
    for (int b = 0; b < kGvRowsPerBatch; ++b) prev[b] = 0.0f;
    int prev_row0 = -1, prev_rows = 0;
    auto reduce_store = [&](const float* v, int row0, int rows) {
      float k;
      const int row_sel = gv_reduce_batch<kGvRowsPerBatch>(v, lane, k);
      if (lane < kGvRowsPerBatch) {
        const int rr = rg + a.RG * row_sel;
        if (rr < rows) red[(row0 + rr) * a.WPR + wr] = k;
      }
    };
    int s = 0;            // ring position and phase of stage i, kept
    uint32_t phase = 0;   // incrementally (no division by S in the loop)
    for (int i = 0; i < nloads; ++i) {
      bool ok = tc::mbar_wait(full(s), phase, a.err, kGvSiteFull);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      const int rows_i = min(a.R, nrows - i * a.R);
      float p[kGvRowsPerBatch];
      gv_batch<B>(ring + s * a.stage_bytes + jc * 16, sz_base + (i * a.R * G) * 4, rows_i, a.RG, rg, row_bytes, G, xp,
                  xsum, sx, p);
      // The stage's codes are in registers: hand it back to the producer.
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(empty(s));
      if (++s == S) {
        s = 0;
        phase ^= 1u;
      }
      if (prev_row0 >= 0) reduce_store(prev, prev_row0, prev_rows);
#pragma unroll
      for (int b = 0; b < kGvRowsPerBatch; ++b) prev[b] = p[b];
      prev_row0 = i * a.R;
      prev_rows = rows_i;
    }
    if (prev_row0 >= 0) reduce_store(prev, prev_row0, prev_rows);
  }
  named_sync(1, nct);
  if (*abort_flag) return;
  for (int r = threadIdx.x; r < nrows; r += nct) {
    float v = 0.0f;
    for (int w = 0; w < a.WPR; ++w) v += red[r * a.WPR + w];
    int first;
    const int p = gv_matrix(a, r0 + r, first);
    a.y[p][r0 + r - first] = __float2half_rn(v);
  }
}

__host__ __device__ constexpr int gv_rows_per_batch(int RG) { return RG >= 2 ? 8 : 4; }

// Shared-memory plan of one launch; false when the band's scales do not
// leave room for a double-buffered ring within the per-CTA budget.
bool gv_plan(int64_t N, int64_t K, GvArgs& a, int& grid, int& smem, int warps = 8) {
  if (K > static_cast<int64_t>(kGvMaxWarpsPerRow) * 32 * 32 || N <= 0) return false;
  const int G = static_cast<int>(K / 128), KC = static_cast<int>(K / 32), row_bytes = static_cast<int>(K / 2);
  a.WPR = (KC + 31) / 32;
  a.RG = a.WPR >= warps ? 1 : warps / a.WPR;
  grid = static_cast<int>(std::min<int64_t>(sm_count(), (N + a.RG - 1) / a.RG));
  const int rows_max = static_cast<int>((N + grid - 1) / grid);
  // A stage holds one batch of rows for every row group: 8 rows per warp
  // when there are several row groups, 4 when one (long rows, large stages).
  a.R = std::min(gv_rows_per_batch(a.RG) * a.RG, rows_max);
  a.stage_bytes = a.R * row_bytes;
  auto up = [](int v, int m) { return (v + m - 1) / m * m; };
  const int zpitch = (G + 1) / 2;
  // raw staging: the band's bytes plus up to 32 bytes of alignment window per segment
  const int raw_s_bytes = up(rows_max * G * 2, 16) + 32 * kGvMaxGroup;
  const int raw_z_bytes = up(rows_max * zpitch, 16) + 32 * kGvMaxGroup;
  const int extras = up(rows_max * G * 4, 16) + up(rows_max * a.WPR * 4, 16) + raw_s_bytes + raw_z_bytes +
                     16 * kGvMaxStages + 16 + 128;
  const int loads_max = (rows_max + a.R - 1) / a.R;
  a.S = std::min({kGvMaxStages, (kGvCtaBytes - extras) / a.stage_bytes, loads_max});
  if (a.S < std::min(kGvMinStages, loads_max)) return false;
  a.off_sz = up(a.S * a.stage_bytes, 128);
  a.off_red = a.off_sz + up(rows_max * G * 4, 16);
  a.off_raw_s = a.off_red + up(rows_max * a.WPR * 4, 16);
  a.off_raw_z = a.off_raw_s + raw_s_bytes;
  a.off_bar = a.off_raw_z + raw_z_bytes;
  smem = a.off_bar + 16 * a.S + 16;
  return true;
}

// Launch shapes of consecutive GEMVs.  With programmatic dependent launch the
// next layer's CTAs take whatever SM slots free up while the current layer
// runs, and the block scheduler then puts two CTAs of one layer on some SMs
// and none on others, layer after layer (measured: 100 of 152 SMs per layer).
// Launches alternate between two shapes of the same kernel instead: shape R
// holds more than half of an SM's registers (idle ballast warps on top of the
// working ones), shape S more than half of its shared memory; two CTAs of one
// shape never share an SM, one of each does.  Each layer therefore lands one
// CTA per SM, beside one CTA of its neighbour.  (Twelve working warps in
// shape R instead of ballast measured the same.)
// The shapes come from the device's limits and the kernel's register count;
// when they cannot be met every launch keeps the plain shape.
struct GvShapeInfo {
  bool ok = false;
  int regs_per_warp = 0, rf = 0, sm_smem = 0, reserved = 0, block_smem = 0;
};

const GvShapeInfo& gv_shape_info() {
  static GvShapeInfo info;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaFuncAttributes f8 = {}, f4 = {};
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaFuncGetAttributes(&f8, reinterpret_cast<const void*>(w4a16_gemv_kernel<8>)) != cudaSuccess ||
        cudaFuncGetAttributes(&f4, reinterpret_cast<const void*>(w4a16_gemv_kernel<4>)) != cudaSuccess)
      return;
    const int regs = std::max(f8.numRegs, f4.numRegs);
    cudaDeviceGetAttribute(&info.rf, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&info.sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&info.reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    cudaDeviceGetAttribute(&info.block_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    info.regs_per_warp = 32 * ((regs + 7) / 8 * 8);
    info.ok = regs <= kGvMaxRegs && info.rf > 0 && info.sm_smem > 0 &&
              kGvCtaBytes + info.reserved <= info.sm_smem / 2;
  });
  return info;
}

// The shared memory of a shape-S CTA: more than half of the SM's.
int gv_smem_shape_s(const GvShapeInfo& si) { return si.sm_smem / 2 - si.reserved + 16; }

// The warps of a shape-R CTA with `warps` working warps: enough to hold more
// than half of the SM's registers; 0 when that leaves no room for the largest
// shape-S CTA (kGvMaxComputeWarps + 1 warps) beside it.
int gv_warps_shape_r(const GvShapeInfo& si, int warps) {
  int w = warps;
  while (2 * w * si.regs_per_warp <= si.rf) ++w;
  return (w + kGvMaxComputeWarps + 1) * si.regs_per_warp <= si.rf ? w : 0;
}

// Both kernels' attributes, once per device: dynamic shared memory up to the
// per-block maximum (each launch asks for its own amount), and the largest
// shared-memory carveout, so that the SM can hold a CTA and the neighbouring
// layer's whatever launch shape reached it first.
struct GvAttrs {
  std::once_flag once;
  cudaError_t status = cudaSuccess;
};
GvAttrs g_gv_attrs[64];

cudaError_t gv_set_attrs() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  GvAttrs& g = g_gv_attrs[dev];
  std::call_once(g.once, [&] {
    int block_smem = 0;
    g.status = cudaDeviceGetAttribute(&block_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const void* fns[2] = {reinterpret_cast<const void*>(w4a16_gemv_kernel<8>),
                          reinterpret_cast<const void*>(w4a16_gemv_kernel<4>)};
    for (const void* fn : fns) {
      if (g.status == cudaSuccess)
        g.status = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, block_smem);
      if (g.status == cudaSuccess)
        g.status = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                        cudaSharedmemCarveoutMaxShared);
    }
  });
  return g.status;
}

}  // namespace

bool w4a16_gemv_supported(int64_t T, int64_t N, int64_t K) {
  GvArgs a = {};
  int grid = 0, smem = 0;
  return T == 1 && N <= kMaxGemvRows && gv_plan(N, K, a, grid, smem);
}

cudaError_t launch_w4a16_gemv_grouped(const void* x, int64_t K, int count, const int64_t* N,
                                      const uint8_t* const* wq, const void* const* scales,
                                      const uint8_t* const* zeros, void* const* y, cudaStream_t stream) {
  if (count < 1 || count > kGvMaxGroup) return cudaErrorInvalidValue;
  GvArgs a = {};
  int64_t total = 0;
  a.np = 0;
  for (int p = 0; p < count; ++p) {
    if (N[p] == 0) continue;  // an empty matrix takes no rows
    total += N[p];
    a.wq[a.np] = wq[p];
    a.scales[a.np] = static_cast<const __half*>(scales[p]);
    a.zeros[a.np] = zeros[p];
    a.y[a.np] = static_cast<__half*>(y[p]);
    a.row_end[a.np] = static_cast<int>(total);
    ++a.np;
  }
  if (total == 0) return cudaSuccess;
  if (total > kMaxGemvRows) return cudaErrorInvalidValue;
  // launch shape: 0 plain, 1 register-heavy, 2 shared-memory-heavy
  static std::atomic<unsigned> parity{0};
  const GvShapeInfo& si = gv_shape_info();
  int shape = si.ok ? 1 + static_cast<int>(parity.fetch_add(1, std::memory_order_relaxed) & 1u) : 0;
  int grid = 0, smem = 0;
  if (!gv_plan(total, K, a, grid, smem)) return cudaErrorInvalidValue;
  a.x = static_cast<const __half*>(x);
  a.err = device_error_word();
  a.N = static_cast<int>(total);
  a.K = static_cast<int>(K);
  a.zpitch = static_cast<int>((K / 128 + 1) / 2);
  const bool b8 = gv_rows_per_batch(a.RG) == 8;
  int threads = (a.RG * a.WPR + 1) * 32;
  int dyn = smem;
  if (shape == 1) {
    const int w = gv_warps_shape_r(si, threads / 32);
    if (w > 0) threads = w * 32;
  } else if (shape == 2) {
    dyn = std::max(smem, gv_smem_shape_s(si));
    if (dyn > si.block_smem) dyn = smem;
  }
  const cudaError_t e = gv_set_attrs();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return b8 ? cudaLaunchKernelEx(&cfg, w4a16_gemv_kernel<8>, a) : cudaLaunchKernelEx(&cfg, w4a16_gemv_kernel<4>, a);
}

cudaError_t w4a16_gemv_launch_info(int* alternating, int* registers) {
  const GvShapeInfo& si = gv_shape_info();
  if (alternating) *alternating = si.ok ? 1 : 0;
  if (registers) {
    cudaFuncAttributes f8 = {}, f4 = {};
    cudaError_t e = cudaFuncGetAttributes(&f8, reinterpret_cast<const void*>(w4a16_gemv_kernel<8>));
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&f4, reinterpret_cast<const void*>(w4a16_gemv_kernel<4>));
    if (e != cudaSuccess) return e;
    *registers = std::max(f8.numRegs, f4.numRegs);
  }
  return cudaSuccess;
}

cudaError_t launch_w4a16_gemv(const void* x, int64_t N, int64_t K, const uint8_t* wq, const void* scales,
                              const uint8_t* zeros, void* y, cudaStream_t stream) {
  if (N == 0) return cudaSuccess;
  return launch_w4a16_gemv_grouped(x, K, 1, &N, &wq, &scales, &zeros, &y, stream);
}

}  // namespace qlin
