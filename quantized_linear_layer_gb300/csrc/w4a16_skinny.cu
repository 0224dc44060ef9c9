// W4A16 skinny GEMM for a few tokens (T <= 16) on the warp-level tensor core,
// with the weights streamed through a shared-memory ring of bulk copies.
//
//   Y[t,n] = sum_g s[n,g] . sum_{k in g} X[t,k] . (q[n,k] - z[n,g])
//
// ("Chapter 9 - Quantization kernels", 9.5: dequantize in registers right
// before the tensor core, HBM and SMEM only ever hold the 4-bit codes; 9.6:
// the magic-number unpack; 9.7: the multi-token decode GEMM, with the weight
// rows as the MMA's M side and the tokens as its N side; "LLM and AIGC
// quantization", W4A16 section.)
//
// What bounds it.  A few tokens still read every weight byte once, but at T
// > 1 the exact unpack (two bit operations and one half2 op per pair of
// codes) plus the MMAs cost more issue slots per byte than the one-token
// dp4a GEMV, so the kernel is bound by instruction issue of its compute
// warps as much as by HBM; the activations (T . K . 2 bytes per CTA, read
// from L2) cost about as much per byte on their way into the SM as weights
// from HBM.  K is split over a cluster of C CTAs only when one CTA cannot
// hold a warp per group of its K range (the smallest C in {1, 2, 4} with a
// launch plan; measured faster than larger C, which mostly adds stages per
// CTA).  The split depends on T and K alone, so every output element is the
// same sum in the same order whatever N is and however matrices are grouped.
//
// Data path.  Warp W (the producer) stages the band's raw scales and
// zero-points with 1-D bulk copies, then loads the band's rows restricted to
// the CTA's K range into a ring of 16-row stages, one 2-D TMA box (16 rows x
// Gc groups, 8-byte elements) per stage; a 1-D copy per row would cost a
// TMA issue slot per row (about 50 ns each, measured), far more than the
// bytes.  A band's stages never cross a matrix of a grouped launch; a short
// stage's box ends at its last row and repeats earlier rows, which the
// compute ignores.  Each compute warp owns one or two consecutive 128-code
// groups of the K range and holds their activations in registers for the
// whole kernel, already in the layout of the MMA's B fragments; per stage it
// turns its codes of the 16 rows into exact fp16 (q - z) A fragments and runs
// the m16n8k16 MMAs, accumulating each group in fp32 before scaling it by
// s[n,g], then writes its partial sums into a slot of a reduction ring and
// moves on (one row of token sums per float2 store, tokens contiguous).  Warp
// W + 1 (the reducer) adds the warps' sums of each stage, four tokens per
// load, the even and the odd warps each in warp order and then the two
// chains; with a cluster it sends them into the shared memory of the
// rank that owns the stage (stage i: rank i mod C), and once the band is
// done every rank adds the C sums of its stages in rank order.  So every
// output element is the same sum in the same order on every run, and no CTA
// reads another CTA's memory (each leaves only after every sum meant for it
// has arrived).
#include <algorithm>
#include <mutex>

#include "device_common.cuh"
#include "qlin_internal.h"
#include "tc_common.cuh"
#include "tmap.h"
#include "w4a16_mma_common.cuh"

namespace qlin {
namespace {

using namespace w4mma;

constexpr int kSkMaxGroup = QLIN_W4A16_MAX_GROUP;
constexpr int kSkTile = 16;           // rows per stage: one MMA tile
// compute warps (plus the producer and the reducer): 16 with one token tile
// (576 threads, 113 registers each), 14 with two (512 threads, 128 registers)
__host__ __device__ constexpr int sk_max_warps(int NT) { return NT == 1 ? 16 : 14; }
// Floats per (warp, row) of a reduction slot: the row's NT x 8 token sums,
// padded so that the compute warps' float2 stores hit distinct banks within
// each half warp.
__host__ __device__ constexpr int sk_red_pitch(int NT) { return NT == 1 ? 8 : 24; }
constexpr int kSkMinStages = 2, kSkMaxStages = 8;
constexpr int kSkSiteFull = 1, kSkSiteEmpty = 2, kSkSiteDrain = 3, kSkSiteReady = 4, kSkSiteMeta = 5,
              kSkSiteRedFull = 6, kSkSiteRedEmpty = 7;
constexpr int kSkBandBudget = 64 * 1024;  // per-CTA staged scales and received sums of one band
constexpr int kSkMaxTokens = 16;
constexpr int kSkMaxBoxGroups = 32;    // 256 elements of 8 bytes: the widest TMA box row
constexpr int kSkMaxGpw = 2;           // groups of K per compute warp

struct SkArgs {
  // per matrix: rows x (K / 16) 8-byte elements, boxes of 16 rows x 8 Gcmax
  CUtensorMap tm[kSkMaxGroup];
  const __half* x;
  // matrix p covers rows [row_end[p-1], row_end[p]) of the launch
  const uint8_t* wq[kSkMaxGroup];
  const __half* scales[kSkMaxGroup];
  const uint8_t* zeros[kSkMaxGroup];
  __half* y[kSkMaxGroup];
  int row_end[kSkMaxGroup];
  int np;
  int32_t* err;
  int T, N, K, zpitch;
  int C, NC, NU;                 // CTAs per cluster, clusters, bands
  int W, S, RS;                  // compute warps, ring stages, reduction slots
  int pitch, stage_bytes;        // ring: stages of 16 rows x pitch bytes
  int slots, recv_bufs;          // stages a rank owns per band; band buffers
  int off_raw_s, off_raw_z, off_red, off_recv, off_seg, off_bar;
};

// Matrix of launch row r, and the first launch row of that matrix.
__device__ __forceinline__ int sk_matrix(const SkArgs& a, int r, int& first) {
  int p = 0;
#pragma unroll
  for (int i = 0; i < kSkMaxGroup - 1; ++i)
    if (i < a.np - 1 && r >= a.row_end[i]) p = i + 1;
  first = p > 0 ? a.row_end[p - 1] : 0;
  return p;
}

// Rows [r0, r0 + n) of band u (bands split the N rows evenly).
__device__ __forceinline__ void sk_band(const SkArgs& a, int u, int& r0, int& n) {
  const int base = a.N / a.NU, extra = a.N % a.NU;
  r0 = u * base + min(u, extra);
  n = base + (u < extra ? 1 : 0);
}

// The stages of a band: each matrix segment of the band in 16-row stages, a
// segment's last stage possibly shorter.  A stage's box always holds 16 rows
// and ends at the stage's last row, so a short stage also loads rows before
// its first one (the previous stage's, or rows outside the band) and uses
// rows [16 - rows, 16) of the box.  `cur` is the band-local first row of the
// stage; returns its row count and the matrix.
__device__ __forceinline__ int sk_stage(const SkArgs& a, int ur0, int un, int cur, int& p, int& mfirst) {
  p = sk_matrix(a, ur0 + cur, mfirst);
  const int seg_end = min(un, a.row_end[p] - ur0);
  return min(kSkTile, seg_end - cur);
}

// The band's scales and zero-points are staged raw in shared memory, one
// bulk copy per matrix segment and array, each copy widened to the 16-byte
// blocks that hold the segment (so it never leaves them).
struct SkSeg {
  int row0;             // band-local first row of the segment
  int sc_off, z_off;    // staging offsets of the segment's first scale / zero byte (z_off -1: symmetric)
  const char* sc_lo;
  uint32_t sc_bytes;
  const char* z_lo;
  uint32_t z_bytes;
};

// Segment k of the band [r0, r0 + nrows); false past the last.
__device__ __forceinline__ bool sk_segment(const SkArgs& a, int r0, int nrows, int G, int k, SkSeg& sg) {
  int done = 0, sc_off = 0, z_off = 0;
  for (int i = 0; done < nrows; ++i) {
    const int r = r0 + done;
    int first;
    const int p = sk_matrix(a, r, first);
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

// Bounded wait (acquire, cluster scope) on a local mbarrier.
__device__ __forceinline__ bool sk_wait_cluster(uint32_t bar, uint32_t parity, int32_t* err, int site) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (clock64() - t0 > tc::kWaitTimeoutCycles) {
      record_device_error(err, kDevErrTimeoutBase + site);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// NT token tiles of 8 (T <= 8 NT); GPW groups of K per compute warp.
// Warps 0 .. W-1 compute, warp W produces (TMA), warp W + 1 reduces.
template <int NT, int GPW>
__global__ void __launch_bounds__((sk_max_warps(NT) + 2) * 32, 1) w4a16_skinny_kernel(const __grid_constant__ SkArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = a.W, C = a.C, S = a.S, RS = a.RS;
  const int rank = C > 1 ? static_cast<int>(cluster_rank()) : 0;
  const int cl = blockIdx.x / C;
  const int G = a.K >> 7;
  // this CTA's groups [g0, g0 + Gc) of K
  const int g0 = rank * (G / C) + min(rank, G % C);
  const int Gc = G / C + (rank < G % C ? 1 : 0);
  const uint32_t ring = tc::smem_u32(smem);
  const uint32_t raw_s = tc::smem_u32(smem + a.off_raw_s), raw_z = tc::smem_u32(smem + a.off_raw_z);
  float* red = reinterpret_cast<float*>(smem + a.off_red);
  // per matrix segment k of the current band: row0, sc_off, z_off; [3] = segments
  int* seg_tab = reinterpret_cast<int*>(smem + a.off_seg);
  const uint32_t bar0 = tc::smem_u32(smem + a.off_bar);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (S + s); };
  auto red_full = [&](int r) { return bar0 + 8u * (2 * S + r); };
  auto red_empty = [&](int r) { return bar0 + 8u * (2 * S + RS + r); };
  const uint32_t meta_full = bar0 + 8u * (2 * S + 2 * RS), meta_empty = meta_full + 8u, ready = meta_full + 16u;
  // with a cluster: the last band's sums have all arrived and the compute
  // warps may help add them (the reducer arrives)
  const uint32_t final_go = meta_full + 32u;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + a.off_bar + 8 * (2 * S + 2 * RS) + 24);
  // A failed wait stops every later wait of the CTA (they return at once);
  // every arrive still happens, so no barrier count goes wrong.
  auto wait = [&](uint32_t bar, uint32_t parity, int site) {
    if (*abort_flag) return false;
    const bool ok = tc::mbar_wait(bar, parity, a.err, site);
    if (!ok) *abort_flag = 1;
    return ok;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(full(s), 1);
      tc::mbar_init(empty(s), W);
    }
    for (int r = 0; r < RS; ++r) {
      tc::mbar_init(red_full(r), W);
      tc::mbar_init(red_empty(r), 1);
    }
    tc::mbar_init(meta_full, 1);
    tc::mbar_init(meta_empty, W);
    tc::mbar_init(ready, C);
    tc::mbar_init(final_go, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (C > 1) cluster_sync_all();  // every CTA's barriers exist before any remote arrive
  pdl_launch_dependents();

  // With a cluster, once every rank's sums of band u (the CTA's kbb-th) have
  // landed: this rank adds the C sums of each of its stages in rank order and
  // stores them.  Worker `worker` of `nworkers` takes every nworkers-th of the
  // rank's stages (the outputs do not depend on the split).
  auto owner_sums = [&](int kbb, int u, int worker, int nworkers) {
    int ur0, un;
    sk_band(a, u, ur0, un);
    const int Tp = (a.T + 3) & ~3, nq = Tp >> 2;
    const int bufo = ((kbb & 1) % a.recv_bufs) * (C * a.slots * kSkTile * Tp);
    const float4* rf = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(smem + a.off_recv) + bufo);
    for (int cur = 0, i = 0; cur < un; ++i) {
      int p, mfirst;
      const int rows_i = sk_stage(a, ur0, un, cur, p, mfirst);
      if (i % C == rank && (i / C) % nworkers == worker) {
        const int off = kSkTile - rows_i, slot = i / C;
        const int np = a.row_end[p] - mfirst;
        __half* yp = a.y[p] + (ur0 + cur - off - mfirst);
        for (int e = lane; e < kSkTile * nq; e += 32) {
          const int rr = e & 15, tq = e >> 4;
          if (rr >= off) {
            float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            for (int q = 0; q < C; ++q) {
              const float4 w4 = rf[((q * a.slots + slot) * kSkTile + rr) * nq + tq];
              v.x += w4.x;
              v.y += w4.y;
              v.z += w4.z;
              v.w += w4.w;
            }
            const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (4 * tq + j < a.T) yp[static_cast<int64_t>(4 * tq + j) * np + rr] = __float2half_rn(vv[j]);
          }
        }
      }
      cur += rows_i;
    }
  };

  if (warp == W) {
    // ---------------- producer: the band's scales, then its weight stages ----------------
    if (lane == 0) {
      for (int p = 0; p < a.np; ++p) tc::prefetch_tmap(&a.tm[p]);
      const uint32_t box_bytes = static_cast<uint32_t>(a.stage_bytes);
      int s = 0, it = 0, kb = 0;
      uint32_t ph = 0;
      for (int u = cl; u < a.NU; u += a.NC, ++kb) {
        int ur0, un;
        sk_band(a, u, ur0, un);
        // the previous band's scales are no longer read
        if (kb > 0) wait(meta_empty, (kb - 1) & 1, kSkSiteMeta);
        uint32_t meta_bytes = 0;
        SkSeg sg;
        int nseg = 0;
        for (; sk_segment(a, ur0, un, G, nseg, sg); ++nseg) {
          seg_tab[4 * nseg] = sg.row0;
          seg_tab[4 * nseg + 1] = sg.sc_off;
          seg_tab[4 * nseg + 2] = sg.z_off;
          meta_bytes += sg.sc_bytes + sg.z_bytes;
        }
        seg_tab[3] = nseg;
        tc::mbar_arrive_expect_tx(meta_full, meta_bytes);
        uint32_t so = 0, zo = 0;
        for (int k = 0; sk_segment(a, ur0, un, G, k, sg); ++k) {
          tc::bulk_load(raw_s + so, sg.sc_lo, sg.sc_bytes, meta_full);
          so += sg.sc_bytes;
          if (sg.z_bytes) tc::bulk_load(raw_z + zo, sg.z_lo, sg.z_bytes, meta_full);
          zo += sg.z_bytes;
        }
        for (int cur = 0; cur < un; ++it) {
          if (it >= S) wait(empty(s), ph ^ 1u, kSkSiteEmpty);
          int p, mfirst;
          const int rows_i = sk_stage(a, ur0, un, cur, p, mfirst);
          tc::mbar_arrive_expect_tx(full(s), box_bytes);
          if (!*abort_flag)
            // 16 rows ending at the stage's last row (matrix-relative; rows
            // before the matrix's first are zero-filled)
            tc::tma_load_2d(ring + s * a.stage_bytes, &a.tm[p], g0 * 8, ur0 + cur + rows_i - kSkTile - mfirst, full(s));
          cur += rows_i;
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // the last copies into the ring and the last band's scales must have
      // landed before the CTA exits
      for (int j = max(0, it - S); j < it; ++j) tc::mbar_wait(full(j % S), (j / S) & 1, a.err, kSkSiteDrain);
      if (kb > 0) tc::mbar_wait(meta_full, (kb - 1) & 1, a.err, kSkSiteDrain);
    }
    return;
  }

  constexpr int kRedPitch = sk_red_pitch(NT);
  const int red_slot = W * kSkTile * kRedPitch;  // floats per reduction slot: [warp][row][token]

  if (warp == W + 1) {
    // ---------------- reducer: the warps' sums of each stage, in warp order ----------------
    // A lane takes row rr of the stage and four consecutive tokens.  With a
    // cluster, stage i of a band belongs to rank i mod C: every rank sends
    // its sums of the stage into slot i / C of the owner's receive buffer,
    // and the owner adds the C sums in rank order once the band is done.
    const int Tp = (a.T + 3) & ~3, nq = Tp >> 2;
    const uint32_t recv = tc::smem_u32(smem + a.off_recv);
    const int buf_floats = C * a.slots * kSkTile * Tp;
    int r = 0, kb = 0;
    uint32_t rph = 0;
    for (int u = cl; u < a.NU; u += a.NC, ++kb) {
      int ur0, un;
      sk_band(a, u, ur0, un);
      const int bufo = ((kb & 1) % a.recv_bufs) * buf_floats;
      for (int cur = 0, i = 0; cur < un; ++i) {
        int p, mfirst;
        const int rows_i = sk_stage(a, ur0, un, cur, p, mfirst);
        const int off = kSkTile - rows_i;
        const int np = a.row_end[p] - mfirst;
        __half* yp = a.y[p] + (ur0 + cur - off - mfirst);  // + t * np + rr
        wait(red_full(r), rph, kSkSiteRedFull);
        const float* rb = red + r * red_slot;
        const int q = i % C, slot = i / C;
        for (int e = lane; e < kSkTile * nq; e += 32) {
          const int rr = e & 15, t0 = (e >> 4) * 4;
          if (rr >= off) {
            // four tokens per load; even and odd warps in two chains, then
            // added (a fixed order)
            float4 v0 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), v1 = v0;
            const float* pr = rb + rr * kRedPitch + t0;
            int w = 0;
            for (; w + 1 < W; w += 2) {
              const float4 a0 = *reinterpret_cast<const float4*>(pr + w * kSkTile * kRedPitch);
              const float4 a1 = *reinterpret_cast<const float4*>(pr + (w + 1) * kSkTile * kRedPitch);
              v0.x += a0.x; v0.y += a0.y; v0.z += a0.z; v0.w += a0.w;
              v1.x += a1.x; v1.y += a1.y; v1.z += a1.z; v1.w += a1.w;
            }
            if (w < W) {
              const float4 a0 = *reinterpret_cast<const float4*>(pr + w * kSkTile * kRedPitch);
              v0.x += a0.x; v0.y += a0.y; v0.z += a0.z; v0.w += a0.w;
            }
            const float4 v = make_float4(v0.x + v1.x, v0.y + v1.y, v0.z + v1.z, v0.w + v1.w);
            if (C == 1) {
              const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (t0 + j < a.T) yp[static_cast<int64_t>(t0 + j) * np + rr] = __float2half_rn(vv[j]);
            } else {
              const uint32_t dst = recv + static_cast<uint32_t>(bufo + ((rank * a.slots + slot) * kSkTile + rr) * Tp + t0) * 4u;
              st_cluster_v4(map_to_rank(dst, q), v);
            }
          }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(red_empty(r));
        if (++r == RS) {
          r = 0;
          rph ^= 1u;
        }
        cur += rows_i;
      }
      if (C > 1) {
        // every rank's sums of the band have landed in their owners' memory
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
        __syncwarp();
        if (lane == 0)
          for (int q = 0; q < C; ++q) mbar_arrive_cluster(map_to_rank(ready, q));
        const bool ok = __all_sync(0xffffffffu, sk_wait_cluster(ready, kb & 1, a.err, kSkSiteReady));
        if (!ok && lane == 0) *abort_flag = 1;
        if (u + a.NC >= a.NU) {
          // the CTA's last band: the compute warps, done with their stages,
          // take a share of the additions
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(final_go);
          if (ok) owner_sums(kb, u, W, W + 1);
        } else if (ok) {
          owner_sums(kb, u, 0, 1);
        }
      }
    }
    return;
  }

  // ---------------- compute warps ----------------
  const int g = lane >> 2, c = lane & 3;
  const int gw = warp * GPW;                    // first CTA-local group of this warp
  const int ngw = max(0, min(GPW, Gc - gw));    // its groups (warp-uniform)

  // The activations may come from the previous kernel in the stream; read
  // through L2 only (an L1 line filled before it finished could be stale).
  pdl_wait();
  uint4 xb[GPW][NT][4];
#pragma unroll
  for (int j = 0; j < GPW; ++j)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int t = nt * 8 + g;
      if (j < ngw && t < a.T) {
        const uint4* xp = reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(t) * a.K +
                                                         (g0 + gw + j) * 128 + c * 32);
        uint4 u[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) u[w] = ldg_cg_v4(xp + w);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t pr[4];
          pair_x(u[w], pr);
          xb[j][nt][w] = make_uint4(pr[0], pr[1], pr[2], pr[3]);
        }
      } else {
#pragma unroll
        for (int w = 0; w < 4; ++w) xb[j][nt][w] = make_uint4(0u, 0u, 0u, 0u);
      }
    }

  const UnpackConsts uk = unpack_consts();
  int s = 0, r = 0, it = 0, kb = 0;
  uint32_t ph = 0, rph = 0;
  for (int u = cl; u < a.NU; u += a.NC, ++kb) {
    int ur0, un;
    sk_band(a, u, ur0, un);
    wait(meta_full, kb & 1, kSkSiteMeta);
    for (int cur = 0; cur < un; ++it) {
      int p, mfirst;
      const int rows_i = sk_stage(a, ur0, un, cur, p, mfirst);
      const int off = kSkTile - rows_i;  // box row of the stage's first row
      // the stage's matrix segment: its first band row and staged scales
      int k = 0;
      const int nseg = seg_tab[3];
#pragma unroll
      for (int q = 1; q < kSkMaxGroup; ++q)
        if (q < nseg && seg_tab[4 * q] <= cur) k = q;
      const int srow0 = seg_tab[4 * k], sc_off = seg_tab[4 * k + 1], z_off = seg_tab[4 * k + 2];
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
      const bool ok = __all_sync(0xffffffffu, wait(full(s), ph, kSkSiteFull));
      if (ok && ngw > 0) {
        const uint32_t cA = ring + s * a.stage_bytes + g * a.pitch + gw * 64 + c * 16;
        const uint32_t cB = cA + 8 * a.pitch;
        // segment rows of box rows g and g + 8 (rows before the segment use
        // its first row's scales; their sums are never stored)
        const int sA = max(cur - off + g - srow0, 0), sB = max(cur - off + g + 8 - srow0, 0);
        uint4 qa[GPW], qb[GPW];
        uint32_t sa[GPW], sb[GPW], za[GPW], zb[GPW];
#pragma unroll
        for (int j = 0; j < GPW; ++j) {
          if (j < ngw) {
            const int gg = g0 + gw + j;
            qa[j] = tc::lds128(cA + j * 64);
            qb[j] = tc::lds128(cB + j * 64);
            sa[j] = lds_u16(raw_s + sc_off + (sA * G + gg) * 2);
            sb[j] = lds_u16(raw_s + sc_off + (sB * G + gg) * 2);
            if (z_off >= 0) {
              const int sh = (gg & 1) * 4;
              za[j] = (lds_u8(raw_z + z_off + sA * a.zpitch + (gg >> 1)) >> sh) & 0xFu;
              zb[j] = (lds_u8(raw_z + z_off + sB * a.zpitch + (gg >> 1)) >> sh) & 0xFu;
            } else {
              za[j] = zb[j] = 8u;
            }
          }
        }
#pragma unroll
        for (int j = 0; j < GPW; ++j) {
          if (j < ngw) {
            const float fA = __half2float(__ushort_as_half(static_cast<unsigned short>(sa[j])));
            const float fB = __half2float(__ushort_as_half(static_cast<unsigned short>(sb[j])));
            float p0[NT][4], p1[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) p0[nt][e] = p1[nt][e] = 0.0f;
            group_mma<NT>(qa[j], qb[j], zp_sub(za[j]), zp_add(za[j]), zp_sub(zb[j]), zp_add(zb[j]), xb[j], p0, p1, uk);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              acc[nt][0] = fmaf(fA, p0[nt][0] + p1[nt][0], acc[nt][0]);
              acc[nt][1] = fmaf(fA, p0[nt][1] + p1[nt][1], acc[nt][1]);
              acc[nt][2] = fmaf(fB, p0[nt][2] + p1[nt][2], acc[nt][2]);
              acc[nt][3] = fmaf(fB, p0[nt][3] + p1[nt][3], acc[nt][3]);
            }
          }
        }
      }
      // the stage's codes are consumed: hand it back to the producer
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(empty(s));
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
      // this warp's sums of the stage into a free reduction slot
      if (it >= RS) wait(red_empty(r), rph ^ 1u, kSkSiteRedEmpty);
      float* rw = red + r * red_slot + warp * kSkTile * kRedPitch;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int t0 = nt * 8 + 2 * c;
        *reinterpret_cast<float2*>(rw + g * kRedPitch + t0) = make_float2(acc[nt][0], acc[nt][1]);
        *reinterpret_cast<float2*>(rw + (g + 8) * kRedPitch + t0) = make_float2(acc[nt][2], acc[nt][3]);
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(red_full(r));
      if (++r == RS) {
        r = 0;
        rph ^= 1u;
      }
      cur += rows_i;
    }
    // the band's staged scales are no longer read by this warp
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(meta_empty);
  }
  if (C > 1 && kb > 0) {
    // help add the last band's sums once they have all arrived
    const bool go = __all_sync(0xffffffffu, tc::mbar_wait(final_go, 0, a.err, kSkSiteReady));
    if (go && !*abort_flag) owner_sums(kb - 1, cl + (kb - 1) * a.NC, warp, W + 1);
  }
}

// ---------------------------------------------------------------- host side

struct SkPlan {
  int NT = 0, GPW = 0, C = 0, W = 0, NC = 0, NU = 0, S = 0, RS = 0, pitch = 0, stage_bytes = 0, Umax = 0;
  int slots = 0, recv_bufs = 1;
  int off_raw_s = 0, off_raw_z = 0, off_red = 0, off_recv = 0, off_seg = 0, off_bar = 0, smem = 0;
  const void* fn = nullptr;
};

template <int NT, int GPW>
const void* sk_fn() {
  return reinterpret_cast<const void*>(w4a16_skinny_kernel<NT, GPW>);
}

// The instantiations: one or two token tiles, one or two groups per warp
// (a TMA box row holds at most 32 groups, so 16 or 14 warps need at most two).
const void* sk_kernel(int NT, int GPW) {
  if (NT == 1) {
    switch (GPW) {
      case 1: return sk_fn<1, 1>();
      case 2: return sk_fn<1, 2>();
    }
  } else if (NT == 2) {
    switch (GPW) {
      case 1: return sk_fn<2, 1>();
      case 2: return sk_fn<2, 2>();
    }
  }
  return nullptr;
}


struct SkDevice {
  bool ok = false;
  int sms = 0, sm_smem = 0, reserved = 0, block_smem = 0;
  int clusters[5] = {0, 0, 0, 0, 0};  // co-resident clusters of size 1, 2, 4 at one CTA per SM
};

// The device's limits, and how many clusters of each size fit with one CTA
// per SM (a CTA asks for more than half of an SM's shared memory).
const SkDevice& sk_device() {
  static SkDevice d;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return;
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&d.reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    cudaDeviceGetAttribute(&d.block_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const int half = d.sm_smem / 2 - d.reserved + 16;
    const void* fn = sk_kernel(1, 1);
    if (d.sms <= 0 || half > d.block_smem ||
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, d.block_smem) != cudaSuccess)
      return;
    for (int C : {1, 2, 4}) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(C * d.sms);
      cfg.blockDim = dim3((sk_max_warps(1) + 2) * 32);
      cfg.dynamicSmemBytes = half;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = C;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
      d.clusters[C] = std::min(n, d.sms / C);
    }
    cudaGetLastError();
    d.ok = d.clusters[1] > 0;
  });
  return d;
}

// Shared-memory plan for cluster size C and GPW groups per warp; false when
// it does not fit.
bool sk_layout(int64_t T, int64_t N, int64_t K, int C, int GPW, const SkDevice& d, SkPlan& p) {
  const int G = static_cast<int>(K / 128), zpitch = (G + 1) / 2;
  if (G < C || d.clusters[C] <= 0) return false;
  p.NT = T <= 8 ? 1 : 2;
  p.GPW = GPW;
  p.C = C;
  const int Gc = (G + C - 1) / C;
  p.W = (Gc + GPW - 1) / GPW;
  if (GPW > kSkMaxGpw || p.W > sk_max_warps(p.NT)) return false;
  // a stage is one TMA box of 16 rows x Gc groups (8 Gc elements of 8 bytes)
  if (Gc > kSkMaxBoxGroups) return false;
  p.NC = static_cast<int>(std::min<int64_t>(d.clusters[C], (N + kSkTile - 1) / kSkTile));
  p.pitch = Gc * 64;
  p.stage_bytes = kSkTile * p.pitch;
  auto up = [](int v, int m) { return (v + m - 1) / m * m; };
  p.RS = p.NT == 1 ? 4 : 2;
  const int red_bytes = p.RS * p.W * kSkTile * sk_red_pitch(p.NT) * 4;
  // bands: as few as fit the per-CTA budget of staged scales and received sums
  const int per_row = G * 2 + zpitch + (C > 1 ? 2 * (static_cast<int>(T) + 3) / 4 * 16 : 0);
  const int64_t rows_cl = (N + p.NC - 1) / p.NC;
  const int64_t umax_budget = std::max<int64_t>(kSkTile, kSkBandBudget / per_row);
  const int64_t bands_cl = (rows_cl + umax_budget - 1) / umax_budget;
  p.NU = static_cast<int>(std::min<int64_t>(N, p.NC * bands_cl));
  p.Umax = static_cast<int>((N + p.NU - 1) / p.NU);
  const int band_stages = (p.Umax + kSkTile - 1) / kSkTile + kSkMaxGroup;  // a segment adds one short stage
  p.slots = (band_stages + C - 1) / C;
  p.recv_bufs = bands_cl > 1 ? 2 : 1;
  // raw staging: the band's bytes plus up to 32 bytes of alignment window per segment
  const int raw_s_bytes = up(p.Umax * G * 2, 16) + 32 * kSkMaxGroup;
  const int raw_z_bytes = up(p.Umax * zpitch, 16) + 32 * kSkMaxGroup;
  const int Tp = (static_cast<int>(T) + 3) & ~3;
  const int recv_bytes = C > 1 ? p.recv_bufs * C * p.slots * kSkTile * Tp * 4 : 0;
  const int bar_bytes = 8 * (2 * kSkMaxStages + 2 * p.RS) + 40;
  const int fixed = raw_s_bytes + raw_z_bytes + red_bytes + up(recv_bytes, 16) + 64 + bar_bytes + 128;
  const int cap = d.block_smem;
  const int bands_per_cl = static_cast<int>((p.NU + p.NC - 1) / p.NC);
  const int stages_max = bands_per_cl * ((p.Umax + kSkTile - 1) / kSkTile + kSkMaxGroup);
  p.S = std::min({kSkMaxStages, (cap - fixed) / p.stage_bytes, std::max(stages_max, kSkMinStages)});
  if (p.S < kSkMinStages) return false;
  p.off_raw_s = up(p.S * p.stage_bytes, 128);
  p.off_raw_z = p.off_raw_s + raw_s_bytes;
  p.off_red = up(p.off_raw_z + raw_z_bytes, 16);
  p.off_recv = p.off_red + red_bytes;
  p.off_seg = up(p.off_recv + recv_bytes, 16);
  p.off_bar = p.off_seg + 64;
  p.smem = p.off_bar + 8 * (2 * p.S + 2 * p.RS) + 40;
  // more than half of the SM, so that no two CTAs share one
  p.smem = std::max(p.smem, d.sm_smem / 2 - d.reserved + 16);
  if (p.smem > cap) return false;
  p.fn = sk_kernel(p.NT, p.GPW);
  return p.fn != nullptr;
}

// The K split depends on T and K only, so that every output element is the
// same sum in the same order whatever N is and however matrices are grouped:
// the smallest C with a launch plan (measured fastest: the compute of a
// stage, not the activations' traffic, sets the pace).
bool sk_plan(int64_t T, int64_t N, int64_t K, SkPlan& best) {
  if (T < 1 || T > kSkMaxTokens || N <= 0 || K < 128 || K % 128 != 0) return false;
  const SkDevice& d = sk_device();
  if (!d.ok) return false;
  bool found = false;
  for (int C : {1, 2, 4}) {
    const int G = static_cast<int>(K / 128), Gc = (G + C - 1) / C;
    const int NT = T <= 8 ? 1 : 2;
    // the fewest groups per warp that keep the warps within the limit
    const int GPW = std::max(1, (Gc + sk_max_warps(NT) - 1) / sk_max_warps(NT));
    if (GPW > kSkMaxGpw) continue;
    SkPlan p;
    if (!sk_layout(T, N, K, C, GPW, d, p)) continue;
    best = p;
    found = true;
    break;
  }
  return found;
}

}  // namespace

bool w4a16_skinny_supported(int64_t T, int64_t N, int64_t K) {
  SkPlan p;
  return N <= (int64_t(1) << 30) && sk_plan(T, N, K, p);
}

cudaError_t launch_w4a16_skinny_grouped(const void* x, int64_t T, int64_t K, int count, const int64_t* N,
                                        const uint8_t* const* wq, const void* const* scales,
                                        const uint8_t* const* zeros, void* const* y, cudaStream_t stream) {
  if (count < 1 || count > kSkMaxGroup) return cudaErrorInvalidValue;
  SkArgs a = {};
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
  if (total == 0 || T == 0) return cudaSuccess;
  SkPlan p;
  if (total > (int64_t(1) << 30) || !sk_plan(T, total, K, p)) return cudaErrorInvalidValue;
  a.x = static_cast<const __half*>(x);
  a.err = device_error_word();
  a.T = static_cast<int>(T);
  a.N = static_cast<int>(total);
  a.K = static_cast<int>(K);
  a.zpitch = static_cast<int>((K / 128 + 1) / 2);
  a.C = p.C;
  a.NC = p.NC;
  a.NU = p.NU;
  a.W = p.W;
  a.S = p.S;
  a.RS = p.RS;
  a.pitch = p.pitch;
  a.stage_bytes = p.stage_bytes;
  a.slots = p.slots;
  a.recv_bufs = p.recv_bufs;
  a.off_raw_s = p.off_raw_s;
  a.off_raw_z = p.off_raw_z;
  a.off_red = p.off_red;
  a.off_recv = p.off_recv;
  a.off_seg = p.off_seg;
  a.off_bar = p.off_bar;
  const int Gc = (static_cast<int>(K / 128) + p.C - 1) / p.C;
  for (int q = 0; q < a.np; ++q) {
    const int64_t rows = a.row_end[q] - (q > 0 ? a.row_end[q - 1] : 0);
    cudaError_t e = make_tmap_2d_u64(&a.tm[q], a.wq[q], static_cast<uint64_t>(K / 16), static_cast<uint64_t>(rows),
                                     static_cast<uint32_t>(8 * Gc), kSkTile);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = ensure_max_dynamic_smem(p.fn);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.NC * p.C);
  cfg.blockDim = dim3((p.W + 2) * 32);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = p.C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.C > 1 ? 2 : 1;
  void* args[] = {&a};
  return cudaLaunchKernelExC(&cfg, p.fn, args);
}

}  // namespace qlin
