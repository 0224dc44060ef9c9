// W4A16 decode for up to 16 tokens: a chain of dependent linears (a
// decoder's layers at decode time) run step after step in ONE persistent
// launch on the warp-level tensor cores.
//
//   Y_s[t,n] = sum_g s[n,g] . sum_{k in g} X_s[t,k] . (q[n,k] - z[n,g])
//
// ("Chapter 9 - Quantization kernels", 9.1: decode reads every weight once
// per token, so a layer is a weight-bandwidth problem; 9.5: dequantize in
// registers right before the tensor core, memory only ever holds the 4-bit
// codes; 9.6: the magic-number unpack with the zero-point folded in; 9.7:
// multi-token decode with the weight rows as the MMA's M side.  "LLM and
// AIGC quantization", W4A16 section.)
//
// Why one launch.  The layers of a decoder depend on one another (q,k,v ->
// o -> gate,up -> down) and each one of a 7B-class model holds only 8-45 MB
// of codes, 1.3-6.6 us at HBM speed.  Launched one by one, every layer pays
// its launch, the latency of its first copies and its tail.  Here every CTA
// (exactly one per SM) streams its share of EVERY step's weights into a
// shared-memory ring in step order, waiting for nothing but free slots, so
// the copies of step s+1 are in flight while step s still computes on other
// SMs.  Only the compute waits for a step's input: one counter per step in
// the plan's workspace (each CTA adds one with release semantics once its
// outputs of the step are stored; one thread per CTA polls it with acquire
// semantics) orders the steps.
//
// Work split.  The matrices of a step (e.g. q, k and v, which read the same
// x) form one range of 32-row units (a matrix's last unit may be short: the
// copy fills the rows past its end with zeros and their sums are never
// stored); CTA c takes a contiguous share of the units (shares differ by at
// most one unit).  K is cut into chunks of 16 groups (2048 codes, 1 KB per
// row); a stage is one unit x one chunk, one 2-D TMA box of 32 rows.  Each of
// the 8 compute warps owns two consecutive groups of the chunk and holds
// their activations in registers for all the CTA's units, already in the
// layout of the m16n8k16 B fragments; per stage it turns its 32 x 256 codes
// into exact fp16 (q - z) A fragments (two MMA tiles of 16 rows), runs the
// MMAs (fp32 accumulation per group, then scaled by s[n,g] in fp32) and
// writes its partial sums into a double-buffered slot.  Half of the warps
// (alternating with the slot) add the 8 warps' partial sums of each (row,
// token) in warp order and either store the fp16 output (a single chunk) or
// add them to the row's sum in shared memory, chunk by chunk in order.
// Every output is the same sum in the same order on every run.
//
// Waits are bounded: a wait that expires records its site in the device
// error word and makes the CTA skip the rest of its work; the other CTAs'
// bounded waits on the step counters then expire the same way.  After such
// an error the plan's counters are stale and the plan must be prepared again.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "device_common.cuh"
#include "qlin_internal.h"
#include "tc_common.cuh"
#include "tmap.h"
#include "w4a16_mma_common.cuh"

namespace qlin {
namespace {

using namespace w4mma;

constexpr int kDcKWarps = 8;                     // warps along K: each owns two groups of a chunk
constexpr int kDcUnit = 32;                      // rows per stage: two MMA tiles of 16
constexpr int kDcChunkGroups = 2 * kDcKWarps;    // groups per K chunk
constexpr int kDcChunkU64 = kDcChunkGroups * 8;  // 128 8-byte elements: 1 KB of codes per row
constexpr int kDcStageBytes = kDcUnit * kDcChunkU64 * 8;  // 32 KB
constexpr int kDcMaxGroup = QLIN_W4A16_MAX_GROUP;
constexpr int kDcPitch = 36;                     // floats per token of a partial-sum slot: 32 rows + 4 pad
constexpr int kDcMetaBytes = 20 * 1024;          // per buffer: a share's segment table, scales and zero-points
constexpr int kDcSegTable = 256;                 // bytes of the segment table at the start of a meta buffer
constexpr int kDcAccBytes = 16 * 1024;           // cross-chunk sums of a CTA's rows
constexpr int kDcSmemMax = 227 * 1024;
constexpr uint32_t kDcMagic = 0x51444331u;
constexpr int kDcSiteFull = 1, kDcSiteEmpty = 2, kDcSiteMeta = 3, kDcSiteMetaEmpty = 4, kDcSitePartFull = 5,
              kDcSitePartEmpty = 6, kDcSiteGrid = 7, kDcSiteDrain = 8, kDcSitePlan = 9;
constexpr int kDcSiteBase = 0x300;  // sites of this kernel in the device error word: timeout base + 0x300 + site

// One step of a plan, as the kernel reads it from the workspace.
struct DcStep {
  const __half* x;
  const __half* scales[kDcMaxGroup];
  const uint8_t* zeros[kDcMaxGroup];  // nullptr: symmetric, z = 8
  __half* y[kDcMaxGroup];
  int unit_end[kDcMaxGroup];          // matrix p covers units [unit_end[p-1], unit_end[p])
  int N[kDcMaxGroup];
  int np, K, G, zpitch, nchunks, chunk_u64, units, map0;
};

// Workspace: header, steps, tensor maps (64-byte aligned), one counter per step.
struct DcHeader {
  uint32_t magic;
  int nsteps, T, grid;
  int steps_off, maps_off, counters_off, pad;
};

// A matrix segment of a CTA's share of a step, written by the producer into
// the first bytes of the step's meta buffer.
struct DcSeg {
  int unit_begin;  // first unit of the matrix (step-wide index)
  int unit_end;
  int sc_off;      // meta-buffer offset of the scale of (matrix row 0, group 0) (may be negative)
  int z_off;       // same for the packed zero-points (may be negative)
  int N;
  int has_z;       // 0: symmetric matrix, z = 8
  __half* y;
};
static_assert(sizeof(DcSeg) * kDcMaxGroup + 16 <= kDcSegTable, "segment table too large");

__host__ __device__ constexpr int dc_part_slot_bytes(int NT) { return kDcKWarps * 8 * NT * kDcPitch * 4; }

struct DcLayout {
  int S, meta, part, acc, bars, total;
};
__host__ __device__ inline DcLayout dc_layout(int NT, int S) {
  DcLayout l;
  l.S = S;
  l.meta = S * kDcStageBytes;
  l.part = l.meta + 2 * kDcMetaBytes;
  l.acc = l.part + 2 * dc_part_slot_bytes(NT);
  l.bars = l.acc + kDcAccBytes;
  l.total = l.bars + 8 * (2 * S + 8) + 16;
  return l;
}

// Contiguous share of `units` units for CTA `cta` of `grid`.
__device__ __forceinline__ void dc_share(int units, int grid, int cta, int& ub, int& ue) {
  const int base = units / grid, extra = units % grid;
  ub = cta * base + min(cta, extra);
  ue = ub + base + (cta < extra ? 1 : 0);
}

__device__ __forceinline__ uint32_t dc_lds_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t dc_lds_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ unsigned int dc_ld_acquire(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned int dc_atom_add_acq_rel(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void dc_red_release(unsigned int* p, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Barrier over the compute warps (`threads` threads) with an OR of the
// threads' predicates: every thread gets the same answer, so a decision
// taken on it cannot diverge.
__device__ __forceinline__ bool dc_sync_or(bool pred, int threads) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, 1, %2, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(threads)
      : "memory");
  return r != 0;
}

// 2-D TMA tile load with an L2 cache policy (the weights are read once).
__device__ __forceinline__ void dc_tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// NT token tiles of 8 (T <= 8 NT).  W compute warps (8: each warp takes both
// MMA tiles of a unit; 16: warps 0-7 the first, 8-15 the second), then the
// producer warp.
template <int NT, int W>
__global__ void __launch_bounds__((W + 1) * 32, 1)
    w4a16_decode_kernel(const unsigned char* __restrict__ ws, int nsteps, int T, int S, int32_t* err) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const DcHeader* hdr = reinterpret_cast<const DcHeader*>(ws);
  if (hdr->magic != kDcMagic || hdr->nsteps != nsteps || hdr->T != T || hdr->grid != static_cast<int>(gridDim.x) ||
      T < 1 || T > 8 * NT) {
    if (threadIdx.x == 0) record_device_error(err, kDevErrTimeoutBase + kDcSiteBase + kDcSitePlan);
    return;
  }
  const DcStep* steps = reinterpret_cast<const DcStep*>(ws + hdr->steps_off);
  const CUtensorMap* maps = reinterpret_cast<const CUtensorMap*>(ws + hdr->maps_off);
  unsigned int* counters = reinterpret_cast<unsigned int*>(const_cast<unsigned char*>(ws) + hdr->counters_off);
  const DcLayout L = dc_layout(NT, S);
  constexpr int kRedWarps = W / 2;  // warps that add up one stage's partial sums
  constexpr int kRowSplit = W / kDcKWarps;  // warps per (unit, pair of groups): 1 (W = 8) or 2 (W = 16)
  constexpr int kTilesPerWarp = 2 / kRowSplit;  // MMA tiles of a unit per warp
  const int grid = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  const uint32_t ring = tc::smem_u32(smem);
  const uint32_t bar0 = tc::smem_u32(smem + L.bars);
  auto full = [&](int i) { return bar0 + 8u * i; };
  auto empty = [&](int i) { return bar0 + 8u * (S + i); };
  const uint32_t meta_full = bar0 + 8u * (2 * S), meta_empty = meta_full + 16u;
  const uint32_t part_full = meta_full + 32u, part_empty = meta_full + 48u;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.bars + 8 * (2 * S + 8));
  // A failed wait stops every later wait of the CTA (they return at once).
  auto wait = [&](uint32_t bar, uint32_t parity, int where) {
    if (*abort_flag) return false;
    const bool ok = tc::mbar_wait(bar, parity, err, kDcSiteBase + where);
    if (!ok) *abort_flag = 1;
    return ok;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(full(i), 1);
      tc::mbar_init(empty(i), W);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(meta_full + 8u * b, 1);
      tc::mbar_init(meta_empty + 8u * b, W);
      tc::mbar_init(part_full + 8u * b, W);
      tc::mbar_init(part_empty + 8u * b, kRedWarps);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();

  if (warp == W) {
    // ---------------- producer: every step's share, in step order ----------------
    if (lane == 0) {
      const uint64_t policy = tc::l2_policy_evict_first();
      int it = 0, last_meta = -1;
      for (int s = 0; s < nsteps; ++s) {
        if (*abort_flag) break;
        const DcStep& st = steps[s];
        int ub, ue;
        dc_share(st.units, grid, cta, ub, ue);
        const int mb = s & 1;
        if (s >= 2 && !wait(meta_empty + 8u * mb, ((s >> 1) - 1) & 1, kDcSiteMetaEmpty)) break;
        unsigned char* meta = smem + L.meta + mb * kDcMetaBytes;
        DcSeg* seg = reinterpret_cast<DcSeg*>(meta);
        // the scale and zero-point windows of each matrix segment of the share
        // (16-byte aligned windows around the rows' bytes)
        int at = kDcSegTable, nseg = 0, ncopy = 0;
        uint32_t bytes = 0;
        const char* src_lo[2 * kDcMaxGroup];
        uint32_t src_bytes[2 * kDcMaxGroup];
        int dst_at[2 * kDcMaxGroup];
        for (int p = 0; p < st.np; ++p) {
          const int u0 = p > 0 ? st.unit_end[p - 1] : 0, u1 = st.unit_end[p];
          const int a = max(u0, ub), b = min(u1, ue);
          if (a >= b) continue;
          // matrix rows of the segment (the last unit of a matrix may be short)
          const int r0 = (a - u0) * kDcUnit, r1 = min((b - u0) * kDcUnit, st.N[p]);
          const uintptr_t sc = reinterpret_cast<uintptr_t>(st.scales[p]) + static_cast<uintptr_t>(r0) * st.G * 2;
          const uintptr_t sc_lo = sc & ~uintptr_t(15);
          const uint32_t sc_bytes = static_cast<uint32_t>(
              ((sc + static_cast<uintptr_t>(r1 - r0) * st.G * 2 + 15) & ~uintptr_t(15)) - sc_lo);
          DcSeg& sg = seg[nseg];
          sg.unit_begin = u0;
          sg.unit_end = u1;
          sg.sc_off = at + static_cast<int>(sc - sc_lo) - r0 * st.G * 2;
          sg.N = st.N[p];
          sg.y = st.y[p];
          src_lo[ncopy] = reinterpret_cast<const char*>(sc_lo);
          src_bytes[ncopy] = sc_bytes;
          dst_at[ncopy++] = at;
          at += static_cast<int>(sc_bytes);
          bytes += sc_bytes;
          if (st.zeros[p]) {
            const uintptr_t z = reinterpret_cast<uintptr_t>(st.zeros[p]) + static_cast<uintptr_t>(r0) * st.zpitch;
            const uintptr_t z_lo = z & ~uintptr_t(15);
            const uint32_t z_bytes = static_cast<uint32_t>(
                ((z + static_cast<uintptr_t>(r1 - r0) * st.zpitch + 15) & ~uintptr_t(15)) - z_lo);
            sg.z_off = at + static_cast<int>(z - z_lo) - r0 * st.zpitch;
            sg.has_z = 1;
            src_lo[ncopy] = reinterpret_cast<const char*>(z_lo);
            src_bytes[ncopy] = z_bytes;
            dst_at[ncopy++] = at;
            at += static_cast<int>(z_bytes);
            bytes += z_bytes;
          } else {
            sg.z_off = 0;
            sg.has_z = 0;
          }
          ++nseg;
        }
        *reinterpret_cast<int*>(meta + sizeof(DcSeg) * kDcMaxGroup) = nseg;
        const uint32_t mbar = meta_full + 8u * mb;
        tc::mbar_arrive_expect_tx(mbar, bytes);  // release: the table is visible to the waiters
        for (int i = 0; i < ncopy; ++i)
          tc::bulk_load(tc::smem_u32(meta + dst_at[i]), src_lo[i], src_bytes[i], mbar);
        last_meta = s;
        // the step's tensor maps were written into the workspace by earlier
        // kernels (generic proxy): make those writes visible to the copies
        for (int p = 0; p < st.np; ++p)
          asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(
                           reinterpret_cast<uint64_t>(&maps[st.map0 + p]))
                       : "memory");
        // the weight stages: chunk by chunk, the share's units in order
        const uint32_t box_bytes = static_cast<uint32_t>(kDcUnit * st.chunk_u64 * 8);
        bool stop = false;
        for (int j = 0; j < st.nchunks && !stop; ++j) {
          int p = 0;
          for (int u = ub; u < ue; ++u, ++it) {
            while (p + 1 < st.np && u >= st.unit_end[p]) ++p;
            const int slot = it % S;
            if (it >= S && !wait(empty(slot), ((it / S) - 1) & 1, kDcSiteEmpty)) {
              stop = true;
              break;
            }
            const int u0 = p > 0 ? st.unit_end[p - 1] : 0;
            tc::mbar_arrive_expect_tx(full(slot), box_bytes);
            // rows past the matrix's last row are filled with zeros
            dc_tma_load_2d(ring + slot * kDcStageBytes, &maps[st.map0 + p], j * kDcChunkU64, (u - u0) * kDcUnit,
                           full(slot), policy);
          }
        }
        if (stop) break;
      }
      // every copy still in flight lands before the CTA exits
      for (int i = max(0, it - S); i < it; ++i) tc::mbar_wait(full(i % S), (i / S) & 1, err, kDcSiteBase + kDcSiteDrain);
      for (int s = max(0, last_meta - 1); s <= last_meta; ++s)
        tc::mbar_wait(meta_full + 8u * (s & 1), (s >> 1) & 1, err, kDcSiteBase + kDcSiteDrain);
    }
    return;
  }

  // ---------------- compute warps ----------------
  const int g = lane >> 2, c = lane & 3;
  constexpr int Tp = 8 * NT;
  constexpr int kWarpFloats = Tp * kDcPitch;           // one warp's partial sums of a stage
  constexpr int kSlotFloats = kDcKWarps * kWarpFloats;
  const int kw = warp % kDcKWarps;        // this warp's pair of groups in a chunk
  const int h0 = (warp / kDcKWarps) * kTilesPerWarp;  // its first MMA tile of a unit
  float* part = reinterpret_cast<float*>(smem + L.part);
  float* accbuf = reinterpret_cast<float*>(smem + L.acc);
  const UnpackConsts uk = unpack_consts();
  int slot = 0, si = 0;  // ring slot and its phase (kept incrementally), stage count
  uint32_t phase = 0;
  for (int s = 0; s < nsteps; ++s) {
    const DcStep& st = steps[s];
    int ub, ue;
    dc_share(st.units, grid, cta, ub, ue);
    // the step's input: every CTA has stored step s - 1 (and so every step before it)
    if (s > 0) {
      bool failed = false;
      if (threadIdx.x == 0 && !*abort_flag) {
        const unsigned int* cnt = counters + (s - 1);
        if (dc_ld_acquire(cnt) < static_cast<unsigned int>(grid)) {
          const long long t0 = clock64();
          while (dc_ld_acquire(cnt) < static_cast<unsigned int>(grid)) {
            if (clock64() - t0 > tc::kWaitTimeoutCycles || *abort_flag) {
              record_device_error(err, kDevErrTimeoutBase + kDcSiteBase + kDcSiteGrid);
              failed = true;
              *abort_flag = 1;
              break;
            }
          }
        }
      }
      if (dc_sync_or(failed || *abort_flag, W * 32)) break;
    }
    const int mb = s & 1;
    if (!wait(meta_full + 8u * mb, (s >> 1) & 1, kDcSiteMeta)) ue = ub;  // nothing more to do after a failure
    const unsigned char* meta = smem + L.meta + mb * kDcMetaBytes;
    const uint32_t meta_a = tc::smem_u32(meta);
    const DcSeg* seg = reinterpret_cast<const DcSeg*>(meta);
    const int nseg = min(max(*reinterpret_cast<const int*>(meta + sizeof(DcSeg) * kDcMaxGroup), 1), kDcMaxGroup);
    const int K = st.K, G = st.G, zpitch = st.zpitch, nch = st.nchunks, pitch = st.chunk_u64 * 8;
    const __half* x = st.x;
    // this warp's two groups of chunk j, and their activations (raw loads, then
    // the pairing in place: every load in flight at once)
    auto chunk_groups = [&](int j, int& gg0, int& ngw) {
      gg0 = j * kDcChunkGroups + 2 * kw;
      ngw = min(2, max(0, G - gg0));
    };
    auto load_raw = [&](int j, uint4 (*dst)[NT][4]) {
      int gg0, ngw;
      chunk_groups(j, gg0, ngw);
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int t = nt * 8 + g;
          if (jj < ngw && t < T && ub < ue) {
            const uint4* xp =
                reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * K + (gg0 + jj) * 128 + c * 32);
#pragma unroll
            for (int w = 0; w < 4; ++w) dst[jj][nt][w] = ldg_cg_v4(xp + w);
          } else {
#pragma unroll
            for (int w = 0; w < 4; ++w) dst[jj][nt][w] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
    };
    auto pair_all = [&](uint4 (*v)[NT][4]) {
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint32_t pr[4];
            pair_x(v[jj][nt][w], pr);
            v[jj][nt][w] = make_uint4(pr[0], pr[1], pr[2], pr[3]);
          }
    };
    // one token tile: the next chunk's activations are loaded while the
    // chunk's last unit computes (a second set of registers; more tiles have
    // no room for it)
    constexpr bool kPrefetch = NT == 1;
    uint4 xb[2][NT][4], xn[2][NT][4];
    load_raw(0, xb);
    pair_all(xb);
    for (int j = 0; j < nch; ++j) {
      int gg0, ngw;
      chunk_groups(j, gg0, ngw);
      int k = 0;  // segment of the current unit
      for (int u = ub; u < ue; ++u, ++si) {
        if (kPrefetch && u == ue - 1 && j + 1 < nch) load_raw(j + 1, xn);
        while (k + 1 < nseg && u >= seg[k].unit_end) ++k;
        const int row0 = (u - seg[k].unit_begin) * kDcUnit;  // matrix row of the unit's first row
        const int nrow = seg[k].N;
        const bool ready = __all_sync(0xffffffffu, wait(full(slot), phase, kDcSiteFull));
        // this warp's partial sums of the stage go to slot si & 1: [warp][token][row]
        const int ps = si & 1, use = si >> 1;
        const uint32_t pf = part_full + 8u * ps, pe = part_empty + 8u * ps;
        if (si >= 2) wait(pe, (use - 1) & 1, kDcSitePartEmpty);
        float* pw = part + ps * kSlotFloats + kw * kWarpFloats;
#pragma unroll
        for (int hh = 0; hh < kTilesPerWarp; ++hh) {  // this warp's MMA tiles of the unit
          const int h = h0 + hh;
          float acc[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
          if (ready && ngw > 0) {
            const uint32_t cA = ring + slot * kDcStageBytes + (16 * h + g) * pitch + 2 * kw * 64 + c * 16;
            const uint32_t cB = cA + 8 * pitch;
            // scale / zero-point rows (clamped to the matrix: rows past its end
            // hold zero codes and are never stored)
            const int rA = min(row0 + 16 * h + g, nrow - 1), rB = min(row0 + 16 * h + g + 8, nrow - 1);
            const int sc_off = seg[k].sc_off, z_off = seg[k].z_off, has_z = seg[k].has_z;
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              if (jj < ngw) {
                const int gg = gg0 + jj;
                const uint4 qa = tc::lds128(cA + jj * 64), qb = tc::lds128(cB + jj * 64);
                const float fA = __half2float(
                    __ushort_as_half(static_cast<unsigned short>(dc_lds_u16(meta_a + sc_off + (rA * G + gg) * 2))));
                const float fB = __half2float(
                    __ushort_as_half(static_cast<unsigned short>(dc_lds_u16(meta_a + sc_off + (rB * G + gg) * 2))));
                uint32_t za = 8u, zb = 8u;
                if (has_z) {
                  const int sh = (gg & 1) * 4;
                  za = (dc_lds_u8(meta_a + z_off + rA * zpitch + (gg >> 1)) >> sh) & 0xFu;
                  zb = (dc_lds_u8(meta_a + z_off + rB * zpitch + (gg >> 1)) >> sh) & 0xFu;
                }
                float p0[NT][4], p1[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                  for (int e = 0; e < 4; ++e) p0[nt][e] = p1[nt][e] = 0.0f;
                group_mma<NT>(qa, qb, zp_sub(za), zp_add(za), zp_sub(zb), zp_add(zb), xb[jj], p0, p1, uk);
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
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int t0 = nt * 8 + 2 * c, r = 16 * h + g;
            pw[t0 * kDcPitch + r] = acc[nt][0];
            pw[(t0 + 1) * kDcPitch + r] = acc[nt][1];
            pw[t0 * kDcPitch + r + 8] = acc[nt][2];
            pw[(t0 + 1) * kDcPitch + r + 8] = acc[nt][3];
          }
        }
        // the stage's codes are used: hand the slot back
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(empty(slot));
          tc::mbar_arrive(pf);
        }
        if (++slot == S) {
          slot = 0;
          phase ^= 1u;
        }
        // warps W/2 ps .. W/2 ps + W/2 - 1 add up the stage's partial sums:
        // tokens rw + W/2 i, row = lane, the 8 K-warps' sums in order
        const int rw = warp - kRedWarps * ps;
        if (rw >= 0 && rw < kRedWarps) {
          const bool got = __all_sync(0xffffffffu, wait(pf, use & 1, kDcSitePartFull));
          const int row = row0 + lane;
          if (got && row < nrow) {
            __half* yrow = seg[k].y + row;
            for (int tok = rw; tok < T; tok += kRedWarps) {
              const float* pr = part + ps * kSlotFloats + tok * kDcPitch + lane;
              float v = 0.0f;
#pragma unroll
              for (int w = 0; w < kDcKWarps; ++w) v += pr[w * kWarpFloats];
              if (nch == 1) {
                yrow[static_cast<int64_t>(tok) * nrow] = __float2half_rn(v);
              } else {
                float* ap = accbuf + ((u - ub) * Tp + tok) * kDcUnit + lane;
                const float a = j == 0 ? v : *ap + v;
                if (j == nch - 1)
                  yrow[static_cast<int64_t>(tok) * nrow] = __float2half_rn(a);
                else
                  *ap = a;
              }
            }
          }
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(pe);
        }
      }
      // the next chunk's activations
      if (j + 1 < nch) {
        if (kPrefetch && ub < ue) {
#pragma unroll
          for (int jj = 0; jj < 2; ++jj)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int w = 0; w < 4; ++w) xb[jj][nt][w] = xn[jj][nt][w];
        } else {
          load_raw(j + 1, xb);
        }
        pair_all(xb);
      }
    }
    // the meta buffer of this step is no longer read by this warp
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(meta_empty + 8u * mb);
    // every output of the step is stored: arrive on the step's counter
    const bool failed = dc_sync_or(*abort_flag != 0, W * 32);
    if (threadIdx.x == 0 && !failed) {
      if (s + 1 < nsteps) {
        dc_red_release(counters + s, 1u);
      } else if (dc_atom_add_acq_rel(counters + s, 1u) == static_cast<unsigned int>(grid - 1)) {
        // the last CTA to finish the last step: every CTA has passed every
        // wait of this launch, so the counters can be zeroed for the next run
        for (int i = 0; i < nsteps; ++i) counters[i] = 0u;
      }
    }
    if (failed) break;
  }
}

// Compute warps: 8 for every token count.  Measured on the decoder stacks:
// 16 warps, each taking one MMA tile of a unit (96 registers at up to 8
// tokens), were slower (1.53 against 1.45 ms at T = 1, 1.74 against 1.58 ms at
// T = 4); so was folding the producer into a compute warp, which lifts the
// register limit from 168 to 255 and let the next chunk's activations load
// early, but the ring then drains while that warp computes (2.6 -> 3.2 ms at
// T = 16).
constexpr int dc_warps(int) { return 8; }

const void* dc_kernel(int NT) {
  return NT == 1 ? reinterpret_cast<const void*>(w4a16_decode_kernel<1, dc_warps(1)>)
                 : reinterpret_cast<const void*>(w4a16_decode_kernel<2, dc_warps(2)>);
}

// Stages of the ring for NT token tiles: as many as fit.
int dc_stages(int NT) {
  int S = 2;
  while (S < 8 && dc_layout(NT, S + 1).total <= kDcSmemMax) ++S;
  return S;
}

struct DcDev {
  std::once_flag once[2];
  cudaError_t attr[2] = {cudaSuccess, cudaSuccess};
};
constexpr int kDcMaxDevices = 64;
DcDev g_dc_dev[kDcMaxDevices];

// The kernel's shared-memory attribute, set once per device and kernel.
cudaError_t dc_set_attr(int NT) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kDcMaxDevices) return cudaErrorInvalidDevice;
  DcDev& d = g_dc_dev[dev];
  std::call_once(d.once[NT - 1], [&] {
    d.attr[NT - 1] = cudaFuncSetAttribute(dc_kernel(NT), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          dc_layout(NT, dc_stages(NT)).total);
  });
  return d.attr[NT - 1];
}

// Workspace layout for nsteps steps and nmaps tensor maps.
struct DcWs {
  int64_t steps_off, maps_off, counters_off, total;
};
DcWs dc_ws_layout(int64_t nsteps, int64_t nmaps) {
  auto up = [](int64_t v, int64_t m) { return (v + m - 1) / m * m; };
  DcWs w;
  w.steps_off = up(sizeof(DcHeader), 64);
  w.maps_off = up(w.steps_off + nsteps * static_cast<int64_t>(sizeof(DcStep)), 64);
  w.counters_off = up(w.maps_off + nmaps * static_cast<int64_t>(sizeof(CUtensorMap)), 64);
  w.total = up(w.counters_off + 4 * nsteps, 256);
  return w;
}

// Copies a host buffer into device memory through kernel parameters (no
// host-side synchronization, and it can be captured in a graph).
constexpr int kDcBlobBytes = 30 * 1024;
struct DcBlob {
  unsigned char* dst;
  int bytes;
  unsigned char data[kDcBlobBytes];
};

__global__ void dc_blob_kernel(const __grid_constant__ DcBlob b) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < b.bytes; i += gridDim.x * blockDim.x) b.dst[i] = b.data[i];
}

}  // namespace

int64_t w4a16_decode_workspace_bytes(int64_t nsteps) {
  if (nsteps < 0 || nsteps > (int64_t(1) << 20)) return -1;
  return dc_ws_layout(nsteps, nsteps * kDcMaxGroup).total;
}

const char* w4a16_decode_check(const qlin_w4a16_step* steps, int nsteps, int64_t T, int* bad_step) {
  *bad_step = -1;
  if (T < 1 || T > 16) return "T must be 1 .. 16";
  const int grid = sm_count();
  for (int s = 0; s < nsteps; ++s) {
    const qlin_w4a16_step& st = steps[s];
    *bad_step = s;
    if (st.K < 128 || st.K % 128 != 0 || st.K > (int64_t(1) << 24)) return "K must be a multiple of 128 in [128, 2^24]";
    int64_t units = 0, nmax = 0;
    for (int p = 0; p < st.count; ++p) {
      units += (st.N[p] + kDcUnit - 1) / kDcUnit;
      nmax = std::max(nmax, st.N[p]);
    }
    if (units > (int64_t(1) << 24) || nmax > (int64_t(1) << 30)) return "too many rows";
    const int64_t share = (units + grid - 1) / grid;  // units of the largest share
    const int64_t G = st.K / 128, zp = (G + 1) / 2;
    // the largest share's scales and zero-points (with up to 32 bytes of
    // window per array and matrix) must fit one staging buffer
    const int64_t meta = kDcSegTable + share * kDcUnit * (2 * G + zp) + 64 * st.count;
    if (meta > kDcMetaBytes) return "a CTA's share of scales and zero-points exceeds its staging buffer";
    const int64_t nch = (G + kDcChunkGroups - 1) / kDcChunkGroups;
    if (nch > 1 && share * kDcUnit * 16 * 4 > kDcAccBytes) return "a CTA's share of rows exceeds its sum buffer";
  }
  *bad_step = -1;
  return nullptr;
}

cudaError_t w4a16_decode_prepare(const qlin_w4a16_step* steps, int nsteps, int64_t T, void* workspace,
                                 cudaStream_t stream) {
  const int grid = sm_count();
  int nmaps = 0;
  for (int s = 0; s < nsteps; ++s) nmaps += steps[s].count;
  const DcWs w = dc_ws_layout(nsteps, nmaps);
  std::vector<unsigned char> buf(static_cast<size_t>(w.total), 0);
  DcHeader h = {};
  h.magic = kDcMagic;
  h.nsteps = nsteps;
  h.T = static_cast<int>(T);
  h.grid = grid;
  h.steps_off = static_cast<int>(w.steps_off);
  h.maps_off = static_cast<int>(w.maps_off);
  h.counters_off = static_cast<int>(w.counters_off);
  std::memcpy(buf.data(), &h, sizeof(h));
  int map = 0;
  for (int s = 0; s < nsteps; ++s) {
    const qlin_w4a16_step& in = steps[s];
    DcStep d = {};
    d.x = static_cast<const __half*>(in.x);
    d.K = static_cast<int>(in.K);
    d.G = d.K / 128;
    d.zpitch = (d.G + 1) / 2;
    d.nchunks = (d.G + kDcChunkGroups - 1) / kDcChunkGroups;
    d.chunk_u64 = std::min(kDcChunkU64, d.K / 16);
    d.map0 = map;
    int units = 0;
    d.np = 0;
    for (int p = 0; p < in.count; ++p) {
      if (in.N[p] == 0) continue;  // an empty matrix takes no tiles
      const int q = d.np++;
      d.scales[q] = static_cast<const __half*>(in.scales[p]);
      d.zeros[q] = in.zeros[p];
      d.y[q] = static_cast<__half*>(in.y[p]);
      d.N[q] = static_cast<int>(in.N[p]);
      units += (d.N[q] + kDcUnit - 1) / kDcUnit;
      d.unit_end[q] = units;
      CUtensorMap tm;
      cudaError_t e = make_tmap_2d_u64(&tm, in.wq[p], static_cast<uint64_t>(in.K / 16),
                                       static_cast<uint64_t>(in.N[p]), static_cast<uint32_t>(d.chunk_u64), kDcUnit);
      if (e != cudaSuccess) return e;
      std::memcpy(buf.data() + w.maps_off + static_cast<int64_t>(map) * sizeof(CUtensorMap), &tm, sizeof(tm));
      ++map;
    }
    d.units = units;
    std::memcpy(buf.data() + w.steps_off + static_cast<int64_t>(s) * sizeof(DcStep), &d, sizeof(d));
  }
  // the counters are zero in the buffer; the kernel leaves them zero after a
  // run that completes
  unsigned char* dst = static_cast<unsigned char*>(workspace);
  DcBlob* blob = new (std::nothrow) DcBlob;
  if (blob == nullptr) return cudaErrorMemoryAllocation;
  cudaError_t e = cudaSuccess;
  for (int64_t off = 0; off < w.total && e == cudaSuccess; off += kDcBlobBytes) {
    const int n = static_cast<int>(std::min<int64_t>(kDcBlobBytes, w.total - off));
    blob->dst = dst + off;
    blob->bytes = n;
    std::memcpy(blob->data, buf.data() + off, static_cast<size_t>(n));
    dc_blob_kernel<<<(n + 1023) / 1024, 256, 0, stream>>>(*blob);
    e = cudaGetLastError();
  }
  delete blob;
  return e;
}

cudaError_t w4a16_decode_run(const void* workspace, int nsteps, int64_t T, cudaStream_t stream) {
  const int NT = T <= 8 ? 1 : 2;
  cudaError_t e = dc_set_attr(NT);
  if (e != cudaSuccess) return e;
  int S = dc_stages(NT);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sm_count());
  cfg.blockDim = dim3((dc_warps(NT) + 1) * 32);
  cfg.dynamicSmemBytes = dc_layout(NT, S).total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const unsigned char* ws = static_cast<const unsigned char*>(workspace);
  int Ti = static_cast<int>(T);
  int32_t* err = device_error_word();
  void* args[] = {&ws, &nsteps, &Ti, &S, &err};
  return cudaLaunchKernelExC(&cfg, dc_kernel(NT), args);
}

}  // namespace qlin
