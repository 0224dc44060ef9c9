// W4A16 decode: a sequence of GEMV steps in one persistent launch.
//
// A decoder runs its linears one after another at T = 1, each reading what
// an earlier one wrote.  Launched one by one, consecutive layers overlap only
// through the two CTA slots of an SM, and the block scheduler fills those
// slots as the previous layer's CTAs leave, which places two CTAs of one
// layer on a third of the SMs and none on another third, every layer.  Here
// one cooperative launch with exactly one CTA per SM runs the whole sequence:
//
//   - a step's matrices (e.g. q, k and v) are one band of concatenated rows,
//     split evenly over the CTAs, so every SM carries the same share of every
//     step;
//   - warp 12 (one elected thread) streams the CTA's bands, step after step,
//     into a ring of shared-memory slots with 1-D bulk copies: the rows'
//     codes, and 16-byte windows of their fp16 scales and packed zero-points
//     (one copy per matrix a stage's rows fall in).  It never waits on
//     another CTA: while a step still finishes on other SMs, this SM's slots
//     already fill with the next steps' weights;
//   - warp 13 turns each landed stage's raw scales and zero-points into one
//     packed word per (row, group), fp16 scale bits | zero-point << 16, the
//     form the dot-product code reads;
//   - the compute warps finish a step, store its outputs, and arrive on that
//     step's counter in global memory (release); before the next step, one
//     thread waits until every CTA has arrived (acquire) and brings the
//     step's activations into shared memory with one bulk copy, from which
//     every warp builds its chunk's fixed-point planes.
//
// The arithmetic of a row is the one of the single-launch GEMV (the same
// chunk dot products and the same tree of cross-lane and cross-warp
// additions), so every output equals the single-launch result bit for bit.
// Every wait is bounded: on expiry the kernel records the site in the device
// error word and stops, and every other CTA's bounded waits end the same way.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "device_common.cuh"
#include "qlin_internal.h"
#include "tc_common.cuh"
#include "w4a16_gemv_common.cuh"

namespace qlin {
namespace {

using namespace gv;

constexpr int kSqMaxSteps = 128;                              // steps per launch
constexpr int kSqMaxGroup = QLIN_W4A16_MAX_GROUP;
constexpr int kSqWarps = 12;                                  // compute warps (K <= 12 . 1024)
constexpr int kSqProducerWarp = kSqWarps, kSqConverterWarp = kSqWarps + 1;
constexpr int kSqThreads = (kSqWarps + 2) * 32;
constexpr int kSqB = 8;                                       // rows per batch per row group
constexpr int kSqMaxSlots = 16;
constexpr int kSqSmemMax = 227 * 1024;
constexpr int kSqSiteFull = 1, kSqSiteEmpty = 2, kSqSiteDrain = 3, kSqSiteGrid = 4, kSqSiteRaw = 5;

struct SqStep {
  const __half* x;
  const uint8_t* wq[kSqMaxGroup];
  const __half* scales[kSqMaxGroup];
  const uint8_t* zeros[kSqMaxGroup];  // nullptr: symmetric, z = 8
  __half* y[kSqMaxGroup];
  int row_end[kSqMaxGroup];           // matrix p: step rows [row_end[p-1], row_end[p])
  int np, N, K, RG;                   // matrices, rows, K, row groups (WPR = K / 1024 rounded up)
};

struct SqArgs {
  SqStep st[kSqMaxSteps];
  int nsteps;
  int S, slot_bytes, off_red, off_x, off_bar;
  unsigned int* grid_bar;  // [nsteps] arrival counters, zero at launch
  int32_t* err;
};

// Slot layout of a step with R rows per stage: codes, packed {scale, zero}
// words, then the raw scale and zero-point windows (per matrix segment, each
// window 16-byte aligned and up to 30 bytes wider than its rows).
struct SqSlot {
  int pk, rs, rz, need;
};
__host__ __device__ inline SqSlot sq_slot(int R, int K) {
  const int G = K / 128, zpitch = (G + 1) / 2;
  SqSlot l;
  l.pk = R * (K / 2);
  l.rs = l.pk + R * G * 4;
  l.rz = l.rs + (R * G * 2 + 15) / 16 * 16 + 32 * kSqMaxGroup;
  l.need = l.rz + (R * zpitch + 15) / 16 * 16 + 32 * kSqMaxGroup;
  return l;
}

__device__ __forceinline__ int sq_matrix(const SqStep& st, int r, int& first) {
  int p = 0;
#pragma unroll
  for (int i = 0; i < kSqMaxGroup - 1; ++i)
    if (i < st.np - 1 && r >= st.row_end[i]) p = i + 1;
  first = p > 0 ? st.row_end[p - 1] : 0;
  return p;
}

// Even split of n items over `parts`: start and count of part i.
__device__ __forceinline__ void sq_split(int n, int parts, int i, int& start, int& count) {
  const int base = n / parts, extra = n % parts;
  start = i * base + min(i, extra);
  count = base + (i < extra ? 1 : 0);
}

// Segment k (matrix boundaries) of stage rows [row, row + rows): the rows
// and the raw windows of their scales and zero-points, with the offsets of
// the windows in the slot's raw areas.
struct SqSeg {
  int row, rows, p, first;
  uintptr_t sc_lo, z_lo;
  uint32_t sc_bytes, z_bytes;
  int sc_at, z_at;        // slot-area offsets of the windows
};
__device__ __forceinline__ bool sq_segment(const SqStep& st, int row, int rows, int k, int G, int zpitch, SqSeg& sg) {
  int done = 0, sc_at = 0, z_at = 0;
  for (int i = 0; done < rows; ++i) {
    const int r = row + done;
    int first;
    const int p = sq_matrix(st, r, first);
    const int seg = min(rows - done, st.row_end[p] - r);
    const uintptr_t sc = reinterpret_cast<uintptr_t>(st.scales[p] + static_cast<int64_t>(r - first) * G);
    const uintptr_t sc_lo = sc & ~uintptr_t(15);
    const uint32_t sc_bytes =
        static_cast<uint32_t>(((sc + static_cast<uintptr_t>(seg) * G * 2 + 15) & ~uintptr_t(15)) - sc_lo);
    uintptr_t z_lo = 0;
    uint32_t z_bytes = 0;
    if (st.zeros[p]) {
      const uintptr_t z = reinterpret_cast<uintptr_t>(st.zeros[p] + static_cast<int64_t>(r - first) * zpitch);
      z_lo = z & ~uintptr_t(15);
      z_bytes = static_cast<uint32_t>(((z + static_cast<uintptr_t>(seg) * zpitch + 15) & ~uintptr_t(15)) - z_lo);
    }
    if (i == k) {
      sg.row = r;
      sg.rows = seg;
      sg.p = p;
      sg.first = first;
      sg.sc_lo = sc_lo;
      sg.z_lo = z_lo;
      sg.sc_bytes = sc_bytes;
      sg.z_bytes = z_bytes;
      sg.sc_at = sc_at;
      sg.z_at = z_at;
      return true;
    }
    sc_at += static_cast<int>(sc_bytes);
    z_at += static_cast<int>(z_bytes);
    done += seg;
  }
  return false;
}

// Named barrier with an OR over the threads' predicates: every thread gets the
// same answer, so decisions taken after it cannot diverge across warps.
__device__ __forceinline__ bool named_sync_or(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(unsigned int* p, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__global__ void __launch_bounds__(kSqThreads, 1) w4a16_seq_kernel(const __grid_constant__ SqArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.S;
  const uint32_t ring = tc::smem_u32(smem);
  const uint32_t bar0 = tc::smem_u32(smem + a.off_bar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + a.off_bar + 24 * S);
  float* red = reinterpret_cast<float*>(smem + a.off_red);
  auto full = [&](int s) { return bar0 + 8u * s; };            // codes landed and scales packed
  auto empty = [&](int s) { return bar0 + 8u * (S + s); };     // compute warps done with the slot
  auto raw = [&](int s) { return bar0 + 8u * (2 * S + s); };   // raw scale / zero windows landed
  const uint32_t x_full = bar0 + 24u * S + 8u;                 // the step's activations
  const uint32_t xs = tc::smem_u32(smem + a.off_x);
  const int grid = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(full(s), 2);     // producer (code bytes) + converter
      tc::mbar_init(empty(s), kSqWarps);
      tc::mbar_init(raw(s), 1);
    }
    tc::mbar_init(x_full, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();

  if (warp == kSqProducerWarp) {
    // ---------------- producer: the CTA's bands of every step ----------------
    if (lane == 0) {
      const uint64_t policy = tc::l2_policy_evict_first();
      int g = 0;
      bool stop = false;
      for (int s = 0; s < a.nsteps && !stop; ++s) {
        const SqStep& st = a.st[s];
        const int K = st.K, G = K / 128, row_bytes = K / 2, zpitch = (G + 1) / 2, R = kSqB * st.RG;
        const SqSlot L = sq_slot(R, K);
        int r0, nrows;
        sq_split(st.N, grid, cta, r0, nrows);
        const int nst = (nrows + R - 1) / R;
        for (int i = 0; i < nst; ++i, ++g) {
          const int slot = g % S;
          if (g >= S && !tc::mbar_wait_sleep(empty(slot), ((g / S) - 1) & 1, a.err, kSqSiteEmpty, 128)) *abort_flag = 1;
          if (*abort_flag) {
            stop = true;
            break;
          }
          int off, rows_i;
          sq_split(nrows, nst, i, off, rows_i);
          const int row = r0 + off;
          const uint32_t dst = ring + slot * a.slot_bytes;
          uint32_t raw_bytes = 0;
          SqSeg sg;
          for (int k = 0; sq_segment(st, row, rows_i, k, G, zpitch, sg); ++k) raw_bytes += sg.sc_bytes + sg.z_bytes;
          tc::mbar_arrive_expect_tx(raw(slot), raw_bytes);
          tc::mbar_arrive_expect_tx(full(slot), static_cast<uint32_t>(rows_i * row_bytes));
          for (int k = 0; sq_segment(st, row, rows_i, k, G, zpitch, sg); ++k) {
            tc::bulk_load(dst + L.rs + sg.sc_at, reinterpret_cast<const void*>(sg.sc_lo), sg.sc_bytes, raw(slot));
            if (sg.z_bytes)
              tc::bulk_load(dst + L.rz + sg.z_at, reinterpret_cast<const void*>(sg.z_lo), sg.z_bytes, raw(slot));
            tc::bulk_load_policy(dst + (sg.row - row) * row_bytes,
                                 st.wq[sg.p] + static_cast<int64_t>(sg.row - sg.first) * row_bytes,
                                 static_cast<uint32_t>(sg.rows * row_bytes), full(slot), policy);
          }
        }
      }
      // copies still in flight must land before the CTA exits
      for (int j = max(0, g - S); j < g; ++j) {
        tc::mbar_wait(raw(j % S), (j / S) & 1, a.err, kSqSiteDrain);
        tc::mbar_wait(full(j % S), (j / S) & 1, a.err, kSqSiteDrain);
      }
    }
    return;
  }

  if (warp == kSqConverterWarp) {
    // ---------------- converter: raw scales / zeros -> packed words ----------------
    int g = 0;
    bool stop = false;
    for (int s = 0; s < a.nsteps && !stop; ++s) {
      const SqStep& st = a.st[s];
      const int K = st.K, G = K / 128, zpitch = (G + 1) / 2, R = kSqB * st.RG;
      const SqSlot L = sq_slot(R, K);
      int r0, nrows;
      sq_split(st.N, grid, cta, r0, nrows);
      const int nst = (nrows + R - 1) / R;
      for (int i = 0; i < nst; ++i, ++g) {
        const int slot = g % S;
        bool ok = tc::mbar_wait_sleep(raw(slot), (g / S) & 1, a.err, kSqSiteRaw, 64);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          *abort_flag = 1;
          stop = true;
          break;
        }
        int off, rows_i;
        sq_split(nrows, nst, i, off, rows_i);
        const int row = r0 + off;
        unsigned char* base = smem + slot * a.slot_bytes;
        uint32_t* pk = reinterpret_cast<uint32_t*>(base + L.pk);
        SqSeg sg;
        for (int k = 0; sq_segment(st, row, rows_i, k, G, zpitch, sg); ++k) {
          const uintptr_t sc = reinterpret_cast<uintptr_t>(st.scales[sg.p] + static_cast<int64_t>(sg.row - sg.first) * G);
          const unsigned char* rs = base + L.rs + sg.sc_at + (sc - sg.sc_lo);
          const unsigned char* rz = nullptr;
          if (sg.z_bytes) {
            const uintptr_t z =
                reinterpret_cast<uintptr_t>(st.zeros[sg.p] + static_cast<int64_t>(sg.row - sg.first) * zpitch);
            rz = base + L.rz + sg.z_at + (z - sg.z_lo);
          }
          uint32_t* pr = pk + (sg.row - row) * G;
          for (int r = 0; r < sg.rows; ++r, rs += 2 * G, pr += G) {
            for (int gg = lane; gg < G; gg += 32) {
              const uint32_t sv = *reinterpret_cast<const unsigned short*>(rs + 2 * gg);
              const uint32_t zv = rz ? (rz[r * zpitch + (gg >> 1)] >> ((gg & 1) * 4)) & 0xFu : 8u;
              pr[gg] = sv | (zv << 16);
            }
          }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(full(slot));  // release: the packed words are visible to waiters
      }
    }
    return;
  }

  // ---------------- compute warps ----------------
  const int nct = kSqWarps * 32;
  int slot = 0;          // ring position and phase of the next stage, kept
  uint32_t phase = 0;    // incrementally (no division by S in the loop)
  for (int s = 0; s < a.nsteps; ++s) {
    const SqStep& st = a.st[s];
    const int K = st.K, G = K / 128, KC = K / 32, row_bytes = K / 2;
    const int WPR = (KC + 31) / 32, RG = st.RG, R = kSqB * RG;
    const SqSlot L = sq_slot(R, K);
    const int rg = warp / WPR, wr = warp - rg * WPR;
    const bool active = rg < RG;  // warps past RG row groups idle in this step
    const int j = wr * 32 + lane;
    const bool act = active && j < KC;
    const int jc = min(j, KC - 1);

    // The activations of step s > 0 come from earlier steps: wait until every
    // CTA has stored step s - 1.
    if (s > 0) {
      bool failed = false;
      if (threadIdx.x == 0) {
        const unsigned int* cnt = a.grid_bar + (s - 1);
        if (ld_acquire_gpu(cnt) < static_cast<unsigned int>(grid)) {
          const long long t0 = clock64();
          while (ld_acquire_gpu(cnt) < static_cast<unsigned int>(grid)) {
            if (clock64() - t0 > tc::kWaitTimeoutCycles || *abort_flag) {
              record_device_error(a.err, kDevErrTimeoutBase + kSqSiteGrid);
              failed = true;
              *abort_flag = 1;
              break;
            }
          }
        }
      }
      if (named_sync_or(1, nct, failed)) break;
    }
    // the step's activations into shared memory, one bulk copy (the async
    // proxy reads what other CTAs stored through the generic proxy)
    if (threadIdx.x == 0) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      tc::mbar_arrive_expect_tx(x_full, static_cast<uint32_t>(K * 2));
      tc::bulk_load(xs, st.x, static_cast<uint32_t>(K * 2), x_full);
    }
    {
      bool xok = tc::mbar_wait(x_full, s & 1, a.err, kSqSiteFull);
      xok = __all_sync(0xffffffffu, xok);
      if (named_sync_or(1, nct, !xok)) {
        *abort_flag = 1;
        break;
      }
    }
    GvX X;
    gv_load_x_smem(xs, j, act, X);

    int r0, nrows;
    sq_split(st.N, grid, cta, r0, nrows);
    const int nst = (nrows + R - 1) / R;
    const int st_base = nst ? nrows / nst : 0, st_extra = nst ? nrows % nst : 0;  // even split into stages
    bool ok = true;
    {
      float prev[kSqB];
      int prev_row0 = -1, prev_rows = 0;
      auto reduce_store = [&](const float* v, int row0, int rows) {
        float k;
        const int row_sel = gv_reduce_batch<kSqB>(v, lane, k);
        if (lane < kSqB) {
          const int rr = rg + RG * row_sel;
          if (rr < rows) red[(row0 + rr) * WPR + wr] = k;
        }
      };
      for (int i = 0, off = 0; i < nst; ++i) {
        bool ready = tc::mbar_wait(full(slot), phase, a.err, kSqSiteFull);
        ready = __all_sync(0xffffffffu, ready);
        if (!ready) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        const int rows_i = st_base + (i < st_extra ? 1 : 0);
        float p[kSqB];
        if (active) {
          const uint32_t base = ring + slot * a.slot_bytes;
          gv_batch<kSqB>(base + jc * 16, base + L.pk + (jc >> 2) * 4, rows_i, RG, rg, row_bytes, G, X.xp, X.xsum,
                         X.sx, p);
        }
        // the stage is in registers: hand the slot back
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(empty(slot));
        if (++slot == S) {
          slot = 0;
          phase ^= 1u;
        }
        if (active) {
          if (prev_row0 >= 0) reduce_store(prev, prev_row0, prev_rows);
#pragma unroll
          for (int b = 0; b < kSqB; ++b) prev[b] = p[b];
          prev_row0 = off;
          prev_rows = rows_i;
        }
        off += rows_i;
      }
      if (active && prev_row0 >= 0) reduce_store(prev, prev_row0, prev_rows);
    }
    if (named_sync_or(1, nct, !ok)) break;
    // outputs of this step: the warps' partial sums of each row, in order
    for (int r = threadIdx.x; r < nrows; r += nct) {
      float v = 0.0f;
      for (int w = 0; w < WPR; ++w) v += red[r * WPR + w];
      int first;
      const int p = sq_matrix(st, r0 + r, first);
      st.y[p][r0 + r - first] = __float2half_rn(v);
    }
    named_sync(1, nct);  // stores done (and red free for the next step)
    if (s + 1 < a.nsteps && threadIdx.x == 0) red_release_gpu_add(a.grid_bar + s, 1u);
  }
}

// Grid-barrier counters of the no-allocation entry point: one per step of a
// launch, zeroed by the launch's memset.  Launches that use them must not run
// at the same time.
static __device__ __align__(256) unsigned int g_seq_counters[kSqMaxSteps];

constexpr int kSqMaxDevices = 64;
std::mutex g_seq_mutex;
unsigned int* g_seq_counter_addr[kSqMaxDevices] = {};  // device address of g_seq_counters, per device
std::atomic<int> g_seq_smem_set[kSqMaxDevices];         // largest dynamic shared memory granted, per device

// The launch arguments are built in a per-thread host buffer (about 22 KB),
// so a launch allocates nothing on the host either; cudaLaunchKernelEx copies
// them before it returns.
thread_local SqArgs t_sq_args;

}  // namespace

cudaError_t w4a16_sequence_static_workspace(unsigned int** out) {
  *out = nullptr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kSqMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_seq_mutex);
  if (g_seq_counter_addr[dev] == nullptr) {
    // In host code g_seq_counters names a host-side stand-in, not device
    // memory: the kernel must be given the address the runtime reports for
    // this device.
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_seq_counters);
    if (e != cudaSuccess) return e;
    g_seq_counter_addr[dev] = static_cast<unsigned int*>(p);
  }
  *out = g_seq_counter_addr[dev];
  return cudaSuccess;
}

int64_t w4a16_sequence_workspace_bytes(int64_t nsteps) { return (nsteps * 4 + 255) / 256 * 256; }

bool w4a16_sequence_supported(int64_t K) { return K > 0 && K % 128 == 0 && K <= 12288; }

// Raises the kernel's dynamic shared-memory limit on the current device when
// a launch needs more than any earlier one did (one attribute call per new
// maximum instead of one per launch).
static cudaError_t sq_allow_smem(int smem) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kSqMaxDevices)
    return cudaFuncSetAttribute(w4a16_seq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (g_seq_smem_set[dev].load(std::memory_order_acquire) >= smem) return cudaSuccess;
  std::lock_guard<std::mutex> lock(g_seq_mutex);
  if (g_seq_smem_set[dev].load(std::memory_order_relaxed) >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(w4a16_seq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) g_seq_smem_set[dev].store(smem, std::memory_order_release);
  return e;
}

cudaError_t launch_w4a16_sequence(const W4A16SeqStep* steps, int nsteps, unsigned int* workspace,
                                  cudaStream_t stream) {
  const int grid = sm_count();
  for (int s0 = 0; s0 < nsteps; s0 += kSqMaxSteps) {
    const int ns = std::min(kSqMaxSteps, nsteps - s0);
    SqArgs* a = &t_sq_args;
    *a = SqArgs{};
    int slot = 0, red_floats = 0, kmax = 0;
    for (int s = 0; s < ns; ++s) {
      const W4A16SeqStep& in = steps[s0 + s];
      SqStep& st = a->st[s];
      const int K = static_cast<int>(in.K);
      const int WPR = (K / 32 + 31) / 32;
      st.x = static_cast<const __half*>(in.x);
      st.K = K;
      st.RG = kSqWarps / WPR;
      st.np = 0;
      int64_t rows = 0;
      for (int p = 0; p < in.count; ++p) {
        if (in.N[p] == 0) continue;  // an empty matrix takes no rows
        rows += in.N[p];
        st.wq[st.np] = in.wq[p];
        st.scales[st.np] = static_cast<const __half*>(in.scales[p]);
        st.zeros[st.np] = in.zeros[p];
        st.y[st.np] = static_cast<__half*>(in.y[p]);
        st.row_end[st.np] = static_cast<int>(rows);
        ++st.np;
      }
      st.N = static_cast<int>(rows);
      slot = std::max(slot, sq_slot(kSqB * st.RG, K).need);
      red_floats = std::max(red_floats, static_cast<int>((rows + grid - 1) / grid) * WPR);
      kmax = std::max(kmax, K);
    }
    a->nsteps = ns;
    a->slot_bytes = (slot + 127) / 128 * 128;
    const int red_bytes = (red_floats * 4 + 15) / 16 * 16;
    const int x_bytes = kmax * 2;  // a multiple of 256
    const int S = std::min(kSqMaxSlots, (kSqSmemMax - red_bytes - x_bytes - 24 * kSqMaxSlots - 16) / a->slot_bytes);
    if (S < 2) return cudaErrorInvalidValue;
    a->S = S;
    a->off_red = S * a->slot_bytes;
    a->off_x = a->off_red + red_bytes;
    a->off_bar = a->off_x + x_bytes;
    const int smem = a->off_bar + 24 * S + 16;
    a->grid_bar = workspace;
    a->err = device_error_word();
    cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(unsigned int) * ns, stream);
    if (e == cudaSuccess) e = sq_allow_smem(smem);
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(grid);
      cfg.blockDim = dim3(kSqThreads);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeCooperative;
      attr[0].val.cooperative = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, w4a16_seq_kernel, *a);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace qlin
