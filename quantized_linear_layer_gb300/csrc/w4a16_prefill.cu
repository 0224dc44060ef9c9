// W4A16 beyond decode (prefill, many tokens): Y = X . W^T with uint4 g128
// weights dequantized on the fly, on the tcgen05 tensor cores.
//
//   Y[t, n] = sum_k X[t, k] . ((q[n, k] - z[n, k / 128]) . s[n, k / 128])
//
// ("LLM and AIGC quantization: from number formats to W4A4", W4A16: the
// weights stay 4-bit in memory and are dequantized to fp16 next to the
// tensor cores, which multiply in fp16 and accumulate in fp32.)  Each weight
// is rounded once to fp16 after its scale, (q - z) . s, with (q - z) exact.
//
// Design for GB300.  The weight tile is the MMA's A operand and is read from
// tensor memory: dequantized in registers and written with tcgen05.st, so
// only the packed codes (half a byte per weight) pass through shared memory.
// The activations are the B operand, copied by TMA straight into the
// 128-byte swizzled K-major layout the MMA reads.  One CTA per SM walks
// 128 (weight rows) x BN (tokens) output tiles; a K stage of 128 is one
// quantization group, so each row needs one scale and one zero-point per
// stage.  BN = 256 for many tokens: with 128 x 128 tiles the kernel ran its
// kind::f16 MMAs at about half the rate (0.40-0.48 of the bf16 peak against
// 0.65-0.77).  BN = 128 when the tiles are fewer than the SMs: a stage then
// holds 40 instead of 72 KB, so the ring is five stages deep instead of
// three, a stage is half the MMA work, and there are twice the tiles to
// spread over the SMs (the 256-token stages of a 65-token problem were
// latency-bound at 30% tensor-pipe activity).
//
//   warp 0       TMA producer: per stage the activation tile (BN tokens x
//                128 K, two 64-element K blocks) and the packed codes
//                (128 rows x 64 bytes in the 64-byte swizzle, 8 KB) into the
//                ring.
//   warp 1       TMEM allocation and the MMA issuer: 8 x tcgen05.mma
//                kind::f16 (M = 128, N = BN, K = 16, A from TMEM) per stage
//                into one BN-column fp32 accumulator.
//   warps 2-9    dequantizers, two sets of four taking alternate stages: lane
//                l of the warp with TMEM lane quadrant q owns weight row
//                32q + l, turns its 128 codes of the stage into 64 fp16 pairs
//                and stores them into an A ring in TMEM (64 columns per
//                stage); the scale and zero-point of its next stage are
//                loaded while it works on the current one.
//   warps 10-17  epilogue: two warps per lane quadrant; lane l of quadrant q
//                owns weight row 32q + l and writes its BN / 2 tokens of the
//                tile, 32 at a time (only the tokens that exist), then frees
//                the accumulator.
// TMEM columns: [0, BN) the accumulator, then the A ring.
// Few tiles (few tokens): a cluster of two (or, with BN = 128, four) CTAs
// shares each tile, each taking an equal share of K.  Rank q % split owns
// the outputs of TMEM lane quadrant q: the other ranks push their shares of
// those rows (the columns that hold tokens) into its free stage buffers
// through distributed shared memory, and it adds the shares in rank order
// and stores them, so every rank of the cluster receives, adds and stores
// an equal part (one rank receiving everything took longer than the MMAs).
// Every barrier wait is bounded; on expiry the kernel records the site in the
// device error word, stops issuing work, waits (bounded) for copies and MMAs
// already in flight, frees TMEM and exits.
#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "device_common.cuh"
#include "qlin_internal.h"
#include "tc_common.cuh"
#include "tmap.h"
#include "w4a16_mma_common.cuh"

namespace qlin {
namespace {

constexpr int kPfBM = 128;                          // weight rows per tile (MMA M)
constexpr int kPfBK = 128;                          // K per stage: one quantization group
constexpr int kPfTmemCols = 512;
constexpr int kPfSets = 2;                          // dequantizer sets of four warps
constexpr int kPfWarpA0 = 2, kPfWarpE0 = kPfWarpA0 + 4 * kPfSets;
constexpr int kPfEpiWarps = 8;                      // two per TMEM lane quadrant
constexpr int kPfThreads = (kPfWarpE0 + kPfEpiWarps) * 32;
constexpr int kPfWBytes = kPfBM * kPfBK / 2;        // 8 KB of packed codes per stage

// The plan of a tile width BN (tokens per tile, the MMA's N).
template <int BN>
struct PfCfg {
  static constexpr int kStg = BN == 256 ? 3 : 5;              // shared-memory stages
  static constexpr int kOpsA = BN == 256 ? 3 : 4;             // TMEM stages of dequantized weights
  static constexpr int kXBytes = BN * kPfBK * 2;              // fp16 activations per stage
  static constexpr int kStgBytes = kXBytes + kPfWBytes;       // 72 or 40 KB
  static constexpr int kTmemA = BN;                           // A ring after the accumulator
  static constexpr int kSmemBar = kStg * kStgBytes;
  static constexpr int kNumBars = 2 * kStg + 2 * kOpsA + 7;
  static constexpr int kSmemMisc = kSmemBar + kNumBars * 8;
  static constexpr int kSmemTotal = kSmemMisc + 16 + 1024;    // + alignment slack
  static constexpr int kMaxSplit = BN == 256 ? 2 : 4;         // partners' accumulators fit the stage area
  static_assert(BN == 128 || BN == 256, "tile widths");
  static_assert(kSmemTotal <= 227 * 1024, "shared memory budget");
  static_assert(kTmemA + kOpsA * (kPfBK / 2) <= kPfTmemCols, "TMEM budget");
  static_assert(kStgBytes % 1024 == 0, "stages keep the 1024-byte alignment of the swizzled tiles");
  // a split rank's stage area holds 8 shares of 32 rows x BN / 2 tokens in
  // fp32 (its slots), then the shares it sends: 2 (4 - 4 / split)
  static_assert((8 + 2 * (4 - 4 / kMaxSplit)) * (32 * (BN / 2) * 4) <= kStg * kStgBytes,
                "the exchanged shares fit the stage area");
};

enum { kPfSiteStgEmpty = 1, kPfSiteStgFull, kPfSiteAEmpty, kPfSiteAFull, kPfSiteAccEmpty, kPfSiteAccFull,
       kPfSiteDrain, kPfSiteRedReady, kPfSiteRedData };

// A bounded wait (about a second) on a local mbarrier that a CTA of the
// cluster arrives on with release semantics.
__device__ __forceinline__ bool pf_wait_cluster(uint32_t bar, uint32_t parity, int32_t* err, int site) {
  for (int i = 0; i < 1000; ++i)
    if (w4mma::mbar_try_wait_cluster(bar, parity)) return true;
  record_device_error(err, kDevErrTimeoutBase + site);
  return false;
}

// Eight codes of one word (element k + i in bits 4i .. 4i+3) -> four words of
// fp16 pairs ((k, k+1), (k+2, k+3), ...), each (q - z) . s rounded once.
// Byte j of the word holds the pair; one byte permute copies it into both
// halves and one mask leaves the low nibble in the low half's mantissa and
// the high nibble four bits up in the high half's, under fp16 1024 (0x6400):
// 1024 + q and 1024 + 16 q, both exact.  One fma with (1, 1/16) and
// (-(1024 + z), -(64 + z)) gives q - z in both halves, exactly; one multiply
// by s rounds.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t mul, uint32_t add, __half2 s2, uint32_t* out) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t t = __byte_perm(w, 0u, 0x4040u + 0x0101u * j);
    const uint32_t v = (t & 0x00F0000Fu) | 0x64006400u;
    const __half2 d = __hfma2(*reinterpret_cast<const __half2*>(&v), *reinterpret_cast<const __half2*>(&mul),
                              *reinterpret_cast<const __half2*>(&add));
    const __half2 r = __hmul2(d, s2);
    out[j] = *reinterpret_cast<const uint32_t*>(&r);
  }
}

// Output tile `tile` in the persistent order: groups of 8 weight-row tiles
// walk the token tiles together (operand tiles shared through L2).
__device__ __forceinline__ void pf_tile_coords(int tile, int mt_count, int nt_count, int& mt, int& nt) {
  constexpr int kGroup = 8;
  const int per_group = kGroup * nt_count;
  const int grp = tile / per_group;
  const int first_m = grp * kGroup;
  const int rows = min(kGroup, mt_count - first_m);
  const int in = tile - grp * per_group;
  mt = first_m + in % rows;
  nt = in / rows;
}

// 32-column groups of the epilogue warps of token half h of tile column nt
// that hold tokens.
template <int BN>
__device__ __forceinline__ int pf_groups(int T, int nt, int h) {
  const int t0 = nt * BN + h * (BN / 2);
  return T <= t0 ? 0 : min(BN / 64, (T - t0 + 31) / 32);
}

template <int BN>
__global__ void __launch_bounds__(kPfThreads, 1) w4a16_prefill_kernel(const __grid_constant__ CUtensorMap tmX,
                                                                      const __grid_constant__ CUtensorMap tmW,
                                                                      const __half* __restrict__ scales,
                                                                      const uint8_t* __restrict__ zeros, int T,
                                                                      int N, int K, __half* __restrict__ y,
                                                                      int split, int32_t* __restrict__ err) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  pdl_launch_dependents();  // the next layer may start setting up (it waits for this grid before reading Y)
  using Cfg = PfCfg<BN>;
  constexpr int kPfStg = Cfg::kStg, kPfOpsA = Cfg::kOpsA, kPfStgBytes = Cfg::kStgBytes, kPfXBytes = Cfg::kXBytes;
  constexpr int kPfTmemA = Cfg::kTmemA, kPfSmemBar = Cfg::kSmemBar, kPfSmemMisc = Cfg::kSmemMisc;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt_count = (N + kPfBM - 1) / kPfBM, nt_count = (T + BN - 1) / BN;
  const int tiles = mt_count * nt_count;
  // split > 1: a cluster of `split` CTAs shares one tile, each taking an equal
  // share of K (in rank order); the accumulators of ranks 1.. are added to
  // rank 0's through distributed shared memory before the store.  Otherwise
  // CTAs are persistent over the tiles.
  const uint32_t rank = split > 1 ? w4mma::cluster_rank() : 0u;
  const int tile0 = static_cast<int>(blockIdx.x) / split;
  const int tstride = split > 1 ? tiles : static_cast<int>(gridDim.x);
  const int my_tiles = tile0 < tiles ? (split > 1 ? 1 : (tiles - tile0 + tstride - 1) / tstride) : 0;
  const int num_kb = K / kPfBK;
  const int kb_begin = static_cast<int>(rank) * num_kb / split;
  const int kb_count = (static_cast<int>(rank) + 1) * num_kb / split - kb_begin;
  const int G = K / 128, zpitch = (G + 1) / 2;

  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t bar0 = sbase + kPfSmemBar;
  auto stg_full = [&](int s) { return bar0 + 8u * s; };
  auto stg_empty = [&](int s) { return bar0 + 8u * (kPfStg + s); };
  auto a_full = [&](int o) { return bar0 + 8u * (2 * kPfStg + o); };
  auto a_empty = [&](int o) { return bar0 + 8u * (2 * kPfStg + kPfOpsA + o); };
  auto acc_full = [&](int b) { return bar0 + 8u * (2 * kPfStg + 2 * kPfOpsA + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (2 * kPfStg + 2 * kPfOpsA + 2 + b); };
  const uint32_t mma_done = bar0 + 8u * (2 * kPfStg + 2 * kPfOpsA + 4);
  const uint32_t red_ready = mma_done + 8u;  // every other rank's stage buffers are free
  const uint32_t red_data = mma_done + 16u;  // the other ranks' shares of this rank's quadrants have landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kPfSmemMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kPfSmemMisc + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPfStg; ++s) {
      tc::mbar_init(stg_full(s), 1);
      tc::mbar_init(stg_empty(s), 1 + 4);  // the MMA commit and the stage's four dequantizer warps
    }
    for (int o = 0; o < kPfOpsA; ++o) {
      tc::mbar_init(a_full(o), 4);
      tc::mbar_init(a_empty(o), 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(acc_full(b), 1);
      tc::mbar_init(acc_empty(b), kPfEpiWarps);
    }
    tc::mbar_init(mma_done, 1);
    // red_ready: one arrival per epilogue warp of every other rank; red_data:
    // this thread's arrival with the bytes of the shares the other ranks send
    // (a split CTA has one tile, known here)
    tc::mbar_init(red_ready, (split > 1 ? split - 1 : 1) * kPfEpiWarps);
    tc::mbar_init(red_data, 1);
    if (split > 1 && my_tiles > 0) {
      int mt0, nt0;
      pf_tile_coords(tile0, mt_count, nt_count, mt0, nt0);
      const int groups = pf_groups<BN>(T, nt0, 0) + pf_groups<BN>(T, nt0, 1);
      tc::mbar_arrive_expect_tx(red_data, static_cast<uint32_t>((split - 1) * (4 / split) * groups * 4096));
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tc::smem_u32(tmem_slot), kPfTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (split > 1) w4mma::cluster_sync_all();  // every CTA's barriers exist before any remote arrive

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tc::prefetch_tmap(&tmX);
      tc::prefetch_tmap(&tmW);
      pdl_wait();  // the activations may come from the previous kernel in the stream
      int it = 0, issued = 0;
      for (int ti = 0; ti < my_tiles && !*abort_flag; ++ti) {
        int mt, nt;
        pf_tile_coords(tile0 + ti * tstride, mt_count, nt_count, mt, nt);
        for (int kbi = 0; kbi < kb_count; ++kbi, ++it) {
          const int kb = kb_begin + kbi;
          const int s = it % kPfStg;
          if (it >= kPfStg && !tc::mbar_wait(stg_empty(s), ((it / kPfStg) - 1) & 1, err, kPfSiteStgEmpty)) {
            *abort_flag = 1;
            break;
          }
          if (*abort_flag) break;
          const uint32_t dst = sbase + s * kPfStgBytes;
          tc::mbar_arrive_expect_tx(stg_full(s), kPfStgBytes);
          tc::tma_load_2d(dst, &tmX, kb * kPfBK * 2, nt * BN, stg_full(s));
          tc::tma_load_2d(dst + kPfXBytes / 2, &tmX, kb * kPfBK * 2 + 128, nt * BN, stg_full(s));
          tc::tma_load_2d(dst + kPfXBytes, &tmW, kb * kPfBK / 2, mt * kPfBM, stg_full(s));
          issued = it + 1;
        }
      }
      if (*abort_flag) {
        for (int j = (issued > kPfStg ? issued - kPfStg : 0); j < issued; ++j)
          tc::mbar_wait(stg_full(j % kPfStg), (j / kPfStg) & 1, err, kPfSiteDrain);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_f16(kPfBM, BN, 0);  // fp16 x fp16 -> fp32
      bool issued_any = false;
      int it = 0;
      for (int ti = 0; ti < my_tiles && !*abort_flag; ++ti) {
        const int buf = 0;
        // the epilogue has written out the previous tile
        if (ti >= 1 && !tc::mbar_wait(acc_empty(buf), (ti - 1) & 1, err, kPfSiteAccEmpty)) {
          *abort_flag = 1;
          break;
        }
        tc::tc_fence_after();
        for (int kbi = 0; kbi < kb_count; ++kbi, ++it) {
          const int s = it % kPfStg, o = it % kPfOpsA;
          if (!tc::mbar_wait(a_full(o), (it / kPfOpsA) & 1, err, kPfSiteAFull) ||
              !tc::mbar_wait(stg_full(s), (it / kPfStg) & 1, err, kPfSiteStgFull)) {
            *abort_flag = 1;
            break;
          }
          if (*abort_flag) break;
          tc::tc_fence_after();
          const uint32_t xb = sbase + s * kPfStgBytes;
          const uint32_t a_t = tmem + kPfTmemA + o * (kPfBK / 2);
#pragma unroll
          for (int k = 0; k < kPfBK / 16; ++k) {
            const uint32_t b_k = xb + (k >> 2) * (BN * 128) + 32 * (k & 3);  // K block, then 32 B in the atom
            tc::mma_f16_ta(tmem + buf * BN, a_t + 8 * k, tc::sw128_kmajor_desc(b_k), idesc,
                           (kbi > 0 || k > 0) ? 1u : 0u);
          }
          issued_any = true;
          tc::mma_commit(a_empty(o));
          tc::mma_commit(stg_empty(s));
        }
        if (*abort_flag) break;
        tc::mma_commit(acc_full(buf));
      }
      if (*abort_flag && issued_any) {
        tc::mma_commit(mma_done);
        tc::mbar_wait(mma_done, 0, err, kPfSiteDrain);
      }
    }
  } else if (warp < kPfWarpE0) {
    // ---------------- dequantizers (codes -> fp16 weights in TMEM) ----------------
    const int set = (warp - kPfWarpA0) >> 2;  // takes the stages with it % kPfSets == set
    const int q = warp & 3;                   // TMEM lane quadrant of this warp
    const int r = q * 32 + lane;              // weight row of the tile
    pdl_wait();                               // scales and zero-points, like every input
    // Stage i of this CTA is K block kb_begin + i % kb_count of its tile
    // i / kb_count (kb_count = num_kb unless the tile is split).  The
    // scale and zero-point of the set's next stage are loaded while the
    // current stage is dequantized, so their latency stays off the chain.
    const int total = my_tiles * kb_count;
    auto load_sz = [&](int i, __half& sc, uint32_t& z) {
      sc = __ushort_as_half(0);  // rows past N dequantize to 0
      z = 0;
      if (i >= total) return;
      int mt, nt;
      pf_tile_coords(tile0 + (i / kb_count) * tstride, mt_count, nt_count, mt, nt);
      const int n = mt * kPfBM + r, kb = kb_begin + i % kb_count;
      if (n < N) {
        sc = scales[static_cast<int64_t>(n) * G + kb];
        z = zeros != nullptr ? (zeros[static_cast<int64_t>(n) * zpitch + (kb >> 1)] >> (4 * (kb & 1))) & 0xFu : 8u;
      }
    };
    __half sc_next;
    uint32_t z_next;
    load_sz(set, sc_next, z_next);
    for (int it = set; it < total; it += kPfSets) {
      const __half sc = sc_next;
      const uint32_t z = z_next;
      load_sz(it + kPfSets, sc_next, z_next);
      const int s = it % kPfStg, o = it % kPfOpsA;
      bool ok = tc::mbar_wait(stg_full(s), (it / kPfStg) & 1, err, kPfSiteStgFull);
      if (ok && it >= kPfOpsA) ok = tc::mbar_wait(a_empty(o), ((it / kPfOpsA) - 1) & 1, err, kPfSiteAEmpty);
      ok = __all_sync(0xffffffffu, ok && !*abort_flag);  // lanes agree and reconverge
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      tc::tc_fence_after();
      {
        const uint32_t mul = 0x2C003C00u;                          // (1, 1/16)
        const uint32_t add = 0xD400E400u | (z << 20) | z;          // (-(1024 + z), -(64 + z))
        const __half2 s2 = __half2half2(sc);
        // the codes arrive in the 64-byte swizzle: 16-byte chunk c of row r sits
        // at chunk c ^ ((r / 2) % 4), so the eight rows of a quarter warp hit
        // distinct banks
        const uint32_t src = sbase + s * kPfStgBytes + kPfXBytes + r * (kPfBK / 2);
        const int swz = (r >> 1) & 3;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t v[32];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint4 u = tc::lds128(src + (((2 * h + c) ^ swz) << 4));
            dequant_word(u.x, mul, add, s2, v + 16 * c);
            dequant_word(u.y, mul, add, s2, v + 16 * c + 4);
            dequant_word(u.z, mul, add, s2, v + 16 * c + 8);
            dequant_word(u.w, mul, add, s2, v + 16 * c + 12);
          }
          tc::tmem_st_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + kPfTmemA + o * (kPfBK / 2) + 32 * h,
                                 v);
        }
        tc::tmem_wait_st();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(a_full(o));
          tc::mbar_arrive(stg_empty(s));
        }
      }
    }
  } else {
    // ---------------- epilogue ----------------
    constexpr int kHalf = BN / 2;              // tokens of a warp
    constexpr int kShare = 32 * kHalf * 4;     // a warp's rows x tokens in fp32
    constexpr int kRecv = 8 * kShare;          // an owner's slots: (owned quadrant, rank, half)
    const int q = warp & 3;                    // TMEM lane quadrant this warp may access
    const int half = (warp - kPfWarpE0) >> 2;  // token half of the tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16) + half * kHalf;
    // split > 1: rank q % split owns the outputs of quadrant q; every other
    // rank stages its share of those rows in its own shared memory and sends
    // it with one bulk copy into the owner's slots, and the owner adds all
    // shares in rank order
    const int owner = split > 1 ? q % split : 0;
    // (32-column group cg, row `lane`, 16-byte chunk c4) within a share: each
    // group's 32 rows are 4 KB in one piece, chunks rotated by row (no bank
    // conflicts)
    auto share_off = [&](int cg, int c4) { return static_cast<uint32_t>(((cg * 32 + lane) * 8 + (c4 ^ (lane & 7))) * 16); };
    auto slot = [&](int src) { return static_cast<uint32_t>((((q / split) * split + src) * 2 + half) * kShare); };
    int qi = 0;  // index of this quadrant among those the rank sends
    for (int qq = 0; qq < q; ++qq) qi += (qq % split != static_cast<int>(rank)) ? 1 : 0;
    const uint32_t staging = static_cast<uint32_t>(kRecv + (qi * 2 + half) * kShare);
    for (int ti = 0; ti < my_tiles; ++ti) {
      const int buf = 0;
      bool ok = tc::mbar_wait(acc_full(buf), ti & 1, err, kPfSiteAccFull);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      tc::tc_fence_after();
      int mt, nt;
      pf_tile_coords(tile0 + ti * tstride, mt_count, nt_count, mt, nt);
      const int row = q * 32 + lane;  // weight row within the tile
      const int tw0 = nt * BN + half * kHalf;
      const int ncg = pf_groups<BN>(T, nt, half);  // the warp's 32-column groups that hold tokens
      const uint32_t tcol0 = lane_base + buf * BN;
      bool partners = false;
      if (split > 1) {
        // every MMA of this CTA is done: its stage buffers may take the shares
        // of the quadrants it owns
        __syncwarp();
        if (lane == 0)
          for (int p = 0; p < split; ++p)
            if (p != static_cast<int>(rank)) w4mma::mbar_arrive_cluster(w4mma::map_to_rank(red_ready, p));
        // this rank's share of quadrant q into its staging area (a sender) or
        // into its own slot (the owner)
        const uint32_t dst = sbase + (owner != static_cast<int>(rank) ? staging : slot(static_cast<int>(rank)));
#pragma unroll 1
        for (int cg = 0; cg < ncg; ++cg) {
          __syncwarp();
          uint32_t v[32];
          tc::tmem_ld_32x32b_x32(tcol0 + cg * 32, v);
          tc::tmem_wait_ld();
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4)
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst + share_off(cg, c4)), "r"(v[4 * c4]),
                         "r"(v[4 * c4 + 1]), "r"(v[4 * c4 + 2]), "r"(v[4 * c4 + 3])
                         : "memory");
        }
        if (owner != static_cast<int>(rank)) {
          // send it once the owner's stage buffers are free
          tc::fence_proxy_async_smem();
          bool go = pf_wait_cluster(red_ready, 0, err, kPfSiteRedReady);
          go = __all_sync(0xffffffffu, go);
          if (go && ncg > 0 && lane == 0)
            tc::bulk_copy_to_cluster(w4mma::map_to_rank(sbase + slot(static_cast<int>(rank)), owner), dst,
                                     static_cast<uint32_t>(ncg) * 4096u, w4mma::map_to_rank(red_data, owner));
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(acc_empty(buf));
          continue;
        }
        partners = pf_wait_cluster(red_data, 0, err, kPfSiteRedData);
        partners = __all_sync(0xffffffffu, partners);
      }
      // Y[t][n]: the warp's 32 lanes hold 32 consecutive n of each token t, so
      // every store instruction writes 64 contiguous bytes
      const int n = mt * kPfBM + row;
      unsigned short* yr = reinterpret_cast<unsigned short*>(y) + n;
#pragma unroll 1
      for (int cg = 0; cg < ncg; ++cg) {
        __syncwarp();  // reconverge after the bound checks before the aligned TMEM load
        uint32_t v[32];
        if (!partners) {
          tc::tmem_ld_32x32b_x32(tcol0 + cg * 32, v);
          tc::tmem_wait_ld();
        } else {
          // the shares of ranks 0, 1, ... added in that order
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const uint4 a = tc::lds128(sbase + slot(0) + share_off(cg, c4));
            v[4 * c4] = a.x; v[4 * c4 + 1] = a.y; v[4 * c4 + 2] = a.z; v[4 * c4 + 3] = a.w;
          }
#pragma unroll 1
          for (int src = 1; src < split; ++src) {
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const uint4 o = tc::lds128(sbase + slot(src) + share_off(cg, c4));
              v[4 * c4] = __float_as_uint(__fadd_rn(__uint_as_float(v[4 * c4]), __uint_as_float(o.x)));
              v[4 * c4 + 1] = __float_as_uint(__fadd_rn(__uint_as_float(v[4 * c4 + 1]), __uint_as_float(o.y)));
              v[4 * c4 + 2] = __float_as_uint(__fadd_rn(__uint_as_float(v[4 * c4 + 2]), __uint_as_float(o.z)));
              v[4 * c4 + 3] = __float_as_uint(__fadd_rn(__uint_as_float(v[4 * c4 + 3]), __uint_as_float(o.w)));
            }
          }
        }
        const int t0 = tw0 + cg * 32;
        if (n < N) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int t = t0 + i;
            if (t < T) yr[static_cast<int64_t>(t) * N] = __half_as_ushort(__float2half_rn(__uint_as_float(v[i])));
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(acc_empty(buf));
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  // no CTA of a cluster leaves while another may still touch its shared
  // memory (every wait above is bounded, so all threads get here)
  if (split > 1) w4mma::cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kPfTmemCols);
  }
}

}  // namespace

bool w4a16_prefill_supported(int64_t T, int64_t N, int64_t K) {
  return T >= 1 && N >= 1 && K >= kPfBK && K % kPfBK == 0 && T <= (1 << 30) && N <= (1 << 30);
}

// Launch plan: the tile width (tokens per tile) and the number of CTAs that
// share a tile's K, the one with the least estimated time: waves of tiles x
// stages per CTA x the measured time of a stage (about 0.62 us at 128 tokens
// and 0.74 us at 256), plus about 2 us for the exchange of a split tile.  A
// split runs every cluster at once (split x tiles CTAs at most the SMs);
// unsplit tiles run on persistent CTAs.
struct PfPlan {
  int bn, split;
};
PfPlan pf_plan(int64_t T, int64_t N, int64_t K) {
  const int64_t sms = sm_count();
  const int64_t mt = (N + kPfBM - 1) / kPfBM, num_kb = K / kPfBK;
  PfPlan best = {256, 1};
  double best_cost = 1e30;
  for (int bn : {256, 128}) {
    const int64_t tiles = mt * ((T + bn - 1) / bn);
    const double stage = bn == 256 ? 0.74 : 0.62;
    const int max_split = bn == 256 ? PfCfg<256>::kMaxSplit : PfCfg<128>::kMaxSplit;
    for (int s = 1; s <= max_split; s *= 2) {
      if (s > 1 && (s * tiles > sms || num_kb < s)) continue;
      const int64_t waves = s > 1 ? 1 : (tiles + sms - 1) / sms;
      const double cost = static_cast<double>(waves * ((num_kb + s - 1) / s)) * stage + (s > 1 ? 2.0 : 0.0);
      if (cost < best_cost) {
        best_cost = cost;
        best = {bn, s};
      }
    }
  }
  return best;
}

template <int BN>
cudaError_t launch_prefill_bn(const CUtensorMap& tmX, const CUtensorMap& tmW, const void* scales,
                              const uint8_t* zeros, int64_t T, int64_t N, int64_t K, void* y, int split,
                              cudaStream_t stream) {
  using Cfg = PfCfg<BN>;
  // the shared-memory attribute, set once per device
  static std::once_flag once[64];
  static cudaError_t attr_status[64];
  int dev = 0;
  cudaError_t st = cudaGetDevice(&dev);
  if (st != cudaSuccess) return st;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [&] {
    attr_status[dev] = cudaFuncSetAttribute(w4a16_prefill_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            Cfg::kSmemTotal);
  });
  if (attr_status[dev] != cudaSuccess) return attr_status[dev];
  const int64_t tiles = ((N + kPfBM - 1) / kPfBM) * ((T + BN - 1) / BN);
  const int grid = split > 1 ? static_cast<int>(split * tiles) : static_cast<int>(tiles < sm_count() ? tiles : sm_count());
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPfThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemTotal;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = split;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = split > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, w4a16_prefill_kernel<BN>, tmX, tmW, static_cast<const __half*>(scales), zeros,
                            static_cast<int>(T), static_cast<int>(N), static_cast<int>(K), static_cast<__half*>(y),
                            split, device_error_word());
}

cudaError_t launch_w4a16_prefill(const void* x, int64_t T, int64_t N, int64_t K, const uint8_t* wq,
                                 const void* scales, const uint8_t* zeros, void* y, cudaStream_t stream) {
  if (T == 0 || N == 0) return cudaSuccess;
  const PfPlan plan = pf_plan(T, N, K);
  CUtensorMap tmX, tmW;
  cudaError_t st = make_tmap_2d_u8(&tmX, x, static_cast<uint64_t>(K) * 2, static_cast<uint64_t>(T), 128, plan.bn,
                                   /*swizzle_bytes=*/128);
  if (st != cudaSuccess) return st;
  st = make_tmap_2d_u8(&tmW, wq, static_cast<uint64_t>(K) / 2, static_cast<uint64_t>(N), kPfBK / 2, kPfBM,
                       /*swizzle_bytes=*/64);
  if (st != cudaSuccess) return st;
  if (plan.bn == 256) return launch_prefill_bn<256>(tmX, tmW, scales, zeros, T, N, K, y, plan.split, stream);
  return launch_prefill_bn<128>(tmX, tmW, scales, zeros, T, N, K, y, plan.split, stream);
}

}  // namespace qlin
