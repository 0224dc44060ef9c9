/*
 * qlin.h - C ABI of the GB300 (sm_103a) quantized linear layer library.
 *
 * Y = X . W^T with dequantization fused into the matrix product, in three
 * forms:
 *   - W4A16: group-wise (g = 128) unsigned 4-bit weights with fp16 scales and
 *     4-bit zero-points, fp16 activations, fp16 output.
 *   - W8A8: per-token int8 activations (symmetric, or asymmetric with an
 *     integer zero-point), per-channel symmetric int8 weights, int32
 *     accumulation, fused epilogue s_a . s_b . (D^ - azp . azp_adj) + bias.
 *   - NVFP4 W4A4: E2M1 values in 16-element blocks with E4M3 block scales and
 *     an fp32 per-tensor scale, optionally with ARCQuant residual channels
 *     appended along K.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory: every pointer argument is a DEVICE pointer (cudaMalloc / a torch
 *   CUDA tensor) unless stated otherwise.  The caller owns all memory.  The
 *   library allocates nothing, keeps no pointer after it returns and has no
 *   state except one device error word per device (see qlin_get_device_error).
 * Layout: all matrices are row-major with dense rows (row pitch = number of
 *   columns x element size).  W is [N][K] (nn.Linear.weight layout, K
 *   contiguous); X and Y are [T][K] and [T][N].  4-bit codes are packed two
 *   per byte along the row: element 2i in the low nibble of byte i.
 * Alignment: every base pointer must be 16-byte aligned and every row pitch a
 *   multiple of 16 bytes (checked; QLIN_ERR_ALIGNMENT otherwise).
 * Streams: work is enqueued on `stream` (0 = legacy default stream).  No
 *   entry point synchronizes, except qlin_get_device_error.
 * Errors: arguments are checked on the host before anything is launched; a
 *   failed check launches nothing.  A failed launch returns QLIN_ERR_CUDA.
 *   Nothing is thrown across the ABI and nothing aborts.  The text of the last
 *   failure on the calling thread is available from qlin_last_error_message.
 * Device: the current device must be compute capability 10.3 (GB300);
 *   anything else returns QLIN_ERR_UNSUPPORTED.
 * Empty problems (T == 0 or N == 0) are valid and launch nothing.
 *
 * Sources: the method is restated from five web pages (a CUDA engineering
 * book chapter on quantization kernels; "CUDA-Practice 07"; "LLM and AIGC
 * quantization: from number formats to W4A4"; "vLLM W8A8 quantized GEMM:
 * CUTLASS epilogue design"; "NVFP4 quantization and ARCQuant").  Each entry
 * point cites the passage that defines its operation.
 */
#ifndef QLIN_H_
#define QLIN_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  QLIN_OK = 0,
  QLIN_ERR_INVALID_ARG = 1, /* a size, pointer or option is out of range        */
  QLIN_ERR_ALIGNMENT = 2,   /* a base pointer or row pitch is not 16-byte aligned */
  QLIN_ERR_UNSUPPORTED = 3, /* wrong GPU, or an option this build does not cover */
  QLIN_ERR_CUDA = 4,        /* a CUDA runtime call or a kernel launch failed     */
  QLIN_ERR_TIMEOUT = 5      /* a kernel gave up a bounded wait (device error word) */
} qlin_status;

typedef enum {
  QLIN_F16 = 0,
  QLIN_BF16 = 1,
  QLIN_F32 = 2,
  QLIN_I32 = 3
} qlin_dtype;

typedef enum {
  /* activations: append the NVFP4 re-quantized residual of the first S
     (reordered) channels */
  QLIN_NVFP4_RESIDUAL = 0,
  /* weights: append a copy of the codes and scales of the first S
     (reordered) channels */
  QLIN_NVFP4_DUPLICATE = 1
} qlin_nvfp4_mode;

typedef enum {
  /* row-major [rows][K/16], one E4M3 byte per 16-element block */
  QLIN_SF_ROWS = 0,
  /* the layout the tensor core reads: rows in tiles of 128, 64-element K
     blocks in groups of 4 scales; block (rt, kg) is 512 contiguous bytes at
     ((rt * K/64 + kg) * 512), holding row rt*128 + r, scale 4*kg + j at byte
     16*(r%32) + 4*(r/32) + j.  Size ceil(rows/128) * K/64 * 512 bytes. */
  QLIN_SF_MMA = 1
} qlin_sf_layout;

typedef enum {
  QLIN_QFMT_INT8 = 0,     /* symmetric int8, codes in [-127, 127], s = max|y| / 127 */
  QLIN_QFMT_FP8_E4M3 = 1  /* E4M3-FN codes, s = max|y| / 448 */
} qlin_qfmt;

/* Online Hadamard rotations (qlin_hadamard). */
typedef enum {
  QLIN_HADAMARD_SYLVESTER = 0,  /* fast Walsh-Hadamard butterflies, n a power of two */
  QLIN_HADAMARD_REGULAR = 1     /* Kronecker power of the 4 x 4 regular Hadamard H4, n a power of four */
} qlin_hadamard_kind;

/* MX element formats (one E8M0 scale per 32 elements along K). */
typedef enum {
  QLIN_MX_FP8_E4M3 = 0,  /* MXFP8: E4M3-FN elements, one byte each */
  QLIN_MX_FP4_E2M1 = 1   /* MXFP4: E2M1 elements, two per byte (element 2i in the low nibble) */
} qlin_mx_fmt;

/* Human-readable name of a status code (static storage, never NULL). */
const char* qlin_status_string(qlin_status status);

/* Text of the last failure reported on the calling thread (static per-thread
   storage; empty string if none). */
const char* qlin_last_error_message(void);

/* Library ABI version (major * 100 + minor). */
int qlin_version(void);

/* Reads and clears the device error word of the current device.  Kernels that
   wait on barriers give up after a bounded time and record a nonzero code
   there instead of hanging.  Synchronizes `stream` first.  *code_out (host
   pointer, may be NULL) receives the raw code (0 = none).  Returns
   QLIN_ERR_TIMEOUT if a code was set, QLIN_OK otherwise. */
qlin_status qlin_get_device_error(cudaStream_t stream, int32_t* code_out);

/* ------------------------------------------------------------------------
 * a0 - W4A16 weight preparation (offline, at load time)
 *
 * Asymmetric unsigned 4-bit group quantization of W [N][K], one scale and one
 * zero-point per `group` consecutive K elements of a row, following the AWQ
 * offline flow ("LLM and AIGC quantization", AWQ section, pseudo_quant):
 *   s = fp16( max(max_g w - min_g w, 1e-5) / 15 )   (float32 ops, RNE to fp16)
 *   z = clamp(rint(-min_g w / s), 0, 15)
 *   q = clamp(rint(w / s) + z, 0, 15)
 * with s the fp16-rounded scale (the value dequantization uses).
 *   w       [N][K] of w_dtype (F32, F16 or BF16)
 *   group   128 (the only group size of this build; else QLIN_ERR_UNSUPPORTED)
 *   wq      out, uint8 [N][K/2], packed codes
 *   scales  out, fp16 [N][K/group]
 *   zeros   out, uint8 [N][ceil(K/group / 2)], packed zero-points
 * K must be a multiple of `group`; the zero-point and scale rows are dense
 * (their row pitch need not be 16-byte aligned).
 * ---------------------------------------------------------------------- */
qlin_status qlin_quant_w4_g128(const void* w, qlin_dtype w_dtype, int64_t N, int64_t K, int64_t group,
                               uint8_t* wq, void* scales, uint8_t* zeros, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * a1 - W4A16 fused dequant GEMV / skinny GEMM
 *
 * Y[t,n] = sum_g s[n,g] . sum_{k in g} X[t,k] . (q[n,k] - z[n,g])
 * ("Chapter 9 - Quantization kernels", section 9.5 dequant-fused GEMM and
 * 9.6 INT4 unpack; "LLM and AIGC quantization", section W4A16).  The 4-bit
 * codes are unpacked in registers with the zero-point folded into the
 * conversion; products are exact and accumulate in fp32; the group scale is
 * applied once per group in fp32; Y is rounded once to fp16.
 *   x       fp16 [T][K]
 *   wq      uint8 [N][K/2] packed codes (element 2i in the low nibble)
 *   scales  fp16 [N][K/group]
 *   zeros   uint8 [N][ceil(K/group / 2)] packed zero-points, or NULL meaning
 *           the symmetric zero-point 8 for every group
 *   group   128
 *   y       out, fp16 [T][N]
 * K a multiple of `group`; any T >= 0.  Up to 16 tokens run the decode /
 * skinny kernels above.  More tokens (prefill) run a tcgen05 GEMM
 * ("LLM and AIGC quantization", W4A16: dequantize next to the tensor cores,
 * fp16 multiply, fp32 accumulate).  That GEMM rounds each weight once to
 * fp16, (q - z) . s with (q - z) exact, before the fp32 accumulation.
 * Bit stability: a given (x, W) always gives the same bits at the same T on
 * the same device.  Prefill outputs may differ in the last bit between token
 * counts or devices with another SM count: when the output tiles are few,
 * two or four CTAs share K and their fp32 partial sums are added in a fixed
 * order, a different rounding order from the unsplit sum (both within the
 * tolerance).
 * ---------------------------------------------------------------------- */
qlin_status qlin_w4a16_gemm(const void* x, int64_t T, int64_t N, int64_t K, const uint8_t* wq,
                            const void* scales, const uint8_t* zeros, int64_t group, void* y,
                            cudaStream_t stream);

/* ------------------------------------------------------------------------
 * a1, grouped - several W4A16 linears of the same input in one call
 *
 * Y_p = X . dequant(W_p)^T for p = 0 .. count-1, every W_p with the same K:
 * the q, k and v projections of a decoder block, or its gate and up
 * projections, which all read the same activations.  At T = 1 a single GEMV
 * launch covers the concatenated rows of all count matrices, so the group
 * waits once on the kernel that produced X instead of once per matrix; for
 * T > 1 (or a concatenation too large for one launch's plan) each matrix
 * runs as qlin_w4a16_gemm.  Each row is computed exactly as in a separate
 * qlin_w4a16_gemm call, so the results equal count separate calls bit for
 * bit.
 *   x       fp16 [T][K]
 *   count   1 .. QLIN_W4A16_MAX_GROUP
 *   N       host array [count], rows of each W_p (0 allowed)
 *   wq, scales, zeros, y
 *           host arrays [count] of device pointers, each W_p and Y_p laid
 *           out as in qlin_w4a16_gemm (zeros[p] NULL: symmetric, z = 8)
 *   group   128
 * The host arrays are read during the call only.
 * ---------------------------------------------------------------------- */
#define QLIN_W4A16_MAX_GROUP 4
qlin_status qlin_w4a16_gemm_grouped(const void* x, int64_t T, int64_t K, int count, const int64_t* N,
                                    const uint8_t* const* wq, const void* const* scales,
                                    const uint8_t* const* zeros, int64_t group, void* const* y,
                                    cudaStream_t stream);

/* Launch placement of the T = 1 GEMV on the current device.  Consecutive
   GEMV launches alternate between two launch shapes of one kernel (one
   holding more than half of an SM's registers, the other more than half of
   its shared memory), so that each layer's CTAs take one slot per SM beside
   the previous layer's; the shapes are derived from the device's limits and
   the kernel's register count, and every launch keeps the plain shape when
   they cannot be met (a slower placement, same results).
   *alternating (host pointer, may be NULL) receives 1 when the two shapes are
   in use, else 0; *registers (may be NULL) the kernel's registers per
   thread.  No launch, no synchronization. */
qlin_status qlin_w4a16_gemv_launch_info(int* alternating, int* registers);

/* ------------------------------------------------------------------------
 * next 3 - W4A16 with act-order (g_idx)
 *
 * With act-order ("LLM and AIGC quantization", GPTQ engineering details:
 * desc_act quantizes the columns in descending diag(H) order, and g_idx
 * records each input channel's group), column k of the weights uses the
 * scale and zero-point of group g_idx[k]:
 *   Y[t,n] = sum_k X[t,k] . (q[n,k] - z[n, g_idx[k]]) . s[n, g_idx[k]]
 *
 * qlin_w4a16_act_order_prepare (offline, once per weight):
 *   perm[j]       = the j-th column in group order (a stable sort by g_idx:
 *                   group 0's columns in ascending order, then group 1's ...)
 *   wq_sorted     = the codes with their columns in that order
 *   g_idx   int32 [K], each group in [0, K/group) holding exactly `group`
 *           columns (otherwise the device error word records a nonzero
 *           code: see qlin_get_device_error)
 *   wq      uint8 [N][K/2] packed codes in the original column order
 *   perm    out, int32 [K] (16-byte aligned); wq_sorted out, uint8 [N][K/2]
 *   scales / zeros stay as they are ([N][K/group], now per contiguous group).
 * qlin_w4a16_gemm_act_order (run time): x_work[t][j] = x[t][perm[j]] (one
 *   gather kernel), then qlin_w4a16_gemm(x_work, wq_sorted, scales, zeros);
 *   the sums are the same terms in another order.
 *   x, x_work  fp16 [T][K] (16-byte aligned; x_work is a caller workspace)
 *   other arguments as in qlin_w4a16_gemm; group 128; K <= 98304 (a row is
 *   staged in shared memory for the gather, QLIN_ERR_UNSUPPORTED above).
 * ---------------------------------------------------------------------- */
qlin_status qlin_w4a16_act_order_prepare(const int32_t* g_idx, int64_t K, int64_t group, const uint8_t* wq,
                                         int64_t N, int32_t* perm, uint8_t* wq_sorted, cudaStream_t stream);
qlin_status qlin_w4a16_gemm_act_order(const void* x, int64_t T, int64_t N, int64_t K, const int32_t* perm,
                                      const uint8_t* wq_sorted, const void* scales, const uint8_t* zeros,
                                      int64_t group, void* x_work, void* y, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * a1, sequence - a chain of W4A16 decode steps in one persistent launch
 *
 * Runs steps[0], steps[1], ... in order at T = 1, each step a grouped W4A16
 * linear (as qlin_w4a16_gemm_grouped) whose input may be an output of any
 * earlier step: the layers of a decoder at decode time.  One cooperative
 * launch keeps exactly one CTA on every SM; each CTA streams its share of
 * every step's weights into shared memory ahead of time, and a grid-wide
 * barrier in global memory separates the steps.  Every output equals the one
 * qlin_w4a16_gemm gives for the same step bit for bit.
 *   steps      host array [nsteps] (read during the call only):
 *                x        fp16 [K] device pointer, the step's input
 *                K        a multiple of 128, at most 12288
 *                count    1 .. QLIN_W4A16_MAX_GROUP matrices reading x
 *                N[p], wq[p], scales[p], zeros[p], y[p]
 *                         as in qlin_w4a16_gemm_grouped; a step's outputs
 *                         must not overlap its own x or one another (the
 *                         barrier between steps orders everything else: a
 *                         later step may overwrite what an earlier one read
 *                         or wrote)
 *   workspace  device memory of qlin_w4a16_sequence_workspace_bytes(nsteps)
 *              bytes, 4-byte aligned, owned by the caller (the grid
 *              barrier's counters); it must not be used by another
 *              sequence call in flight at the same time
 * The call enqueues a memset of the workspace and one launch per 128 steps
 * on `stream`.  Returns QLIN_ERR_UNSUPPORTED when the device cannot hold one
 * CTA per SM for the launch.
 * ---------------------------------------------------------------------- */
typedef struct {
  const void* x;
  int64_t K;
  int count;
  int64_t N[QLIN_W4A16_MAX_GROUP];
  const uint8_t* wq[QLIN_W4A16_MAX_GROUP];
  const void* scales[QLIN_W4A16_MAX_GROUP];
  const uint8_t* zeros[QLIN_W4A16_MAX_GROUP];
  void* y[QLIN_W4A16_MAX_GROUP];
} qlin_w4a16_step;

/* ------------------------------------------------------------------------
 * a1, chain - a decoder's W4A16 linears in one call, one launch per step
 *
 * Runs steps[0], steps[1], ... in order on `stream` at T tokens, each step
 * exactly as qlin_w4a16_gemm_grouped(steps[s].x, T, ...) (so the outputs equal
 * those calls bit for bit): the chain of dependent linears a decoder runs per
 * token ("Chapter 9 - Quantization kernels", 9.1: decode reads every weight
 * once per token).  Every step is checked before anything is launched, and
 * the launches follow one another with programmatic dependent launch as in
 * separate calls; one call instead of one per layer keeps the host's share of
 * a decode step small.
 *   steps   host array [nsteps] (read during the call only), as for
 *           qlin_w4a16_gemv_sequence; x of step s is fp16 [T][K_s] and each
 *           y[p] fp16 [T][N_p]; a step may read what an earlier step wrote
 *   T       tokens, 0 .. 2^31-1
 *   group   128
 * ---------------------------------------------------------------------- */
qlin_status qlin_w4a16_chain(const qlin_w4a16_step* steps, int nsteps, int64_t T, int64_t group,
                             cudaStream_t stream);

/* ------------------------------------------------------------------------
 * a1, decode plan - a decoder's W4A16 linears at 1 .. 16 tokens in one
 * persistent launch on the tensor cores
 *
 * The same steps as qlin_w4a16_chain, at T <= 16, as one launch with
 * exactly one CTA per SM ("Chapter 9 - Quantization kernels", 9.1: decode
 * reads every weight once per token; 9.5 / 9.7: dequantize in registers
 * right before the tensor core, weight rows as the MMA's M side).  Every CTA
 * streams its share of every step's weights in step order, so the copies of
 * a step are in flight while the step before it still computes; a counter
 * per step in the workspace orders the steps' compute.  Per output:
 *   Y[t,n] = sum_g s[n,g] . sum_{k in g} X[t,k] . (q[n,k] - z[n,g])
 * with exact fp16 (q - z), fp32 products and sums, one fp16 rounding; the
 * sums are taken in a fixed order (the same on every run), which differs
 * from qlin_w4a16_gemm's (equal within the tolerance, not bit for bit).
 *
 * qlin_w4a16_decode_workspace_bytes(nsteps): bytes of a workspace for up to
 *   nsteps steps (-1 for nsteps < 0).
 * qlin_w4a16_decode_prepare: checks the steps and writes the plan into the
 *   workspace with kernel launches on `stream` (no host synchronization):
 *   the step table, one TMA tensor map per matrix, zeroed counters.  The
 *   plan keeps the device pointers of the steps (x, wq, scales, zeros, y)
 *   and is valid as long as they are; prepare it again when they change, or
 *   after a run that left a code in the device error word.
 *     steps      host array [nsteps], read during the call only, as for
 *                qlin_w4a16_chain (x of step s fp16 [T][K_s], y[p] fp16
 *                [T][N_p]; a step may read what an earlier step wrote; a
 *                step's outputs must not overlap its own x)
 *     T          1 .. 16 (QLIN_ERR_UNSUPPORTED otherwise)
 *     group      128
 *     workspace  device memory of qlin_w4a16_decode_workspace_bytes(nsteps)
 *                bytes, 256-byte aligned, owned by the caller
 *   QLIN_ERR_UNSUPPORTED when a CTA's share of a step's scales and
 *   zero-points exceeds its 20 KB staging buffer (rows per SM x (K/64 +
 *   K/256) bytes: about 224 rows per SM, 34 k rows in all, at K = 4096), or,
 *   for K > 2048, a CTA's share exceeds 256 rows (its buffer of sums).
 * qlin_w4a16_decode_run: runs a prepared plan on `stream` (one cooperative
 *   launch).  nsteps and T must be the prepared ones (a mismatch is recorded
 *   in the device error word and nothing runs).  Two runs of one workspace
 *   must not overlap on the GPU (they share its counters); runs on one
 *   stream follow one another and are safe.
 * ---------------------------------------------------------------------- */
int64_t qlin_w4a16_decode_workspace_bytes(int64_t nsteps);
qlin_status qlin_w4a16_decode_prepare(const qlin_w4a16_step* steps, int nsteps, int64_t T, int64_t group,
                                      void* workspace, cudaStream_t stream);
qlin_status qlin_w4a16_decode_run(const void* workspace, int nsteps, int64_t T, cudaStream_t stream);

int64_t qlin_w4a16_sequence_workspace_bytes(int64_t nsteps);
qlin_status qlin_w4a16_gemv_sequence(const qlin_w4a16_step* steps, int nsteps, int64_t group, void* workspace,
                                     cudaStream_t stream);

/* The same sequence without any device memory from the caller.  The pages
   have no counterpart of this entry point; it exists for callers that cannot
   allocate device memory on the path that runs the decoder: an inference
   runtime that loads this library as a plugin and gives it no allocator or
   workspace, or a serving engine that reserved nearly all of HBM for weights
   and KV cache at start-up and lets nothing else call cudaMalloc (which may
   also synchronize the device, a stall a per-token loop cannot take).
   The grid barrier's counters live in a fixed array of 128 four-byte words
   inside the library (a static device variable, 512 bytes, which every GPU
   that loads the library holds until the process exits).
   - No allocation: the call makes no cudaMalloc or cudaFree and no other
     allocating call, on the device or on the host.
   - Size limit: every launch takes at most 128 steps, the array's size; a
     longer sequence runs as several launches on `stream`, one after another,
     each of which first zeroes (memset on `stream`) the counters it uses.
     So any nsteps is accepted, and no counter state carries over from an
     earlier call.
   - Set-up: the first call with a device current looks up the array's
     device address for that device (cudaGetSymbolAddress) and keeps it;
     make that first call before any stream capture begins.  A failed lookup
     returns QLIN_ERR_CUDA.
   - Sharing: all calls on a device share the one array.  Calls issued on
     one stream run one after another and are safe; two calls whose kernels
     can overlap on the GPU (different streams, or concurrently replayed
     graphs) race on the counters and give wrong results or a timeout in the
     device error word.  Such callers must use qlin_w4a16_gemv_sequence with
     a workspace each.
   Outputs equal qlin_w4a16_gemv_sequence's bit for bit. */
qlin_status qlin_w4a16_gemv_sequence_noalloc(const qlin_w4a16_step* steps, int nsteps, int64_t group,
                                             cudaStream_t stream);

/* ------------------------------------------------------------------------
 * b1 - per-token int8 activation quantization
 *
 * Symmetric (azp == NULL): s_t = max_k |x| / 127 (s_t = 1 for an all-zero
 *   row), q = clamp(rint(x / s_t), -127, 127)
 *   ("LLM and AIGC quantization", symmetric quantization, q_max = 2^(b-1)-1;
 *   per-token dynamic scales).
 * Asymmetric (azp != NULL): mn = min(min_k x, 0), mx = max(max_k x, 0),
 *   s_t = max(mx - mn, 1e-5) / 255, z_t = -128 - rint(mn / s_t),
 *   q = clamp(rint(x / s_t) + z_t, -128, 127); dequantization is
 *   s_t (q - z_t) ("vLLM W8A8 ... CUTLASS epilogue design", section 1:
 *   A = s_a (A^ - J z_a)).
 * All arithmetic is IEEE float32 division/subtraction, round-half-to-even.
 * Also used per output channel for the W8A8 weights (rows = N).
 *   x      [T][K] of x_dtype (F16, BF16 or F32)
 *   q      out, int8 [T][K]
 *   scale  out, float32 [T]
 *   azp    out, int32 [T], or NULL for the symmetric form
 * ---------------------------------------------------------------------- */
qlin_status qlin_quant_act_int8(const void* x, qlin_dtype x_dtype, int64_t T, int64_t K, int8_t* q,
                                float* scale, int32_t* azp, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * a0 - W8A8 zero-point adjustment (offline, at load time)
 *
 * azp_adj[n] = sum_k B^[n,k]  (1 . B^, the per-output-channel sum of the int8
 * weight codes; "vLLM W8A8 ... CUTLASS epilogue design", sections 2 and 5:
 * it depends on the weights only and is computed once at load time).
 *   b        int8 [N][K]
 *   azp_adj  out, int32 [N]
 * ---------------------------------------------------------------------- */
qlin_status qlin_int8_row_sum(const int8_t* b, int64_t N, int64_t K, int32_t* azp_adj, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * b2 + b3 - int8 GEMM with int32 accumulation and the fused epilogue
 *
 * D^ = A^ . B^^T (exact int32), then
 *   out = s_a . s_b . (D^ - azp . azp_adj) + bias      (one final rounding)
 * evaluated as float(D^ - azp . azp_adj) * s_b * s_a + bias in float32
 * ("vLLM W8A8 ... CUTLASS epilogue design", sections 2.1-2.4 and 3; "LLM
 * and AIGC quantization", W8A8 section).  The four epilogues:
 *   ScaledEpilogue            azp == NULL, azp_adj == NULL, bias == NULL
 *   ScaledEpilogueBias        azp == NULL, azp_adj == NULL, bias != NULL
 *   ScaledEpilogueAzp         azp == NULL, azp_adj != NULL (azp_adj already
 *                             holds z . (1 . B^), the per-tensor form)
 *   ScaledEpilogueAzpPerToken azp != NULL, azp_adj != NULL
 * A missing bias means 0.
 *   a          int8 [T][K]   (per-token quantized activations)
 *   b          int8 [N][K]   (per-channel symmetric weights)
 *   scale_a    float32 [scale_a_numel], scale_a_numel 1 or T
 *   scale_b    float32 [scale_b_numel], scale_b_numel 1 or N
 *   azp        int32 [T] or NULL
 *   azp_adj    int32 [N] or NULL (must be non-NULL when azp is non-NULL)
 *   bias       [N] of bias_dtype (F16, BF16 or F32) or NULL
 *   out        [T][N] of out_dtype: F16 or BF16; or I32, which writes the raw
 *              accumulator D^ and ignores the epilogue arguments (test hook)
 * K must be a multiple of 16.  GB300 has no int8 tensor-core MMA: the
 * contraction runs on the 16-bit tensor cores on exact fp16 copies of the
 * int8 codes, in K chunks whose partial sums are exact in fp32, converted to
 * int32 and added in int32, so D^ is bit-exact.
 * ---------------------------------------------------------------------- */
qlin_status qlin_w8a8_gemm(const int8_t* a, const int8_t* b, int64_t T, int64_t N, int64_t K,
                           const float* scale_a, int64_t scale_a_numel, const float* scale_b,
                           int64_t scale_b_numel, const int32_t* azp, const int32_t* azp_adj,
                           const void* bias, qlin_dtype bias_dtype, void* out, qlin_dtype out_dtype,
                           cudaStream_t stream);

/* ------------------------------------------------------------------------
 * a0 + b2 + b3 - the same W8A8 GEMM with the int8 weight codes stored as
 * exact fp16 values
 *
 * Because GB300's tensor cores have no int8 MMA, qlin_w8a8_gemm widens both
 * operands to fp16 on chip, and widening the weights through shared memory
 * on every tile is what bounds that kernel.  The weights are static, so they
 * can be widened once at load time instead: qlin_int8_to_f16 writes every
 * int8 code as the fp16 number of the same value (exact: |code| <= 128), and
 * qlin_w8a8_gemm_f16b reads B in that form straight into the MMA's operand
 * layout.  The arithmetic is unchanged: D^, and every output, equal those of
 * qlin_w8a8_gemm on the int8 codes bit for bit.  The trade is twice the
 * weight bytes in memory (2 N K instead of N K) for a faster GEMM where it
 * is bound by the tensor cores (many tokens); the activations stay int8.
 *   qlin_int8_to_f16:   src int8 [count] -> dst fp16 [count] (16-byte aligned)
 *   qlin_w8a8_gemm_f16b: as qlin_w8a8_gemm, with b16 fp16 [N][K] holding
 *                        the codes (16-byte aligned)
 * ---------------------------------------------------------------------- */
qlin_status qlin_int8_to_f16(const int8_t* src, int64_t count, void* dst, cudaStream_t stream);
qlin_status qlin_w8a8_gemm_f16b(const int8_t* a, const void* b16, int64_t T, int64_t N, int64_t K,
                                const float* scale_a, int64_t scale_a_numel, const float* scale_b,
                                int64_t scale_b_numel, const int32_t* azp, const int32_t* azp_adj,
                                const void* bias, qlin_dtype bias_dtype, void* out, qlin_dtype out_dtype,
                                cudaStream_t stream);

/* ------------------------------------------------------------------------
 * b1 + b2 + b3 - per-token int8 quantization and the W8A8 GEMM with both
 * operands' codes stored as exact fp16 values
 *
 * The same arithmetic again, with the activation codes in the fp16 form as
 * well: qlin_quant_act_int8_f16 computes exactly the codes, scales and
 * zero-points of qlin_quant_act_int8 and writes each code as the fp16
 * number of the same value; qlin_w8a8_gemm_f16 then runs the GEMM with both
 * tiles read by TMA straight into the MMA's operand layout (no widening on
 * chip, 128 x 256 output tiles, or 128 x 224 where that gives fewer rounds
 * of tiles on the SMs).  D^ and every output equal those of
 * qlin_w8a8_gemm on the int8 codes bit for bit.  The trade is 2 T K bytes of
 * activation codes instead of T K (written once, read from L2 by the tiles).
 *   qlin_quant_act_int8_f16: as qlin_quant_act_int8, q16 out fp16 [T][K]
 *                            (16-byte aligned)
 *   qlin_w8a8_gemm_f16:      as qlin_w8a8_gemm, with a16 fp16 [T][K] and b16
 *                            fp16 [N][K] holding the codes (16-byte aligned)
 * ---------------------------------------------------------------------- */
qlin_status qlin_quant_act_int8_f16(const void* x, qlin_dtype x_dtype, int64_t T, int64_t K, void* q16,
                                    float* scale, int32_t* azp, cudaStream_t stream);
qlin_status qlin_w8a8_gemm_f16(const void* a16, const void* b16, int64_t T, int64_t N, int64_t K,
                               const float* scale_a, int64_t scale_a_numel, const float* scale_b,
                               int64_t scale_b_numel, const int32_t* azp, const int32_t* azp_adj, const void* bias,
                               qlin_dtype bias_dtype, void* out, qlin_dtype out_dtype, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * c0 - NVFP4 calibration helpers (offline / set-up)
 *
 * qlin_nvfp4_global_scale: g = max |x| / (6 . 448) over the whole tensor, the
 *   per-tensor fp32 scale that puts every block scale in E4M3 range.
 *   x [rows][K] of x_dtype; g out, float32 [1] (device).
 * qlin_arc_perm: ARCQuant channel order ("NVFP4 quantization and ARCQuant",
 *   section 2.1: channels reordered by descending magnitude): perm[i] = the
 *   channel with the i-th largest max over rows of |x|, ties by ascending
 *   channel index.  x [rows][K] of x_dtype; perm out, int32 [K].  K <= 16384.
 * ---------------------------------------------------------------------- */
qlin_status qlin_nvfp4_global_scale(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, float* g,
                                    cudaStream_t stream);
qlin_status qlin_arc_perm(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, int32_t* perm,
                          cudaStream_t stream);

/* ------------------------------------------------------------------------
 * c1 - NVFP4 quantization with ARCQuant residual channels
 *
 * Per row, over the reordered channels xs = x[:, perm] (perm NULL = identity),
 * per 16-element block b ("LLM and AIGC quantization", block-scaled formats,
 * the NVFP4 example; "NVFP4 quantization and ARCQuant", sections 2.1, 3.1):
 *   sf_b = E4M3( (max_b |xs| / 6) / g )          (RNE, saturating at 448)
 *   d_b  = dec(sf_b) . g
 *   q    = E2M1( xs / d_b )                      (RNE ties-to-even; 0 if d_b == 0)
 * then, for the first S reordered channels, columns K .. K+S-1 hold
 *   mode RESIDUAL:  NVFP4 of r = xs - e2m1(q) . d_b (float32), same g
 *   mode DUPLICATE: a copy of the codes and scales of columns 0 .. S-1
 *   x      [rows][K] of x_dtype (F16, BF16 or F32)
 *   perm   int32 [K] permutation of 0..K-1, or NULL
 *   S      0 <= S <= K, a multiple of 16
 *   g      float32 [1] device scalar
 *   q      out, uint8 [rows][(K+S)/2]  packed E2M1 codes
 *   sf     out, E4M3 block scales in sf_layout: QLIN_SF_ROWS [rows][(K+S)/16]
 *          (row pitch need not be 16-byte aligned), or QLIN_SF_MMA, the
 *          layout qlin_nvfp4_gemm reads (K+S a multiple of 64; bytes of the
 *          padding rows are left unwritten)
 * K and K+S must be multiples of 32 (so packed rows are 16-byte aligned).
 * ---------------------------------------------------------------------- */
qlin_status qlin_quant_nvfp4(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, const int32_t* perm,
                             int64_t S, qlin_nvfp4_mode mode, const float* g, uint8_t* q, uint8_t* sf,
                             qlin_sf_layout sf_layout, cudaStream_t stream);

/* Bytes of a scale-factor buffer for `rows` rows of K elements in the given
   layout (-1 if K is not a multiple of 16, or of 64 for QLIN_SF_MMA). */
int64_t qlin_nvfp4_sf_bytes(int64_t rows, int64_t K, qlin_sf_layout sf_layout);

/* Row-major scales [rows][K/16] -> QLIN_SF_MMA layout (rows past `rows`
   written as 0).  K a multiple of 64; src 4-byte aligned, dst 16-byte
   aligned. */
qlin_status qlin_nvfp4_sf_to_mma(const uint8_t* sf_rows, int64_t rows, int64_t K, uint8_t* sf_mma,
                                 cudaStream_t stream);

/* ------------------------------------------------------------------------
 * c2 - NVFP4 block-scaled GEMM
 *
 * Y[t,n] = g_a . g_b . sum_b sfa[t,b] . sfb[n,b] . sum_{k in b} a[t,k] . b[n,k]
 * over the (augmented) K, fp32 accumulation on the block-scaled fp4 tensor
 * cores, one final rounding ("LLM and AIGC quantization", block-scaled
 * formats: the tensor core applies the block scales during accumulation;
 * "NVFP4 quantization and ARCQuant", section 2.2: Y ~ sX_aug QX_aug
 * (sW_aug QW_aug)^T).
 *   a, b      uint8 [T][K/2], [N][K/2]   packed E2M1 codes
 *   sfa, sfb  E4M3 block scales of a and b in the QLIN_SF_MMA layout
 *             (16-byte aligned; qlin_nvfp4_sf_bytes(T or N, K, QLIN_SF_MMA))
 *   g_a, g_b  float32 [1] device scalars
 *   out       [T][N] of out_dtype (BF16 or F16)
 * K must be a multiple of 64 (the tensor-core K step).
 * ---------------------------------------------------------------------- */
qlin_status qlin_nvfp4_gemm(const uint8_t* a, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb,
                            int64_t T, int64_t N, int64_t K, const float* g_a, const float* g_b, void* out,
                            qlin_dtype out_dtype, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * next 1 - FP8 W8A8: per-row E4M3 quantization
 *
 * Per row r (a token of the activations, or an output channel of the
 * weights): s_r = max_k |x[r,k]| / 448 in float32 (s_r = 1 for an all-zero
 * row), q[r,k] = E4M3(x[r,k] / s_r) with x / s_r an IEEE float32 division
 * and the E4M3-FN encode rounding to nearest, ties to even, saturating at
 * 448 ("LLM and AIGC quantization", "W4A4, FP8 and block-scaled formats": x/s
 * is converted to E4M3 instead of rounded to INT8, activations per token and
 * weights per channel; "FP8: robustness from dynamic range": the per-tensor
 * example [0.6, -45.0, 1.1, -0.8] -> 6, -448, 11, -8).
 *   x      [rows][K] of x_dtype (16-byte aligned; K a multiple of 8)
 *   q      out, uint8 [rows][K]: E4M3-FN codes (sign in bit 7)
 *   scale  out, float32 [rows]
 * ---------------------------------------------------------------------- */
qlin_status qlin_quant_fp8(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, uint8_t* q, float* scale,
                           cudaStream_t stream);

/* ------------------------------------------------------------------------
 * next 1 - FP8 W8A8 GEMM on the tcgen05 tensor cores (kind::f8f6f4)
 *
 * out[t,n] = s_a[t] . s_b[n] . sum_k dec(a[t,k]) . dec(b[n,k]) + bias[n]
 * with E4M3 operands, fp32 accumulation in the tensor core and the two scales
 * and the bias applied once in the epilogue, in float32, one final rounding
 * ("LLM and AIGC quantization", "W4A4, FP8 and block-scaled formats": the
 * FP8 tensor core multiplies, FP32 accumulates, the epilogue multiplies by
 * both scales).
 *   a        uint8 [T][K]  E4M3 codes of the activations (per-token scales)
 *   b        uint8 [N][K]  E4M3 codes of the weights (per-channel scales)
 *   scale_a  float32 [T];  scale_b float32 [N]
 *   bias     [N] of bias_dtype (F16, BF16 or F32), or NULL for 0
 *   out      [T][N] of out_dtype (F16 or BF16)
 * a and b 16-byte aligned; K a multiple of 16 (rows of whole 16-byte
 * pieces); codes 0x7F / 0xFF (NaN) are not valid inputs.
 * ---------------------------------------------------------------------- */
qlin_status qlin_fp8_gemm(const uint8_t* a, const uint8_t* b, int64_t T, int64_t N, int64_t K, const float* scale_a,
                          const float* scale_b, const void* bias, qlin_dtype bias_dtype, void* out,
                          qlin_dtype out_dtype, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * next 2 - RMSNorm fused with the per-token quantizer
 *
 * Per row: y = (x . inv) . gamma with inv = 1 / sqrt(mean(x^2) + eps) (one
 * square root and one division per row; a row whose mean(x^2) + eps is 0
 * normalizes to 0), then the per-token
 * quantization of y in `fmt` (int8: s = max|y| / 127, q = clamp(rint(y / s),
 * -127, 127); E4M3: s = max|y| / 448, q = E4M3(y / s); s = 1 for an all-zero
 * y), with y kept in float32 and the row read once ("Chapter 9 -
 * Quantization kernels", practical notes: the per-row max and quantization
 * fused into the upstream operator; "LLM and AIGC quantization", "Static and
 * dynamic quantization": the per-token reduction is usually fused into the
 * preceding RMSNorm).  The mean of squares is the exact sum of the row's
 * squares rounded once to float32 (nearest, ties to even), divided by K in
 * float32: no order of additions is implied, and the result is the same for
 * any number of threads.  Every other step is one IEEE float32 operation.
 *   x      [rows][K] of x_dtype (16-byte aligned; K a multiple of 16)
 *   gamma  [K] of x_dtype (16-byte aligned)
 *   eps    the RMSNorm epsilon (>= 0)
 *   q      out, [rows][K] bytes: int8 codes or E4M3-FN codes (16-byte aligned)
 *   scale  out, float32 [rows]
 * ---------------------------------------------------------------------- */
qlin_status qlin_rmsnorm_quant(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, const void* gamma,
                               float eps, qlin_qfmt fmt, void* q, float* scale, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * next 2 - RMSNorm fused with the NVFP4 / ARCQuant quantizer
 *
 * Per row, y = (x . inv) . gamma exactly as qlin_rmsnorm_quant defines it
 * (the same exactly rounded mean of squares, the same float32 steps),
 * then qlin_quant_nvfp4 of y: the reordered channels ys = y[:, perm], the
 * 16-element blocks with E4M3 scales over the per-tensor g, and the S
 * residual (or duplicated) channels; y stays in float32 and x is read once.
 * g and perm are calibrated on y (the normalized activations the GEMM
 * consumes), e.g. with qlin_nvfp4_global_scale / qlin_arc_perm on a
 * calibration batch of y.
 *   x, perm, S, mode, g, q, sf, sf_layout  as in qlin_quant_nvfp4
 *   gamma  [K] of x_dtype (16-byte aligned)
 *   eps    the RMSNorm epsilon (>= 0)
 * Rows of up to 96 KB (K <= 49152 for 16-bit x, 24576 for F32): a row and
 * gamma are both staged in shared memory (QLIN_ERR_UNSUPPORTED above).
 * ---------------------------------------------------------------------- */
/* ------------------------------------------------------------------------
 * next 1 - MX block-scaled formats: MXFP8 and MXFP4
 *
 * qlin_quant_mx, per row, per block of 32 consecutive elements ("LLM and
 * AIGC quantization", block-scaled formats: the E8M0 scale is the power of
 * two 2^(floor(log2 absmax) - e_max), e_max = 8 for E4M3 and 2 for E2M1):
 *   e  = floor(log2 max|x|) - e_max, clamped to [-127, 127]; -127 for a zero
 *        block
 *   sf = e + 127 (the E8M0 code);  q = E4M3 / E2M1(x . 2^-e)  (float32
 *        multiply; round-to-nearest-even, saturating at 448 / 6, sign kept)
 *   x     [rows][K] of x_dtype (F16, BF16 or F32), 16-byte aligned
 *   q     out: MXFP8 uint8 [rows][K]; MXFP4 uint8 [rows][K/2] (16-byte aligned)
 *   sf    out: E8M0 codes in sf_layout: QLIN_SF_ROWS [rows][K/32], or
 *         QLIN_SF_MMA, the layout qlin_mx_gemm reads: 512-byte blocks of 128
 *         rows x 4 scales, block (r/128, j/4) at ((r/128) . ceil(K/128) +
 *         j/4) . 512, byte 16 (r%32) + 4 ((r%128)/32) + j%4 for row r, scale
 *         j (bytes of padding rows and of a last partial group are left
 *         unwritten)
 * K a multiple of 32.
 *
 * qlin_mx_gemm: out[t][n] = sum_k dec(a)[t,k] 2^(sfa[t,k/32]-127) .
 * dec(b)[n,k] 2^(sfb[n,k/32]-127), fp32 accumulation on the block-scaled
 * tensor cores (the MMA applies both blocks' scales), one rounding to out.
 *   a [T][K] / b [N][K] codes as qlin_quant_mx writes them; sfa, sfb in
 *   QLIN_SF_MMA (16-byte aligned); out [T][N] F16 or BF16, N a multiple of 8.
 *   K a multiple of 32 (MXFP8) or 64 (MXFP4).
 * ---------------------------------------------------------------------- */
int64_t qlin_mx_sf_bytes(int64_t rows, int64_t K, qlin_sf_layout sf_layout);
qlin_status qlin_quant_mx(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, qlin_mx_fmt fmt, uint8_t* q,
                          uint8_t* sf, qlin_sf_layout sf_layout, cudaStream_t stream);
qlin_status qlin_mx_gemm(const uint8_t* a, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb, int64_t T,
                         int64_t N, int64_t K, qlin_mx_fmt fmt, void* out, qlin_dtype out_dtype, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * next 4 - online Hadamard rotation of the activations before 4-bit
 * quantization
 *
 * Every group of n consecutive elements of each row is multiplied by the
 * normalized Hadamard matrix H_n / sqrt(n), then by signs[k] (QuaRot's
 * diag(+-1)) when signs is not NULL, and rounded once to the input dtype:
 *   QLIN_HADAMARD_SYLVESTER ("LLM and AIGC quantization", QuaRot: the
 *     Sylvester matrix, applied as the fast Walsh-Hadamard transform,
 *     log2(n) butterfly stages mapping the pair (a, b) at distance h to
 *     (a + b, a - b)); n a power of two, 2 <= n <= 8192;
 *   QLIN_HADAMARD_REGULAR (ConvRot: each group of N0 times the regular
 *     Hadamard, the Kronecker power of H4 = [[1,1,1,-1],[1,1,-1,1],
 *     [1,-1,1,1],[-1,1,1,1]], applied as radix-4 stages); n in {4, 16, 64,
 *     256}.
 * F32 rows and the other group sizes run butterfly stages in float32: the
 * result is within float32 rounding of the exact rotation (before the final
 * rounding to the input dtype).  F16 / BF16 rows with n = 256 (both kinds)
 * or a Sylvester n of 512 .. 4096 run as 16 x 16 products on the tensor
 * cores (the order-256 matrices are Kronecker squares of a 16 x 16 factor,
 * ConvRot's dense product cut into factors; for n < 4096 the groups after
 * the buffer's last whole block of 4096 elements take the butterflies
 * instead): fp32 accumulation, intermediates kept to
 * 16 significant bits, so the result is within about 2^-16 of the exact
 * rotation's magnitude before the final rounding.  Every path gives the same
 * bits on every run.  The weights take the same rotation offline (W . Q),
 * which leaves X . W^T unchanged.
 *   x      [rows][K] of dtype (F16, BF16 or F32), 16-byte aligned
 *   signs  int8 [K] of +1 / -1 (8-byte aligned), or NULL
 *   y      out, [rows][K] of dtype, 16-byte aligned (y == x allowed)
 * K a multiple of n and of 8.
 * ---------------------------------------------------------------------- */
qlin_status qlin_hadamard(const void* x, qlin_dtype dtype, int64_t rows, int64_t K, qlin_hadamard_kind kind,
                          int64_t n, const int8_t* signs, void* y, cudaStream_t stream);

qlin_status qlin_rmsnorm_quant_nvfp4(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, const void* gamma,
                                     float eps, const int32_t* perm, int64_t S, qlin_nvfp4_mode mode, const float* g,
                                     uint8_t* q, uint8_t* sf, qlin_sf_layout sf_layout, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QLIN_H_ */
