// Internal host-side interface between the C ABI layer (qlin_api.cu) and the
// kernel translation units.  Every launcher enqueues on `stream`, returns the
// launch status and never synchronizes.  Arguments have already been checked
// by the ABI layer.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qlin.h"

namespace qlin {

// Device address of the per-device error word (set up once per device).
int32_t* device_error_word();

// Number of SMs of the current device (cached per device).
int sm_count();

// Raises fn's dynamic shared-memory limit to the device's per-block maximum
// (less fn's static shared memory), once per device and kernel; every launch
// then asks for its own amount.  Returns the status of that one setting.
cudaError_t ensure_max_dynamic_smem(const void* fn);

cudaError_t launch_quant_w4_g128(const void* w, qlin_dtype w_dtype, int64_t N, int64_t K, uint8_t* wq,
                                 void* scales, uint8_t* zeros, cudaStream_t stream);

cudaError_t launch_w4a16_gemm(const void* x, int64_t T, int64_t N, int64_t K, const uint8_t* wq,
                              const void* scales, const uint8_t* zeros, void* y, cudaStream_t stream);

// One-token W4A16 GEMV on the CUDA cores (T == 1, K <= 12288, the CTA's
// band of scales small enough for its shared-memory plan).
bool w4a16_gemv_supported(int64_t T, int64_t N, int64_t K);
// Whether the GEMV's alternating launch shapes are in use on the current
// device, and the kernel's registers per thread.
cudaError_t w4a16_gemv_launch_info(int* alternating, int* registers);
cudaError_t launch_w4a16_gemv(const void* x, int64_t N, int64_t K, const uint8_t* wq, const void* scales,
                              const uint8_t* zeros, void* y, cudaStream_t stream);
// One GEMV launch over the concatenated rows of `count` matrices sharing x
// (cudaErrorInvalidValue when the concatenation has no launch plan).
cudaError_t launch_w4a16_gemv_grouped(const void* x, int64_t K, int count, const int64_t* N,
                                      const uint8_t* const* wq, const void* const* scales,
                                      const uint8_t* const* zeros, void* const* y, cudaStream_t stream);
using W4A16SeqStep = qlin_w4a16_step;
int64_t w4a16_sequence_workspace_bytes(int64_t nsteps);
bool w4a16_sequence_supported(int64_t K);
// The steps in order in persistent cooperative launches (up to 128 steps
// each); workspace holds one arrival counter per step.
cudaError_t launch_w4a16_sequence(const W4A16SeqStep* steps, int nsteps, unsigned int* workspace,
                                  cudaStream_t stream);
// Device address of the library's own counters on the current device (enough
// for every launch of a sequence: each launch takes at most 128 steps and
// zeroes them first).  The address is looked up once per device, on the
// first call with that device current.
cudaError_t w4a16_sequence_static_workspace(unsigned int** out);
// W4A16 decode plan (T <= 16): the steps of a chain in one persistent launch
// on the warp-level tensor cores.  The workspace holds the plan: the step
// table, one tensor map per matrix and one grid-barrier counter per step.
int64_t w4a16_decode_workspace_bytes(int64_t nsteps);
// nullptr when the steps fit the kernel's limits, else the reason (and the
// failing step in *bad_step, -1 for T).
const char* w4a16_decode_check(const qlin_w4a16_step* steps, int nsteps, int64_t T, int* bad_step);
// Writes the plan into the workspace (stream-ordered kernel writes).
cudaError_t w4a16_decode_prepare(const qlin_w4a16_step* steps, int nsteps, int64_t T, void* workspace,
                                 cudaStream_t stream);
cudaError_t w4a16_decode_run(const void* workspace, int nsteps, int64_t T, cudaStream_t stream);
// Streamed tensor-core W4A16 for up to 16 tokens over the concatenated rows
// of `count` matrices sharing x (false / cudaErrorInvalidValue when the
// shape has no launch plan).
bool w4a16_skinny_supported(int64_t T, int64_t N, int64_t K);
cudaError_t launch_w4a16_skinny_grouped(const void* x, int64_t T, int64_t K, int count, const int64_t* N,
                                        const uint8_t* const* wq, const void* const* scales,
                                        const uint8_t* const* zeros, void* const* y, cudaStream_t stream);
cudaError_t launch_hadamard(const void* x, qlin_dtype dtype, int64_t rows, int64_t K, qlin_hadamard_kind kind,
                            int64_t n, const int8_t* signs, void* y, cudaStream_t stream);
// W4A16 act-order: group-sorted column order and codes (offline), activation gather.
cudaError_t launch_w4a16_act_order_prepare(const int32_t* g_idx, int64_t K, int64_t group, const uint8_t* wq,
                                           int64_t N, int32_t* perm, uint8_t* wq_sorted, cudaStream_t stream);
cudaError_t launch_x_permute(const void* x, int64_t T, int64_t K, const int32_t* perm, void* out,
                             cudaStream_t stream);
// W4A16 for many tokens (prefill) on the tcgen05 tensor cores.
bool w4a16_prefill_supported(int64_t T, int64_t N, int64_t K);
cudaError_t launch_w4a16_prefill(const void* x, int64_t T, int64_t N, int64_t K, const uint8_t* wq,
                                 const void* scales, const uint8_t* zeros, void* y, cudaStream_t stream);
cudaError_t launch_w4a16_gemm_grouped(const void* x, int64_t T, int64_t K, int count, const int64_t* N,
                                      const uint8_t* const* wq, const void* const* scales,
                                      const uint8_t* const* zeros, void* const* y, cudaStream_t stream);

// q: int8 [T][K], or (f16_codes) the same codes as exact fp16 values [T][K].
cudaError_t launch_quant_act_int8(const void* x, qlin_dtype x_dtype, int64_t T, int64_t K, void* q, bool f16_codes,
                                  float* scale, int32_t* azp, cudaStream_t stream);

cudaError_t launch_int8_row_sum(const int8_t* b, int64_t N, int64_t K, int32_t* out, cudaStream_t stream);

struct W8A8Epilogue {
  const float* scale_a;
  bool scale_a_per_row;
  const float* scale_b;
  bool scale_b_per_col;
  const int32_t* azp;      // [T] or null
  const int32_t* azp_adj;  // [N] or null
  const void* bias;        // [N] or null
  qlin_dtype bias_dtype;
  qlin_dtype out_dtype;    // F16, BF16 or I32 (raw accumulator)
};

// b: int8 [N][K], or (b_f16) the same codes as exact fp16 values [N][K].
cudaError_t launch_w8a8_gemm(const int8_t* a, const void* b, bool b_f16, int64_t T, int64_t N, int64_t K,
                             const W8A8Epilogue& epi, void* out, cudaStream_t stream);

// Both operands as exact fp16 codes: a16 fp16 [T][K], b16 fp16 [N][K].
cudaError_t launch_w8a8_gemm_f16(const void* a16, const void* b16, int64_t T, int64_t N, int64_t K,
                                 const W8A8Epilogue& epi, void* out, cudaStream_t stream);

// dst[i] = fp16(src[i]) for int8 src (exact).
cudaError_t launch_int8_to_f16(const int8_t* src, int64_t count, void* dst, cudaStream_t stream);

cudaError_t launch_nvfp4_global_scale(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, float* g,
                                      cudaStream_t stream);

cudaError_t launch_arc_perm(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, int32_t* perm,
                            cudaStream_t stream);

cudaError_t launch_quant_nvfp4(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, const int32_t* perm,
                               int64_t S, qlin_nvfp4_mode mode, const float* g, uint8_t* q, uint8_t* sf,
                               qlin_sf_layout sf_layout, const void* gamma, float eps, cudaStream_t stream);

cudaError_t launch_nvfp4_sf_to_mma(const uint8_t* src, int64_t rows, int64_t K, uint8_t* dst, cudaStream_t stream);

cudaError_t launch_nvfp4_gemm(const uint8_t* a, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb,
                              int64_t T, int64_t N, int64_t K, const float* g_a, const float* g_b, void* out,
                              qlin_dtype out_dtype, cudaStream_t stream);

cudaError_t launch_quant_mx(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, qlin_mx_fmt fmt, uint8_t* q,
                            uint8_t* sf, qlin_sf_layout sf_layout, cudaStream_t stream);
cudaError_t launch_mx_gemm(const uint8_t* a, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb, int64_t T,
                           int64_t N, int64_t K, qlin_mx_fmt fmt, void* out, qlin_dtype out_dtype,
                           cudaStream_t stream);
cudaError_t launch_quant_fp8(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, uint8_t* q, float* scale,
                             cudaStream_t stream);

cudaError_t launch_rmsnorm_quant(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, const void* gamma,
                                 float eps, qlin_qfmt fmt, void* q, float* scale, cudaStream_t stream);

cudaError_t launch_fp8_gemm(const uint8_t* a, const uint8_t* b, int64_t T, int64_t N, int64_t K, const float* scale_a,
                            const float* scale_b, const void* bias, qlin_dtype bias_dtype, void* out,
                            qlin_dtype out_dtype, cudaStream_t stream);

}  // namespace qlin
