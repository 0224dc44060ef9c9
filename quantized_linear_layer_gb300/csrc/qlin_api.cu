// The C ABI of the library: argument checks, status codes, the per-device
// error word, and dispatch to the kernel launchers.  Host code only.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "qlin_internal.h"

namespace qlin {
namespace {

constexpr int kMaxDevices = 64;

thread_local char g_last_error[512] = {0};

qlin_status fail(qlin_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

qlin_status ok() {
  g_last_error[0] = '\0';
  return QLIN_OK;
}

qlin_status cuda_fail(cudaError_t e, const char* what) {
  return fail(QLIN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DeviceInfo {
  bool probed = false;
  bool supported = false;
  int sm_count = 0;
  int32_t* err_word = nullptr;
};

DeviceInfo g_devices[kMaxDevices];
std::mutex g_device_mutex;

// The per-device error word lives in this translation unit.
__device__ int32_t g_device_error_word;

qlin_status probe_current_device(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(QLIN_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_device_mutex);
  DeviceInfo& d = g_devices[dev];
  if (!d.probed) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    d.supported = (major == 10 && minor == 3);
    d.sm_count = sms;
    if (d.supported) {
      void* p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_device_error_word)) != cudaSuccess)
        return cuda_fail(e, "cudaGetSymbolAddress(error word)");
      d.err_word = static_cast<int32_t*>(p);
    }
    d.probed = true;
  }
  if (!d.supported) return fail(QLIN_ERR_UNSUPPORTED, "device %d is not compute capability 10.3 (GB300)", dev);
  *out = &d;
  return QLIN_OK;
}

DeviceInfo* current_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return &g_devices[dev];
}

bool is_float_dtype(qlin_dtype d) { return d == QLIN_F16 || d == QLIN_BF16 || d == QLIN_F32; }
int64_t dtype_bytes(qlin_dtype d) { return d == QLIN_F32 || d == QLIN_I32 ? 4 : 2; }

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

}  // namespace

int32_t* device_error_word() {
  DeviceInfo* d = current_info();
  return d != nullptr ? d->err_word : nullptr;
}

int sm_count() {
  DeviceInfo* d = current_info();
  return (d != nullptr && d->sm_count > 0) ? d->sm_count : 152;
}

cudaError_t ensure_max_dynamic_smem(const void* fn) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  struct Done {
    int dev;
    const void* fn;
    cudaError_t status;
  };
  static std::vector<Done> done;
  std::lock_guard<std::mutex> lock(mu);
  for (const Done& d : done)
    if (d.dev == dev && d.fn == fn) return d.status;
  int optin = 0;
  cudaFuncAttributes fa = {};
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, fn);
  // the limit covers the dynamic part; static shared memory comes on top
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - static_cast<int>(fa.sharedSizeBytes));
  done.push_back({dev, fn, e});
  return e;
}

}  // namespace qlin

using namespace qlin;

#define QLIN_REQUIRE(cond, status, ...) \
  do {                                  \
    if (!(cond)) return fail(status, __VA_ARGS__); \
  } while (0)

#define QLIN_DEVICE()                          \
  do {                                         \
    DeviceInfo* info_ = nullptr;               \
    qlin_status st_ = probe_current_device(&info_); \
    if (st_ != QLIN_OK) return st_;            \
  } while (0)

#define QLIN_LAUNCH(expr, what)                       \
  do {                                                \
    cudaError_t e_ = (expr);                          \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    return ok();                                      \
  } while (0)

extern "C" {

const char* qlin_status_string(qlin_status status) {
  switch (status) {
    case QLIN_OK: return "QLIN_OK";
    case QLIN_ERR_INVALID_ARG: return "QLIN_ERR_INVALID_ARG";
    case QLIN_ERR_ALIGNMENT: return "QLIN_ERR_ALIGNMENT";
    case QLIN_ERR_UNSUPPORTED: return "QLIN_ERR_UNSUPPORTED";
    case QLIN_ERR_CUDA: return "QLIN_ERR_CUDA";
    case QLIN_ERR_TIMEOUT: return "QLIN_ERR_TIMEOUT";
  }
  return "QLIN_ERR_UNKNOWN";
}

const char* qlin_last_error_message(void) { return g_last_error; }

int qlin_version(void) { return 100; }

qlin_status qlin_w4a16_gemv_launch_info(int* alternating, int* registers) {
  QLIN_DEVICE();
  const cudaError_t e = w4a16_gemv_launch_info(alternating, registers);
  if (e != cudaSuccess) return cuda_fail(e, "w4a16_gemv_launch_info");
  return ok();
}

qlin_status qlin_get_device_error(cudaStream_t stream, int32_t* code_out) {
  DeviceInfo* info = nullptr;
  qlin_status st = probe_current_device(&info);
  if (st != QLIN_OK) return st;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int32_t code = 0;
  if ((e = cudaMemcpy(&code, info->err_word, sizeof(code), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "read device error word");
  if (code != 0) {
    const int32_t zero = 0;
    if ((e = cudaMemcpy(info->err_word, &zero, sizeof(zero), cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "clear device error word");
  }
  if (code_out != nullptr) *code_out = code;
  if (code != 0) return fail(QLIN_ERR_TIMEOUT, "device error word was 0x%x", code);
  return ok();
}

qlin_status qlin_quant_w4_g128(const void* w, qlin_dtype w_dtype, int64_t N, int64_t K, int64_t group,
                               uint8_t* wq, void* scales, uint8_t* zeros, cudaStream_t stream) {
  QLIN_REQUIRE(group == 128, QLIN_ERR_UNSUPPORTED, "group size %lld (only 128 is built)", (long long)group);
  QLIN_REQUIRE(is_float_dtype(w_dtype), QLIN_ERR_INVALID_ARG, "w_dtype must be F16, BF16 or F32");
  QLIN_REQUIRE(N >= 0 && N <= kMaxDim && K > 0 && K <= kMaxDim, QLIN_ERR_INVALID_ARG, "bad sizes N=%lld K=%lld",
               (long long)N, (long long)K);
  QLIN_REQUIRE(K % group == 0, QLIN_ERR_INVALID_ARG, "K=%lld is not a multiple of the group size", (long long)K);
  if (N == 0) return ok();
  QLIN_REQUIRE(w && wq && scales && zeros, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(aligned16(w) && aligned16(wq), QLIN_ERR_ALIGNMENT, "w and wq must be 16-byte aligned");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(scales) & 1u) == 0, QLIN_ERR_ALIGNMENT, "scales must be 2-byte aligned");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_quant_w4_g128(w, w_dtype, N, K, wq, scales, zeros, stream), "quant_w4_g128 launch");
}

qlin_status qlin_w4a16_gemm(const void* x, int64_t T, int64_t N, int64_t K, const uint8_t* wq,
                            const void* scales, const uint8_t* zeros, int64_t group, void* y,
                            cudaStream_t stream) {
  QLIN_REQUIRE(group == 128, QLIN_ERR_UNSUPPORTED, "group size %lld (only 128 is built)", (long long)group);
  QLIN_REQUIRE(T >= 0 && T <= kMaxDim, QLIN_ERR_INVALID_ARG, "T=%lld out of range", (long long)T);
  QLIN_REQUIRE(N >= 0 && N <= kMaxDim && K > 0 && K <= kMaxDim, QLIN_ERR_INVALID_ARG, "bad sizes N=%lld K=%lld",
               (long long)N, (long long)K);
  QLIN_REQUIRE(K % group == 0, QLIN_ERR_INVALID_ARG, "K=%lld is not a multiple of the group size", (long long)K);
  if (T == 0 || N == 0) return ok();
  QLIN_REQUIRE(x && wq && scales && y, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(aligned16(x) && aligned16(wq), QLIN_ERR_ALIGNMENT, "x and wq must be 16-byte aligned");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(scales) & 1u) == 0 && (reinterpret_cast<uintptr_t>(y) & 1u) == 0,
               QLIN_ERR_ALIGNMENT, "scales and y must be 2-byte aligned");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_w4a16_gemm(x, T, N, K, wq, scales, zeros, y, stream), "w4a16_gemm launch");
}

}  // extern "C"

namespace {

// The checks of one grouped W4A16 call (T tokens, `count` matrices of K
// columns); `what` names the call or step in the message.
qlin_status check_w4a16_group(const char* what, const void* x, int64_t T, int64_t K, int count, const int64_t* N,
                              const uint8_t* const* wq, const void* const* scales, const void* const* y,
                              int64_t group, int64_t* total_out) {
  QLIN_REQUIRE(group == 128, QLIN_ERR_UNSUPPORTED, "group size %lld (only 128 is built)", (long long)group);
  QLIN_REQUIRE(count >= 1 && count <= QLIN_W4A16_MAX_GROUP, QLIN_ERR_INVALID_ARG, "%s: count=%d outside [1, %d]", what,
               count, QLIN_W4A16_MAX_GROUP);
  QLIN_REQUIRE(T >= 0 && T <= kMaxDim, QLIN_ERR_INVALID_ARG, "T=%lld out of range", (long long)T);
  QLIN_REQUIRE(K > 0 && K <= kMaxDim, QLIN_ERR_INVALID_ARG, "%s: bad K=%lld", what, (long long)K);
  QLIN_REQUIRE(K % group == 0, QLIN_ERR_INVALID_ARG, "%s: K=%lld is not a multiple of the group size", what,
               (long long)K);
  int64_t total = 0;
  for (int p = 0; p < count; ++p) {
    QLIN_REQUIRE(N[p] >= 0 && N[p] <= kMaxDim, QLIN_ERR_INVALID_ARG, "%s: bad N[%d]=%lld", what, p, (long long)N[p]);
    total += N[p];
  }
  QLIN_REQUIRE(total <= kMaxDim, QLIN_ERR_INVALID_ARG, "%s: total rows %lld too large", what, (long long)total);
  *total_out = total;
  if (T == 0 || total == 0) return QLIN_OK;
  QLIN_REQUIRE(x && aligned16(x), x ? QLIN_ERR_ALIGNMENT : QLIN_ERR_INVALID_ARG,
               "%s: x must be non-null and 16-byte aligned", what);
  for (int p = 0; p < count; ++p) {
    if (N[p] == 0) continue;
    QLIN_REQUIRE(wq[p] && scales[p] && y[p], QLIN_ERR_INVALID_ARG, "%s: null pointer for matrix %d", what, p);
    QLIN_REQUIRE(aligned16(wq[p]), QLIN_ERR_ALIGNMENT, "%s: wq[%d] must be 16-byte aligned", what, p);
    QLIN_REQUIRE((reinterpret_cast<uintptr_t>(scales[p]) & 1u) == 0 && (reinterpret_cast<uintptr_t>(y[p]) & 1u) == 0,
                 QLIN_ERR_ALIGNMENT, "%s: scales[%d] and y[%d] must be 2-byte aligned", what, p, p);
  }
  return QLIN_OK;
}

}  // namespace

extern "C" {

qlin_status qlin_w4a16_gemm_grouped(const void* x, int64_t T, int64_t K, int count, const int64_t* N,
                                    const uint8_t* const* wq, const void* const* scales,
                                    const uint8_t* const* zeros, int64_t group, void* const* y,
                                    cudaStream_t stream) {
  QLIN_REQUIRE(N && wq && scales && zeros && y, QLIN_ERR_INVALID_ARG, "null host array");
  int64_t total = 0;
  const qlin_status st = check_w4a16_group("w4a16_gemm_grouped", x, T, K, count, N, wq, scales, y, group, &total);
  if (st != QLIN_OK) return st;
  if (T == 0 || total == 0) return ok();
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_w4a16_gemm_grouped(x, T, K, count, N, wq, scales, zeros, y, stream), "w4a16_gemm_grouped launch");
}

qlin_status qlin_w4a16_chain(const qlin_w4a16_step* steps, int nsteps, int64_t T, int64_t group,
                             cudaStream_t stream) {
  QLIN_REQUIRE(nsteps >= 0, QLIN_ERR_INVALID_ARG, "nsteps=%d", nsteps);
  if (nsteps == 0 || T == 0) return ok();
  QLIN_REQUIRE(steps != nullptr, QLIN_ERR_INVALID_ARG, "null steps");
  char what[32];
  for (int s = 0; s < nsteps; ++s) {
    const qlin_w4a16_step& st = steps[s];
    snprintf(what, sizeof(what), "step %d", s);
    int64_t total = 0;
    const qlin_status r = check_w4a16_group(what, st.x, T, st.K, st.count, st.N, st.wq, st.scales, st.y, group,
                                            &total);
    if (r != QLIN_OK) return r;
  }
  QLIN_DEVICE();
  for (int s = 0; s < nsteps; ++s) {
    const qlin_w4a16_step& st = steps[s];
    const cudaError_t e = launch_w4a16_gemm_grouped(st.x, T, st.K, st.count, st.N, st.wq, st.scales, st.zeros,
                                                    st.y, stream);
    if (e != cudaSuccess) return cuda_fail(e, "w4a16_chain launch");
  }
  return ok();
}

int64_t qlin_w4a16_decode_workspace_bytes(int64_t nsteps) { return w4a16_decode_workspace_bytes(nsteps); }

qlin_status qlin_w4a16_decode_prepare(const qlin_w4a16_step* steps, int nsteps, int64_t T, int64_t group,
                                      void* workspace, cudaStream_t stream) {
  QLIN_REQUIRE(nsteps >= 1 && nsteps <= (1 << 20), QLIN_ERR_INVALID_ARG, "nsteps=%d outside [1, 2^20]", nsteps);
  QLIN_REQUIRE(steps != nullptr, QLIN_ERR_INVALID_ARG, "null steps");
  QLIN_REQUIRE(T >= 1 && T <= 16, QLIN_ERR_UNSUPPORTED, "T=%lld: the decode plan takes 1 .. 16 tokens", (long long)T);
  QLIN_REQUIRE(workspace != nullptr, QLIN_ERR_INVALID_ARG, "null workspace");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, QLIN_ERR_ALIGNMENT,
               "workspace must be 256-byte aligned");
  char what[32];
  for (int s = 0; s < nsteps; ++s) {
    const qlin_w4a16_step& st = steps[s];
    snprintf(what, sizeof(what), "step %d", s);
    int64_t total = 0;
    const qlin_status r = check_w4a16_group(what, st.x, T, st.K, st.count, st.N, st.wq, st.scales, st.y, group,
                                            &total);
    if (r != QLIN_OK) return r;
    QLIN_REQUIRE(st.x != nullptr, QLIN_ERR_INVALID_ARG, "step %d: null x", s);
  }
  QLIN_DEVICE();
  int bad = -1;
  const char* why = w4a16_decode_check(steps, nsteps, T, &bad);
  if (why != nullptr) return fail(QLIN_ERR_UNSUPPORTED, "step %d: %s", bad, why);
  QLIN_LAUNCH(w4a16_decode_prepare(steps, nsteps, T, workspace, stream), "w4a16_decode_prepare");
}

qlin_status qlin_w4a16_decode_run(const void* workspace, int nsteps, int64_t T, cudaStream_t stream) {
  QLIN_REQUIRE(nsteps >= 1 && nsteps <= (1 << 20), QLIN_ERR_INVALID_ARG, "nsteps=%d outside [1, 2^20]", nsteps);
  QLIN_REQUIRE(T >= 1 && T <= 16, QLIN_ERR_UNSUPPORTED, "T=%lld: the decode plan takes 1 .. 16 tokens", (long long)T);
  QLIN_REQUIRE(workspace != nullptr, QLIN_ERR_INVALID_ARG, "null workspace");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, QLIN_ERR_ALIGNMENT,
               "workspace must be 256-byte aligned");
  QLIN_DEVICE();
  const cudaError_t e = w4a16_decode_run(workspace, nsteps, T, stream);
  if (e == cudaErrorCooperativeLaunchTooLarge)
    return fail(QLIN_ERR_UNSUPPORTED, "the device cannot hold one CTA per SM for the decode plan");
  QLIN_LAUNCH(e, "w4a16_decode_run launch");
}

qlin_status qlin_w4a16_act_order_prepare(const int32_t* g_idx, int64_t K, int64_t group, const uint8_t* wq,
                                         int64_t N, int32_t* perm, uint8_t* wq_sorted, cudaStream_t stream) {
  QLIN_REQUIRE(group == 128, QLIN_ERR_UNSUPPORTED, "group size %lld (only 128 is built)", (long long)group);
  QLIN_REQUIRE(K > 0 && K <= kMaxDim && K % group == 0, QLIN_ERR_INVALID_ARG, "K=%lld is not a positive multiple of %lld",
               (long long)K, (long long)group);
  QLIN_REQUIRE(N >= 0 && N <= kMaxDim, QLIN_ERR_INVALID_ARG, "bad N=%lld", (long long)N);
  QLIN_REQUIRE(g_idx && perm && (N == 0 || (wq && wq_sorted)), QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(wq != wq_sorted || N == 0, QLIN_ERR_INVALID_ARG, "wq_sorted must not alias wq");
  QLIN_REQUIRE(aligned16(perm), QLIN_ERR_ALIGNMENT, "perm must be 16-byte aligned");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(g_idx) & 3u) == 0, QLIN_ERR_ALIGNMENT, "g_idx must be 4-byte aligned");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_w4a16_act_order_prepare(g_idx, K, group, wq, N, perm, wq_sorted, stream),
              "w4a16_act_order_prepare launch");
}

qlin_status qlin_w4a16_gemm_act_order(const void* x, int64_t T, int64_t N, int64_t K, const int32_t* perm,
                                      const uint8_t* wq_sorted, const void* scales, const uint8_t* zeros,
                                      int64_t group, void* x_work, void* y, cudaStream_t stream) {
  QLIN_REQUIRE(group == 128, QLIN_ERR_UNSUPPORTED, "group size %lld (only 128 is built)", (long long)group);
  QLIN_REQUIRE(T >= 0 && T <= kMaxDim, QLIN_ERR_INVALID_ARG, "T=%lld out of range", (long long)T);
  QLIN_REQUIRE(N >= 0 && N <= kMaxDim && K > 0 && K <= kMaxDim, QLIN_ERR_INVALID_ARG, "bad sizes N=%lld K=%lld",
               (long long)N, (long long)K);
  QLIN_REQUIRE(K % group == 0, QLIN_ERR_INVALID_ARG, "K=%lld is not a multiple of the group size", (long long)K);
  QLIN_REQUIRE(K <= 98304, QLIN_ERR_UNSUPPORTED, "K=%lld: the gathered row must fit shared memory (K <= 98304)",
               (long long)K);
  if (T == 0 || N == 0) return ok();
  QLIN_REQUIRE(x && perm && wq_sorted && scales && x_work && y, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(x_work != x, QLIN_ERR_INVALID_ARG, "x_work must not alias x");
  QLIN_REQUIRE(aligned16(x) && aligned16(wq_sorted) && aligned16(perm) && aligned16(x_work), QLIN_ERR_ALIGNMENT,
               "x, perm, wq_sorted and x_work must be 16-byte aligned");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(scales) & 1u) == 0 && (reinterpret_cast<uintptr_t>(y) & 1u) == 0,
               QLIN_ERR_ALIGNMENT, "scales and y must be 2-byte aligned");
  QLIN_DEVICE();
  cudaError_t e = launch_x_permute(x, T, K, perm, x_work, stream);
  if (e != cudaSuccess) return cuda_fail(e, "x_permute launch");
  QLIN_LAUNCH(launch_w4a16_gemm(x_work, T, N, K, wq_sorted, scales, zeros, y, stream), "w4a16_gemm launch");
}

int64_t qlin_w4a16_sequence_workspace_bytes(int64_t nsteps) {
  return nsteps < 0 ? -1 : w4a16_sequence_workspace_bytes(nsteps);
}

qlin_status qlin_w4a16_gemv_sequence(const qlin_w4a16_step* steps, int nsteps, int64_t group, void* workspace,
                                     cudaStream_t stream) {
  QLIN_REQUIRE(group == 128, QLIN_ERR_UNSUPPORTED, "group size %lld (only 128 is built)", (long long)group);
  QLIN_REQUIRE(nsteps >= 0, QLIN_ERR_INVALID_ARG, "nsteps=%d", nsteps);
  if (nsteps == 0) return ok();
  QLIN_REQUIRE(steps != nullptr, QLIN_ERR_INVALID_ARG, "null steps");
  QLIN_REQUIRE(workspace != nullptr, QLIN_ERR_INVALID_ARG, "null workspace");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 3u) == 0, QLIN_ERR_ALIGNMENT, "workspace must be 4-byte aligned");
  for (int s = 0; s < nsteps; ++s) {
    const qlin_w4a16_step& st = steps[s];
    QLIN_REQUIRE(st.count >= 1 && st.count <= QLIN_W4A16_MAX_GROUP, QLIN_ERR_INVALID_ARG,
                 "step %d: count=%d outside [1, %d]", s, st.count, QLIN_W4A16_MAX_GROUP);
    QLIN_REQUIRE(st.K > 0 && st.K % group == 0, QLIN_ERR_INVALID_ARG, "step %d: K=%lld is not a positive multiple of %lld",
                 s, (long long)st.K, (long long)group);
    QLIN_REQUIRE(w4a16_sequence_supported(st.K), QLIN_ERR_UNSUPPORTED, "step %d: K=%lld above 12288", s,
                 (long long)st.K);
    QLIN_REQUIRE(st.x && aligned16(st.x), st.x ? QLIN_ERR_ALIGNMENT : QLIN_ERR_INVALID_ARG,
                 "step %d: x must be non-null and 16-byte aligned", s);
    for (int p = 0; p < st.count; ++p) {
      QLIN_REQUIRE(st.N[p] >= 0 && st.N[p] < (int64_t(1) << 30), QLIN_ERR_INVALID_ARG, "step %d: bad N[%d]=%lld", s, p,
                   (long long)st.N[p]);
      if (st.N[p] == 0) continue;
      QLIN_REQUIRE(st.wq[p] && st.scales[p] && st.y[p], QLIN_ERR_INVALID_ARG, "step %d: null pointer for matrix %d", s, p);
      QLIN_REQUIRE(aligned16(st.wq[p]), QLIN_ERR_ALIGNMENT, "step %d: wq[%d] must be 16-byte aligned", s, p);
      QLIN_REQUIRE((reinterpret_cast<uintptr_t>(st.scales[p]) & 1u) == 0 && (reinterpret_cast<uintptr_t>(st.y[p]) & 1u) == 0,
                   QLIN_ERR_ALIGNMENT, "step %d: scales[%d] and y[%d] must be 2-byte aligned", s, p, p);
    }
  }
  QLIN_DEVICE();
  const cudaError_t e = launch_w4a16_sequence(steps, nsteps, static_cast<unsigned int*>(workspace), stream);
  if (e == cudaErrorInvalidValue || e == cudaErrorCooperativeLaunchTooLarge)
    return fail(QLIN_ERR_UNSUPPORTED, "no launch plan with one CTA per SM for this sequence (%s)", cudaGetErrorString(e));
  QLIN_LAUNCH(e, "w4a16_gemv_sequence launch");
}

qlin_status qlin_w4a16_gemv_sequence_noalloc(const qlin_w4a16_step* steps, int nsteps, int64_t group,
                                             cudaStream_t stream) {
  if (nsteps == 0) return qlin_w4a16_gemv_sequence(steps, nsteps, group, reinterpret_cast<void*>(16), stream);
  QLIN_DEVICE();
  unsigned int* ws = nullptr;
  const cudaError_t e = w4a16_sequence_static_workspace(&ws);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(sequence counters)");
  return qlin_w4a16_gemv_sequence(steps, nsteps, group, ws, stream);
}

static qlin_status quant_act_int8_checked(const void* x, qlin_dtype x_dtype, int64_t T, int64_t K, void* q,
                                          bool f16_codes, float* scale, int32_t* azp, cudaStream_t stream) {
  QLIN_REQUIRE(is_float_dtype(x_dtype), QLIN_ERR_INVALID_ARG, "x_dtype must be F16, BF16 or F32");
  QLIN_REQUIRE(T >= 0 && T <= kMaxDim && K > 0 && K <= kMaxDim, QLIN_ERR_INVALID_ARG, "bad sizes T=%lld K=%lld",
               (long long)T, (long long)K);
  QLIN_REQUIRE(K % 16 == 0, QLIN_ERR_ALIGNMENT, "K=%lld is not a multiple of 16", (long long)K);
  if (T == 0) return ok();
  QLIN_REQUIRE(x && q && scale, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(aligned16(x) && aligned16(q), QLIN_ERR_ALIGNMENT, "x and q must be 16-byte aligned");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(scale) & 3u) == 0 && (reinterpret_cast<uintptr_t>(azp) & 3u) == 0,
               QLIN_ERR_ALIGNMENT, "scale and azp must be 4-byte aligned");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_quant_act_int8(x, x_dtype, T, K, q, f16_codes, scale, azp, stream), "quant_act_int8 launch");
}

qlin_status qlin_quant_act_int8(const void* x, qlin_dtype x_dtype, int64_t T, int64_t K, int8_t* q,
                                float* scale, int32_t* azp, cudaStream_t stream) {
  return quant_act_int8_checked(x, x_dtype, T, K, q, false, scale, azp, stream);
}

qlin_status qlin_quant_act_int8_f16(const void* x, qlin_dtype x_dtype, int64_t T, int64_t K, void* q16,
                                    float* scale, int32_t* azp, cudaStream_t stream) {
  return quant_act_int8_checked(x, x_dtype, T, K, q16, true, scale, azp, stream);
}

qlin_status qlin_int8_row_sum(const int8_t* b, int64_t N, int64_t K, int32_t* azp_adj, cudaStream_t stream) {
  QLIN_REQUIRE(N >= 0 && N <= kMaxDim && K > 0 && K <= kMaxDim, QLIN_ERR_INVALID_ARG, "bad sizes N=%lld K=%lld",
               (long long)N, (long long)K);
  QLIN_REQUIRE(K % 16 == 0, QLIN_ERR_ALIGNMENT, "K=%lld is not a multiple of 16", (long long)K);
  if (N == 0) return ok();
  QLIN_REQUIRE(b && azp_adj, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(aligned16(b), QLIN_ERR_ALIGNMENT, "b must be 16-byte aligned");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(azp_adj) & 3u) == 0, QLIN_ERR_ALIGNMENT, "azp_adj must be 4-byte aligned");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_int8_row_sum(b, N, K, azp_adj, stream), "int8_row_sum launch");
}

}  // extern "C"

namespace {

// Operand forms of the W8A8 GEMM: int8 codes, or the same codes as exact
// fp16 values for B only or for both operands.
enum W8A8Form { kW8I8, kW8F16B, kW8F16 };

qlin_status w8a8_gemm_checked(const void* a, const void* b, W8A8Form form, int64_t T, int64_t N, int64_t K,
                           const float* scale_a, int64_t scale_a_numel, const float* scale_b,
                           int64_t scale_b_numel, const int32_t* azp, const int32_t* azp_adj,
                           const void* bias, qlin_dtype bias_dtype, void* out, qlin_dtype out_dtype,
                           cudaStream_t stream) {
  QLIN_REQUIRE(T >= 0 && T <= kMaxDim && N >= 0 && N <= kMaxDim && K > 0 && K <= kMaxDim, QLIN_ERR_INVALID_ARG,
               "bad sizes T=%lld N=%lld K=%lld", (long long)T, (long long)N, (long long)K);
  QLIN_REQUIRE(K % 16 == 0, QLIN_ERR_ALIGNMENT, "K=%lld is not a multiple of 16", (long long)K);
  QLIN_REQUIRE(out_dtype == QLIN_F16 || out_dtype == QLIN_BF16 || out_dtype == QLIN_I32, QLIN_ERR_INVALID_ARG,
               "out_dtype must be F16, BF16 or I32");
  const bool raw = out_dtype == QLIN_I32;
  if (!raw) {
    QLIN_REQUIRE(scale_a_numel == 1 || scale_a_numel == T, QLIN_ERR_INVALID_ARG,
                 "scale_a_numel=%lld must be 1 or T", (long long)scale_a_numel);
    QLIN_REQUIRE(scale_b_numel == 1 || scale_b_numel == N, QLIN_ERR_INVALID_ARG,
                 "scale_b_numel=%lld must be 1 or N", (long long)scale_b_numel);
    QLIN_REQUIRE(azp == nullptr || azp_adj != nullptr, QLIN_ERR_INVALID_ARG,
                 "per-token azp needs azp_adj (the per-channel sum of the weight codes)");
    QLIN_REQUIRE(bias == nullptr || is_float_dtype(bias_dtype), QLIN_ERR_INVALID_ARG,
                 "bias_dtype must be F16, BF16 or F32");
  }
  if (T == 0 || N == 0) return ok();
  QLIN_REQUIRE(a && b && out, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(raw || (scale_a && scale_b), QLIN_ERR_INVALID_ARG, "null scale pointer");
  QLIN_REQUIRE(aligned16(a) && aligned16(b) && aligned16(out), QLIN_ERR_ALIGNMENT,
               "a, b and out must be 16-byte aligned");
  QLIN_REQUIRE((N * dtype_bytes(out_dtype)) % 16 == 0, QLIN_ERR_ALIGNMENT,
               "the out row pitch (N x element size) must be a multiple of 16 bytes");
  QLIN_DEVICE();
  W8A8Epilogue epi;
  epi.scale_a = scale_a;
  epi.scale_a_per_row = scale_a_numel != 1;
  epi.scale_b = scale_b;
  epi.scale_b_per_col = scale_b_numel != 1;
  epi.azp = raw ? nullptr : azp;
  epi.azp_adj = raw ? nullptr : azp_adj;
  epi.bias = raw ? nullptr : bias;
  epi.bias_dtype = bias_dtype;
  epi.out_dtype = out_dtype;
  if (form == kW8F16) {
    QLIN_LAUNCH(launch_w8a8_gemm_f16(a, b, T, N, K, epi, out, stream), "w8a8_gemm_f16 launch");
  }
  QLIN_LAUNCH(launch_w8a8_gemm(static_cast<const int8_t*>(a), b, form == kW8F16B, T, N, K, epi, out, stream),
              "w8a8_gemm launch");
}

}  // namespace

extern "C" {

qlin_status qlin_w8a8_gemm(const int8_t* a, const int8_t* b, int64_t T, int64_t N, int64_t K,
                           const float* scale_a, int64_t scale_a_numel, const float* scale_b,
                           int64_t scale_b_numel, const int32_t* azp, const int32_t* azp_adj,
                           const void* bias, qlin_dtype bias_dtype, void* out, qlin_dtype out_dtype,
                           cudaStream_t stream) {
  return w8a8_gemm_checked(a, b, kW8I8, T, N, K, scale_a, scale_a_numel, scale_b, scale_b_numel, azp, azp_adj, bias,
                           bias_dtype, out, out_dtype, stream);
}

qlin_status qlin_w8a8_gemm_f16b(const int8_t* a, const void* b16, int64_t T, int64_t N, int64_t K,
                                const float* scale_a, int64_t scale_a_numel, const float* scale_b,
                                int64_t scale_b_numel, const int32_t* azp, const int32_t* azp_adj,
                                const void* bias, qlin_dtype bias_dtype, void* out, qlin_dtype out_dtype,
                                cudaStream_t stream) {
  return w8a8_gemm_checked(a, b16, kW8F16B, T, N, K, scale_a, scale_a_numel, scale_b, scale_b_numel, azp, azp_adj, bias,
                           bias_dtype, out, out_dtype, stream);
}

qlin_status qlin_w8a8_gemm_f16(const void* a16, const void* b16, int64_t T, int64_t N, int64_t K,
                               const float* scale_a, int64_t scale_a_numel, const float* scale_b,
                               int64_t scale_b_numel, const int32_t* azp, const int32_t* azp_adj, const void* bias,
                               qlin_dtype bias_dtype, void* out, qlin_dtype out_dtype, cudaStream_t stream) {
  return w8a8_gemm_checked(a16, b16, kW8F16, T, N, K, scale_a, scale_a_numel, scale_b, scale_b_numel, azp, azp_adj,
                           bias, bias_dtype, out, out_dtype, stream);
}

qlin_status qlin_int8_to_f16(const int8_t* src, int64_t count, void* dst, cudaStream_t stream) {
  QLIN_REQUIRE(count >= 0 && count <= (int64_t(1) << 40), QLIN_ERR_INVALID_ARG, "bad count=%lld", (long long)count);
  if (count == 0) return ok();
  QLIN_REQUIRE(src && dst, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(aligned16(src) && aligned16(dst), QLIN_ERR_ALIGNMENT, "src and dst must be 16-byte aligned");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_int8_to_f16(src, count, dst, stream), "int8_to_f16 launch");
}

qlin_status qlin_nvfp4_global_scale(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, float* g,
                                    cudaStream_t stream) {
  QLIN_REQUIRE(is_float_dtype(x_dtype), QLIN_ERR_INVALID_ARG, "x_dtype must be F16, BF16 or F32");
  QLIN_REQUIRE(rows >= 0 && K > 0 && rows * K / K == rows, QLIN_ERR_INVALID_ARG, "bad sizes");
  QLIN_REQUIRE(K % 16 == 0, QLIN_ERR_ALIGNMENT, "K=%lld is not a multiple of 16", (long long)K);
  QLIN_REQUIRE(g != nullptr && (rows == 0 || x != nullptr), QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(aligned16(x) && (reinterpret_cast<uintptr_t>(g) & 3u) == 0, QLIN_ERR_ALIGNMENT,
               "x must be 16-byte aligned and g 4-byte aligned");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_nvfp4_global_scale(x, x_dtype, rows, K, g, stream), "nvfp4_global_scale launch");
}

qlin_status qlin_arc_perm(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, int32_t* perm,
                          cudaStream_t stream) {
  QLIN_REQUIRE(is_float_dtype(x_dtype), QLIN_ERR_INVALID_ARG, "x_dtype must be F16, BF16 or F32");
  QLIN_REQUIRE(rows >= 0 && rows <= kMaxDim && K > 0 && K <= 16384, QLIN_ERR_INVALID_ARG,
               "bad sizes rows=%lld K=%lld (K <= 16384)", (long long)rows, (long long)K);
  QLIN_REQUIRE(K % 16 == 0, QLIN_ERR_ALIGNMENT, "K=%lld is not a multiple of 16", (long long)K);
  QLIN_REQUIRE(perm != nullptr && (rows == 0 || x != nullptr), QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(aligned16(x) && aligned16(perm), QLIN_ERR_ALIGNMENT, "x and perm must be 16-byte aligned");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_arc_perm(x, x_dtype, rows, K, perm, stream), "arc_perm launch");
}

int64_t qlin_nvfp4_sf_bytes(int64_t rows, int64_t K, qlin_sf_layout sf_layout) {
  if (rows < 0 || K <= 0 || K % 16 != 0) return -1;
  if (sf_layout == QLIN_SF_ROWS) return rows * (K / 16);
  if (sf_layout == QLIN_SF_MMA && K % 64 == 0) return (rows + 127) / 128 * (K / 64) * 512;
  return -1;
}

qlin_status qlin_nvfp4_sf_to_mma(const uint8_t* sf_rows, int64_t rows, int64_t K, uint8_t* sf_mma,
                                 cudaStream_t stream) {
  QLIN_REQUIRE(rows >= 0 && rows <= kMaxDim && K > 0 && K <= kMaxDim && K % 64 == 0, QLIN_ERR_INVALID_ARG,
               "bad sizes rows=%lld K=%lld (K a multiple of 64)", (long long)rows, (long long)K);
  if (rows == 0) return ok();
  QLIN_REQUIRE(sf_rows && sf_mma, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(sf_rows) & 3u) == 0 && aligned16(sf_mma), QLIN_ERR_ALIGNMENT,
               "sf_rows must be 4-byte and sf_mma 16-byte aligned");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_nvfp4_sf_to_mma(sf_rows, rows, K, sf_mma, stream), "nvfp4_sf_to_mma launch");
}

// Argument checks shared by the NVFP4 quantizer and its fused RMSNorm form
// (gamma != nullptr), then the launch.
static qlin_status quant_nvfp4_checked(const char* name, const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K,
                                       const void* gamma, float eps, const int32_t* perm, int64_t S,
                                       qlin_nvfp4_mode mode, const float* g, uint8_t* q, uint8_t* sf,
                                       qlin_sf_layout sf_layout, cudaStream_t stream) {
  QLIN_REQUIRE(sf_layout == QLIN_SF_ROWS || (sf_layout == QLIN_SF_MMA && (K + S) % 64 == 0), QLIN_ERR_INVALID_ARG,
               "sf_layout must be QLIN_SF_ROWS, or QLIN_SF_MMA with K+S a multiple of 64");
  QLIN_REQUIRE(is_float_dtype(x_dtype), QLIN_ERR_INVALID_ARG, "x_dtype must be F16, BF16 or F32");
  QLIN_REQUIRE(mode == QLIN_NVFP4_RESIDUAL || mode == QLIN_NVFP4_DUPLICATE, QLIN_ERR_INVALID_ARG, "bad mode");
  QLIN_REQUIRE(eps >= 0.0f && eps <= 3.4e38f, QLIN_ERR_INVALID_ARG, "eps must be a finite number >= 0");
  QLIN_REQUIRE(rows >= 0 && rows <= kMaxDim && K > 0, QLIN_ERR_INVALID_ARG, "bad sizes rows=%lld K=%lld",
               (long long)rows, (long long)K);
  QLIN_REQUIRE(K * dtype_bytes(x_dtype) <= (gamma ? 96 : 160) * 1024, QLIN_ERR_UNSUPPORTED,
               "a row of %lld elements does not fit the shared-memory staging buffer", (long long)K);
  QLIN_REQUIRE(S >= 0 && S <= K && S % 16 == 0, QLIN_ERR_INVALID_ARG, "S=%lld must be a multiple of 16 in [0, K]",
               (long long)S);
  QLIN_REQUIRE(K % 32 == 0 && (K + S) % 32 == 0, QLIN_ERR_ALIGNMENT,
               "K and K+S must be multiples of 32 (16-byte aligned packed rows)");
  if (rows == 0) return ok();
  QLIN_REQUIRE(x && g && q && sf, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(aligned16(x) && aligned16(q) && aligned16(perm), QLIN_ERR_ALIGNMENT,
               "x, q and perm must be 16-byte aligned");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(g) & 3u) == 0, QLIN_ERR_ALIGNMENT, "g must be 4-byte aligned");
  QLIN_REQUIRE(aligned16(gamma), QLIN_ERR_ALIGNMENT, "gamma must be 16-byte aligned");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_quant_nvfp4(x, x_dtype, rows, K, perm, S, mode, g, q, sf, sf_layout, gamma, eps, stream), name);
}

qlin_status qlin_quant_nvfp4(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, const int32_t* perm,
                             int64_t S, qlin_nvfp4_mode mode, const float* g, uint8_t* q, uint8_t* sf,
                             qlin_sf_layout sf_layout, cudaStream_t stream) {
  return quant_nvfp4_checked("quant_nvfp4 launch", x, x_dtype, rows, K, nullptr, 0.0f, perm, S, mode, g, q, sf,
                             sf_layout, stream);
}

qlin_status qlin_rmsnorm_quant_nvfp4(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, const void* gamma,
                                     float eps, const int32_t* perm, int64_t S, qlin_nvfp4_mode mode, const float* g,
                                     uint8_t* q, uint8_t* sf, qlin_sf_layout sf_layout, cudaStream_t stream) {
  QLIN_REQUIRE(rows == 0 || gamma != nullptr, QLIN_ERR_INVALID_ARG, "null gamma");
  return quant_nvfp4_checked("rmsnorm_quant_nvfp4 launch", x, x_dtype, rows, K, gamma, eps, perm, S, mode, g, q, sf,
                             sf_layout, stream);
}

qlin_status qlin_nvfp4_gemm(const uint8_t* a, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb,
                            int64_t T, int64_t N, int64_t K, const float* g_a, const float* g_b, void* out,
                            qlin_dtype out_dtype, cudaStream_t stream) {
  QLIN_REQUIRE(T >= 0 && T <= kMaxDim && N >= 0 && N <= kMaxDim && K > 0 && K <= kMaxDim, QLIN_ERR_INVALID_ARG,
               "bad sizes T=%lld N=%lld K=%lld", (long long)T, (long long)N, (long long)K);
  QLIN_REQUIRE(K % 64 == 0, QLIN_ERR_INVALID_ARG, "K=%lld is not a multiple of 64", (long long)K);
  QLIN_REQUIRE(out_dtype == QLIN_F16 || out_dtype == QLIN_BF16, QLIN_ERR_INVALID_ARG, "out_dtype must be F16 or BF16");
  if (T == 0 || N == 0) return ok();
  QLIN_REQUIRE(a && sfa && b && sfb && g_a && g_b && out, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(aligned16(a) && aligned16(b) && aligned16(out), QLIN_ERR_ALIGNMENT,
               "a, b and out must be 16-byte aligned");
  QLIN_REQUIRE(aligned16(sfa) && aligned16(sfb), QLIN_ERR_ALIGNMENT,
               "sfa and sfb (QLIN_SF_MMA layout) must be 16-byte aligned");
  QLIN_REQUIRE((N * 2) % 16 == 0, QLIN_ERR_ALIGNMENT, "the out row pitch (2N bytes) must be a multiple of 16");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_nvfp4_gemm(a, sfa, b, sfb, T, N, K, g_a, g_b, out, out_dtype, stream), "nvfp4_gemm launch");
}

qlin_status qlin_hadamard(const void* x, qlin_dtype dtype, int64_t rows, int64_t K, qlin_hadamard_kind kind,
                          int64_t n, const int8_t* signs, void* y, cudaStream_t stream) {
  QLIN_REQUIRE(is_float_dtype(dtype), QLIN_ERR_INVALID_ARG, "dtype must be F16, BF16 or F32");
  QLIN_REQUIRE(kind == QLIN_HADAMARD_SYLVESTER || kind == QLIN_HADAMARD_REGULAR, QLIN_ERR_INVALID_ARG,
               "unknown Hadamard kind %d", static_cast<int>(kind));
  const bool pow2 = n >= 2 && (n & (n - 1)) == 0;
  QLIN_REQUIRE(kind != QLIN_HADAMARD_SYLVESTER || (pow2 && n <= 8192), QLIN_ERR_INVALID_ARG,
               "n=%lld: the Sylvester transform takes a power of two in [2, 8192]", (long long)n);
  QLIN_REQUIRE(kind != QLIN_HADAMARD_REGULAR || n == 4 || n == 16 || n == 64 || n == 256, QLIN_ERR_INVALID_ARG,
               "n=%lld: the regular transform takes 4, 16, 64 or 256", (long long)n);
  QLIN_REQUIRE(rows >= 0 && rows <= kMaxDim && K > 0 && K <= kMaxDim, QLIN_ERR_INVALID_ARG,
               "bad sizes rows=%lld K=%lld", (long long)rows, (long long)K);
  QLIN_REQUIRE(K % n == 0 && K % 8 == 0, QLIN_ERR_INVALID_ARG, "K=%lld must be a multiple of n=%lld and of 8",
               (long long)K, (long long)n);
  if (rows == 0) return ok();
  QLIN_REQUIRE(x && y, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(aligned16(x) && aligned16(y), QLIN_ERR_ALIGNMENT, "x and y must be 16-byte aligned");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(signs) & 7u) == 0, QLIN_ERR_ALIGNMENT, "signs must be 8-byte aligned");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_hadamard(x, dtype, rows, K, kind, n, signs, y, stream), "hadamard launch");
}

int64_t qlin_mx_sf_bytes(int64_t rows, int64_t K, qlin_sf_layout sf_layout) {
  if (rows < 0 || K <= 0 || K % 32 != 0) return -1;
  if (sf_layout == QLIN_SF_ROWS) return rows * (K / 32);
  if (sf_layout == QLIN_SF_MMA) return (rows + 127) / 128 * ((K + 127) / 128) * 512;
  return -1;
}

qlin_status qlin_quant_mx(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, qlin_mx_fmt fmt, uint8_t* q,
                          uint8_t* sf, qlin_sf_layout sf_layout, cudaStream_t stream) {
  QLIN_REQUIRE(is_float_dtype(x_dtype), QLIN_ERR_INVALID_ARG, "x_dtype must be F16, BF16 or F32");
  QLIN_REQUIRE(fmt == QLIN_MX_FP8_E4M3 || fmt == QLIN_MX_FP4_E2M1, QLIN_ERR_INVALID_ARG, "unknown MX format %d",
               static_cast<int>(fmt));
  QLIN_REQUIRE(sf_layout == QLIN_SF_ROWS || sf_layout == QLIN_SF_MMA, QLIN_ERR_INVALID_ARG, "unknown sf_layout");
  QLIN_REQUIRE(rows >= 0 && rows <= kMaxDim && K > 0 && K <= kMaxDim, QLIN_ERR_INVALID_ARG,
               "bad sizes rows=%lld K=%lld", (long long)rows, (long long)K);
  QLIN_REQUIRE(K % 32 == 0, QLIN_ERR_INVALID_ARG, "K=%lld is not a multiple of 32", (long long)K);
  if (rows == 0) return ok();
  QLIN_REQUIRE(x && q && sf, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(aligned16(x) && aligned16(q), QLIN_ERR_ALIGNMENT, "x and q must be 16-byte aligned");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_quant_mx(x, x_dtype, rows, K, fmt, q, sf, sf_layout, stream), "quant_mx launch");
}

qlin_status qlin_mx_gemm(const uint8_t* a, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb, int64_t T,
                         int64_t N, int64_t K, qlin_mx_fmt fmt, void* out, qlin_dtype out_dtype, cudaStream_t stream) {
  QLIN_REQUIRE(fmt == QLIN_MX_FP8_E4M3 || fmt == QLIN_MX_FP4_E2M1, QLIN_ERR_INVALID_ARG, "unknown MX format %d",
               static_cast<int>(fmt));
  QLIN_REQUIRE(T >= 0 && T <= kMaxDim && N >= 0 && N <= kMaxDim && K > 0 && K <= kMaxDim, QLIN_ERR_INVALID_ARG,
               "bad sizes T=%lld N=%lld K=%lld", (long long)T, (long long)N, (long long)K);
  const int64_t kmul = fmt == QLIN_MX_FP8_E4M3 ? 32 : 64;
  QLIN_REQUIRE(K % kmul == 0, QLIN_ERR_INVALID_ARG, "K=%lld is not a multiple of %lld", (long long)K,
               (long long)kmul);
  QLIN_REQUIRE(out_dtype == QLIN_F16 || out_dtype == QLIN_BF16, QLIN_ERR_INVALID_ARG, "out_dtype must be F16 or BF16");
  if (T == 0 || N == 0) return ok();
  QLIN_REQUIRE(a && sfa && b && sfb && out, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(aligned16(a) && aligned16(b) && aligned16(out) && aligned16(sfa) && aligned16(sfb), QLIN_ERR_ALIGNMENT,
               "a, b, sfa, sfb and out must be 16-byte aligned");
  QLIN_REQUIRE((N * 2) % 16 == 0, QLIN_ERR_ALIGNMENT, "the out row pitch (2N bytes) must be a multiple of 16");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_mx_gemm(a, sfa, b, sfb, T, N, K, fmt, out, out_dtype, stream), "mx_gemm launch");
}

qlin_status qlin_quant_fp8(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, uint8_t* q, float* scale,
                           cudaStream_t stream) {
  QLIN_REQUIRE(is_float_dtype(x_dtype), QLIN_ERR_INVALID_ARG, "x_dtype must be F16, BF16 or F32");
  QLIN_REQUIRE(rows >= 0 && rows <= kMaxDim && K > 0 && K <= kMaxDim, QLIN_ERR_INVALID_ARG,
               "bad sizes rows=%lld K=%lld", (long long)rows, (long long)K);
  QLIN_REQUIRE(K % 16 == 0, QLIN_ERR_ALIGNMENT, "K=%lld is not a multiple of 16", (long long)K);
  if (rows == 0) return ok();
  QLIN_REQUIRE(x && q && scale, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(aligned16(x) && aligned16(q), QLIN_ERR_ALIGNMENT, "x and q must be 16-byte aligned");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(scale) & 3u) == 0, QLIN_ERR_ALIGNMENT, "scale must be 4-byte aligned");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_quant_fp8(x, x_dtype, rows, K, q, scale, stream), "quant_fp8 launch");
}

qlin_status qlin_fp8_gemm(const uint8_t* a, const uint8_t* b, int64_t T, int64_t N, int64_t K, const float* scale_a,
                          const float* scale_b, const void* bias, qlin_dtype bias_dtype, void* out,
                          qlin_dtype out_dtype, cudaStream_t stream) {
  QLIN_REQUIRE(T >= 0 && T <= kMaxDim && N >= 0 && N <= kMaxDim && K > 0 && K <= kMaxDim, QLIN_ERR_INVALID_ARG,
               "bad sizes T=%lld N=%lld K=%lld", (long long)T, (long long)N, (long long)K);
  QLIN_REQUIRE(K % 16 == 0, QLIN_ERR_ALIGNMENT, "K=%lld is not a multiple of 16", (long long)K);
  QLIN_REQUIRE(out_dtype == QLIN_F16 || out_dtype == QLIN_BF16, QLIN_ERR_INVALID_ARG, "out_dtype must be F16 or BF16");
  QLIN_REQUIRE(bias == nullptr || is_float_dtype(bias_dtype), QLIN_ERR_INVALID_ARG,
               "bias_dtype must be F16, BF16 or F32");
  if (T == 0 || N == 0) return ok();
  QLIN_REQUIRE(a && b && scale_a && scale_b && out, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(aligned16(a) && aligned16(b) && aligned16(out), QLIN_ERR_ALIGNMENT,
               "a, b and out must be 16-byte aligned");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(scale_a) & 3u) == 0 && (reinterpret_cast<uintptr_t>(scale_b) & 3u) == 0,
               QLIN_ERR_ALIGNMENT, "scale_a and scale_b must be 4-byte aligned");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(bias) & 3u) == 0, QLIN_ERR_ALIGNMENT, "bias must be 4-byte aligned");
  QLIN_REQUIRE((N * 2) % 16 == 0, QLIN_ERR_ALIGNMENT, "the out row pitch (2N bytes) must be a multiple of 16");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_fp8_gemm(a, b, T, N, K, scale_a, scale_b, bias, bias_dtype, out, out_dtype, stream),
              "fp8_gemm launch");
}

qlin_status qlin_rmsnorm_quant(const void* x, qlin_dtype x_dtype, int64_t rows, int64_t K, const void* gamma,
                               float eps, qlin_qfmt fmt, void* q, float* scale, cudaStream_t stream) {
  QLIN_REQUIRE(is_float_dtype(x_dtype), QLIN_ERR_INVALID_ARG, "x_dtype must be F16, BF16 or F32");
  QLIN_REQUIRE(fmt == QLIN_QFMT_INT8 || fmt == QLIN_QFMT_FP8_E4M3, QLIN_ERR_INVALID_ARG, "unknown output format %d",
               static_cast<int>(fmt));
  QLIN_REQUIRE(eps >= 0.0f && eps <= 3.4e38f, QLIN_ERR_INVALID_ARG, "eps must be a finite number >= 0");
  QLIN_REQUIRE(rows >= 0 && rows <= kMaxDim && K > 0 && K <= kMaxDim, QLIN_ERR_INVALID_ARG,
               "bad sizes rows=%lld K=%lld", (long long)rows, (long long)K);
  QLIN_REQUIRE(K % 16 == 0, QLIN_ERR_ALIGNMENT, "K=%lld is not a multiple of 16", (long long)K);
  if (rows == 0) return ok();
  QLIN_REQUIRE(x && gamma && q && scale, QLIN_ERR_INVALID_ARG, "null pointer");
  QLIN_REQUIRE(aligned16(x) && aligned16(gamma) && aligned16(q), QLIN_ERR_ALIGNMENT,
               "x, gamma and q must be 16-byte aligned");
  QLIN_REQUIRE((reinterpret_cast<uintptr_t>(scale) & 3u) == 0, QLIN_ERR_ALIGNMENT, "scale must be 4-byte aligned");
  QLIN_DEVICE();
  QLIN_LAUNCH(launch_rmsnorm_quant(x, x_dtype, rows, K, gamma, eps, fmt, q, scale, stream), "rmsnorm_quant launch");
}

}  // extern "C"
