// Temporary: tensor-core GEMM launchers not yet built.
#include "qlin_internal.h"
namespace qlin {
cudaError_t launch_nvfp4_gemm(const uint8_t*, const uint8_t*, const uint8_t*, const uint8_t*, int64_t, int64_t,
                              int64_t, const float*, const float*, void*, qlin_dtype, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace qlin
