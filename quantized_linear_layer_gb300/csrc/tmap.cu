// Host helper: TMA tensor maps, encoded through the driver entry point that
// the runtime hands out (no link-time dependency on libcuda).
#include <cudaTypedefs.h>
#include <mutex>

#include "tmap.h"

namespace qlin {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_status = cudaSuccess;

void resolve_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  g_encode_status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (g_encode_status == cudaSuccess && (q != cudaDriverEntryPointSuccess || fn == nullptr))
    g_encode_status = cudaErrorNotSupported;
  if (g_encode_status == cudaSuccess) g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

cudaError_t make_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                            uint32_t box_rows, int swizzle_bytes) {
  std::call_once(g_encode_once, resolve_encode);
  if (g_encode == nullptr) return g_encode_status != cudaSuccess ? g_encode_status : cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};  // bytes between rows
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t elem_strides[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                        elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                        : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_2d_u64(CUtensorMap* map, const void* base, uint64_t cols8, uint64_t rows, uint32_t box_cols8,
                             uint32_t box_rows) {
  std::call_once(g_encode_once, resolve_encode);
  if (g_encode == nullptr) return g_encode_status != cudaSuccess ? g_encode_status : cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols8, rows};
  const cuuint64_t strides[1] = {cols8 * 8};  // bytes between rows
  const cuuint32_t box[2] = {box_cols8, box_rows};
  const cuuint32_t elem_strides[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(base), dims, strides, box,
                        elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace qlin
