// Host helper: TMA tensor maps for row-major 2-D byte matrices.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace qlin {

// Tiled tensor map over a row-major uint8 matrix of `rows` x `cols` bytes
// (dense rows, row pitch = cols, which must be a multiple of 16), loading
// boxes of box_rows x box_cols bytes with no swizzle; out-of-range parts of a
// box are filled with zeros.
cudaError_t make_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                            uint32_t box_rows);

}  // namespace qlin
