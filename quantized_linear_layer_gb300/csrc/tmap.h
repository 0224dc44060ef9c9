// Host helper: TMA tensor maps for row-major 2-D byte matrices.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace qlin {

// Tiled tensor map over a row-major uint8 matrix of `rows` x `cols` bytes
// (dense rows, row pitch = cols, which must be a multiple of 16), loading
// boxes of box_rows x box_cols bytes; out-of-range parts of a box are filled
// with zeros.  swizzle_bytes selects the shared-memory layout of the box:
//   0    plain rows;
//   64   box_cols = 64: 16-byte chunk c of row r stored at chunk
//        c ^ ((r / 2) % 4) of the row (destination 512-byte aligned);
//   128  box_cols = 128: 16-byte chunk c of row r stored at chunk c ^ (r % 8)
//        of the row (destination 1024-byte aligned).
cudaError_t make_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                            uint32_t box_rows, int swizzle_bytes = 0);

// Tiled tensor map over a row-major matrix of `rows` rows of `cols8` 8-byte
// elements (row pitch cols8 * 8 bytes, a multiple of 16), loading boxes of
// box_rows x box_cols8 elements (box_cols8 <= 256) into plain dense rows;
// out-of-range parts of a box are filled with zeros.
cudaError_t make_tmap_2d_u64(CUtensorMap* map, const void* base, uint64_t cols8, uint64_t rows, uint32_t box_cols8,
                             uint32_t box_rows);

}  // namespace qlin
