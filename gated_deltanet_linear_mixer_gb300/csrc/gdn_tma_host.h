// Host-side creation of TMA tensor maps (cuTensorMapEncodeTiled), reached
// through the runtime's driver entry point so the library does not link the
// driver library directly.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// A 2-D row-major bf16 matrix [rows, cols] with a row pitch of `pitch_elems`
// elements, read in boxes of box_rows x box_cols with the 128-byte swizzle
// (box_cols * 2 must be <= 128).  Returns false on failure.
bool make_tma_map_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                          uint64_t pitch_elems, uint32_t box_rows, uint32_t box_cols);
// The same for fp32 elements (box_cols * 4 <= 128).
bool make_tma_map_f32_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                         uint64_t pitch_elems, uint32_t box_rows, uint32_t box_cols);

}  // namespace gdn
