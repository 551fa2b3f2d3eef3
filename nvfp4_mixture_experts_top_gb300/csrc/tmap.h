// tmap.h -- TMA tensor-map creation (driver entry point fetched through the
// runtime, so the library does not link libcuda directly).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4moe {

// 2-D uint8 tensor [rows, inner] with row pitch `pitch` bytes; box of
// box_inner bytes x box_rows rows; swizzle_bytes = 0 (none), 64 or 128.
// Out-of-bounds box elements are zero-filled by the copy.
cudaError_t make_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t pitch,
                            uint32_t box_inner, uint32_t box_rows, int swizzle_bytes);

// 2-D fp32 tensor [rows, inner] with row pitch `pitch_bytes`; box of
// box_inner x box_rows elements, no swizzle (used as the destination of TMA
// reduce-add; box elements outside the tensor are neither read nor written).
cudaError_t make_tmap_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t pitch_bytes,
                             uint32_t box_inner, uint32_t box_rows);

}  // namespace nvfp4moe
