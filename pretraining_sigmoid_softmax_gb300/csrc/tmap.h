// TMA descriptors shared by the tensor-core kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace moe {

// 2-D tensor map over a row-major [outer, inner] bf16 matrix with boxes of
// box_inner x box_outer elements and the 128-byte swizzle (box_inner * 2 <= 128). Elements
// outside the matrix read as zero. Returns false when the driver rejects the map (base not
// 16-byte aligned, row pitch not a multiple of 16 bytes, box too large).
bool make_tmap_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                       uint32_t box_inner, uint32_t box_outer);

// The same over a row-major [outer, inner] fp32 matrix (box_inner * 4 <= 128).
bool make_tmap_f32_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                      uint32_t box_inner, uint32_t box_outer);

}  // namespace moe
