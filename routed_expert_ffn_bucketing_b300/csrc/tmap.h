// Tiled TMA tensor maps of 2-D row-major arrays (host side), for the tensor-core kernels.
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace moe {

// True when the driver's tensor-map encoder is available.
bool tmap_available();

// A rows x inner array of elements of type dt (row stride row_bytes, a multiple of 16), boxes of
// box_inner x box_rows elements with the given swizzle; out-of-range boxes read zeros.
bool tmap_encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw);

}  // namespace moe
