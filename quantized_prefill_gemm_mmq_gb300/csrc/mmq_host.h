// mmq_host.h -- host-side helpers shared by the libmmq entry points:
// argument checks, the architecture check, and TMA tensor-map encoding.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "mmq.h"

namespace mmq {

// MMQ_OK if the current device is compute capability 10.3 (cached per device).
int check_arch();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch-error translation: clears the sticky-free error state and maps it.
int launch_status();

// 2-D tiled tensor map over a row-major array: `inner` elements per row of
// `elem_bytes` each, `rows` rows, `row_stride_bytes` apart; box of
// box_inner x box_rows elements; swizzle as given.  Returns MMQ_OK or
// MMQ_ERR_DRIVER.
int make_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, uint64_t inner,
                 uint64_t rows, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                 CUtensorMapSwizzle swizzle);
// 4-D tiled map: dims innermost first, strides of dims 1..3 in bytes (each a
// multiple of 16, in any order), box extents per dim
int make_tmap_4d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, const uint64_t (&dims)[4],
                 const uint64_t (&strides_bytes)[3], const uint32_t (&box)[4], CUtensorMapSwizzle swizzle);

}  // namespace mmq
