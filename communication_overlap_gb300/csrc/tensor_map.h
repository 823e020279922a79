// Host-side TMA tensor-map encoding shared by the GEMM and the reorder.
#pragma once

#include <cstdint>

#include <cuda.h>

namespace fo {

// 2-D bf16 tensor of `outer` rows x `inner` columns, row-major and densely
// packed (row pitch inner * 2 bytes), read or written in boxes of
// box_outer x box_inner elements; swizzle128 selects the 128-byte swizzle
// (else none).  Returns false if the driver entry point is unavailable or
// the encoding is rejected.
bool encode_tensor_map_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                          uint32_t box_inner, uint32_t box_outer, bool swizzle128);

}  // namespace fo
