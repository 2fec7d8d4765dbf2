// kda_tma_host.h -- host-side construction of TMA tensor maps over the library's token-major
// [T, H, d] tensors (defined in kda_chunked.cu).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace kda {

// A 3-D map over a [T, H, d] tensor of bf16 or fp32 elements: dims (channel, head, token),
// boxes of box_d channels x 1 head x box_t tokens, 128-byte swizzle or none. Out-of-range
// parts of a box read as zero. Returns false if the driver's encoder is unavailable or
// rejects the map (the base must be 16-byte aligned and d * element size a multiple of 16).
bool tensor_map_3d(CUtensorMap *map, const void *base, bool bf16, int64_t T, int H, int d, uint32_t box_d,
                   uint32_t box_t, bool swizzle128);

}  // namespace kda
