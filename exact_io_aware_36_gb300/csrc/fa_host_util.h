// fa_host_util.h -- host helpers shared by the launchers: TMA descriptors.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// Encodes a 3-D tiled TMA descriptor over a contiguous bf16 tensor
// [T, H, d] (dims innermost first: d, H, T) with a box of 64 columns x 1
// head x box_rows tokens, 128-byte swizzle, zero fill out of bounds.
// Returns 0 or a cudaError_t value.
int make_tmap_bf16_3d(CUtensorMap* map, const void* base, int d, int H, long long T,
                      int box_rows);

}  // namespace fa
