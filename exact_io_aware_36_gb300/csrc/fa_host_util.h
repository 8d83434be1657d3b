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

// As make_tmap_bf16_3d with a box of 64 columns x box_h heads x box_t
// tokens (a box over several heads of several tokens).
int make_tmap_bf16_3d_box(CUtensorMap* map, const void* base, int d, int H, long long T,
                          int box_h, int box_t);

// As make_tmap_bf16_3d over a float32 tensor [T, H, d], with a box of 32
// columns (128 bytes) x 1 head x box_rows tokens.
int make_tmap_f32_3d(CUtensorMap* map, const void* base, int d, int H, long long T, int box_rows);

// Encodes a 3-D tiled TMA descriptor over a byte tensor (e4m3 codes) with
// dims (innermost first) n0, n1, n2, byte strides s1 (of dim 1) and s2 (of
// dim 2), box b0 x b1 x b2, 128-byte swizzle (b0 = 128), zero fill.  s1 and
// s2 must be multiples of 16.  Returns 0 or a cudaError_t value.
int make_tmap_u8_3d(CUtensorMap* map, const void* base, long long n0, long long n1, long long n2,
                    long long s1, long long s2, int b0, int b1, int b2);

}  // namespace fa
