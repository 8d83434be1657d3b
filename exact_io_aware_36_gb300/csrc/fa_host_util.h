// fa_host_util.h -- host helpers shared by the launchers: TMA descriptors
// (cached per shape and address), the per-kernel shared-memory limit and the
// SM count (each set or read once per device).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// Every make_tmap_* returns a descriptor from a per-shape cache: a call whose
// base address, sizes, strides, box and element type equal an earlier one's
// reuses that call's encoding (descriptors hold no other state).
//
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

// cudaFuncAttributeMaxDynamicSharedMemorySize of `kernel` in the current
// device's context, set on the first call per (device, kernel) only.
// Returns 0 or a cudaError_t value.
int set_max_dynamic_smem(const void* kernel, int bytes);

// Number of SMs of the current device (read once per device).  Returns 0 or
// a cudaError_t value.
int sm_count(int* nsm);

// Counts since the library was loaded: descriptors encoded, descriptors
// served from the cache, shared-memory limits set.
void host_cache_stats(unsigned long long* encoded, unsigned long long* reused,
                      unsigned long long* attr_set);

}  // namespace fa
