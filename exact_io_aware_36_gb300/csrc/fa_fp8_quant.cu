// fa_fp8_quant.cu -- incoherent processing and per-block e4m3 quantization
// of Q, K and V for the FP8 forward (sm_103a).
//
// Method ("FlashAttention: Faster Attention Without Dropping a Single
// Interaction", FA3: per-block quantization, and the same random orthogonal
// Hadamard transform applied to Q and K so that (QM)(KM)^T = QK^T before
// quantization).  Here M = D H with D = diag(signs) and H the unnormalised
// Sylvester Hadamard matrix, so (QM)(KM)^T = d QK^T and the forward divides
// the scores by d.  One block of 128 rows of one head of one sequence shares
// one scale, amax / 448 (e4m3's largest finite value).
//
// Every step that decides a code is taken in float32 in a fixed order, so the
// codes do not depend on the schedule: the sign flip (exact), the butterfly
// with strides 1, 2, 4, ..., 64 ((a, b) -> (a + b, a - b)), the maximum, the
// divisions amax / 448 (the stored scale) and 448 / amax (the block's
// reciprocal, IEEE, round to nearest), the product x * (448 / amax), and the
// conversion to e4m3 (round to nearest even, saturated).
//
// Two kernels, each one pass over its input with the block's values held in
// registers from the load to the codes: Q and K with one thread per row
// (the butterfly entirely in registers), V with one warp per row, 4 columns
// per lane, and a shared-memory tile for its transposed codes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kD = 128;
constexpr int kRows = 128;

__device__ __forceinline__ bool block_bounds(const QuantParams& p, int b, long long* seq0, int* L) {
  if (p.cu_seqlens) {
    const int c0 = __ldg(p.cu_seqlens + b);
    const int c1 = __ldg(p.cu_seqlens + b + 1);
    if ((b == 0 && c0 != 0) || c1 < c0 || (long long)c1 > p.T || c1 - c0 > p.N) return false;
    *seq0 = c0;
    *L = c1 - c0;
  } else {
    *seq0 = (long long)b * p.N;
    *L = p.N;
  }
  return true;
}

// Two e4m3 codes of (lo, hi), lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float block_amax(float m, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  return fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
}

// The block's scale (amax / 448) and the reciprocal its values are scaled
// by (448 / amax), both 1 for an all-zero block.
__device__ __forceinline__ void block_scales(float amax, float* scale, float* inv) {
  *scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  *inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
}

// Q and K: one thread per row (token) of one head, the whole row of d = 128
// in registers: the sign flip, the butterfly with strides 1, 2, ..., 64
// ((a, b) -> (a + b, a - b), a the lower index), the row's |max|, the
// block's max (128 rows, one block), then codes = e4m3(x * inv) written as
// 128 bytes per row.  One pass over the input; grid (B * nblk, Hq + Hkv),
// y < Hq: Q, else K.
__global__ void __launch_bounds__(kRows, 2) quant_qk_kernel(const QuantParams p) {
  __shared__ float red[4];
  __shared__ __align__(16) float sg[kD];
  const bool isq = (int)blockIdx.y < p.Hq;
  const int h = isq ? blockIdx.y : blockIdx.y - p.Hq;
  const int H = isq ? p.Hq : p.Hkv;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(isq ? p.q : p.k);
  const int bi = blockIdx.x;
  const int b = bi / p.nblk;
  const int i = bi % p.nblk;
  long long seq0;
  int L;
  if (!block_bounds(p, b, &seq0, &L)) {
    if (threadIdx.x == 0) record_status(p.status, FA_ERR_CU_SEQLENS);
    return;
  }
  float* sc_out = (isq ? p.q_scale : p.k_scale) + (long long)h * p.B * p.nblk + bi;
  const int r0 = kRows * i;
  const int rows = min(kRows, L - r0);
  if (rows <= 0) {                                 // uniform over the block
    if (threadIdx.x == 0) *sc_out = 1.f;
    return;
  }
  sg[threadIdx.x] = __ldg(p.signs + threadIdx.x);
  const int r = threadIdx.x;
  const bool valid = r < rows;
  const long long row = ((seq0 + r0 + r) * H + h) * kD;
  float v[kD];
  if (valid) {
    uint4 raw[kD / 8];
#pragma unroll
    for (int c = 0; c < kD / 8; ++c) raw[c] = reinterpret_cast<const uint4*>(x + row)[c];
#pragma unroll
    for (int c = 0; c < kD / 8; ++c) {
      const uint32_t w[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[8 * c + 2 * e] = __uint_as_float(w[e] << 16);
        v[8 * c + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
      }
    }
  } else {
#pragma unroll
    for (int c = 0; c < kD; ++c) v[c] = 0.f;
  }
  __syncthreads();                                 // sg
#pragma unroll
  for (int c = 0; c < kD; ++c) v[c] *= sg[c];
#pragma unroll
  for (int st = 0; st < 7; ++st) {                 // strides 1, 2, 4, ..., 64
    const int hs = 1 << st;
#pragma unroll
    for (int k = 0; k < kD / 2; ++k) {             // pair k: (c, c + hs)
      const int c = (k / hs) * 2 * hs + k % hs;
      const float a = v[c], bb = v[c + hs];
      v[c] = a + bb;
      v[c + hs] = a - bb;
    }
  }
  float m = 0.f;
#pragma unroll
  for (int c = 0; c < kD; c += 2) m = fmax3(m, fabsf(v[c]), fabsf(v[c + 1]));
  const float amax = block_amax(m, red);
  float scale, inv;
  block_scales(amax, &scale, &inv);
  if (threadIdx.x == 0) *sc_out = scale;
  if (!valid) return;
  uint8_t* codes = (isq ? p.q8 : p.k8) + row;
#pragma unroll
  for (int c = 0; c < kD; c += 16) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = e4m3x2(v[c + 4 * e] * inv, v[c + 4 * e + 1] * inv) |
             (e4m3x2(v[c + 4 * e + 2] * inv, v[c + 4 * e + 3] * inv) << 16);
    reinterpret_cast<uint4*>(codes)[c / 16] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// V: codes transposed into [Hkv, 128, B * nblk * 128], scales, and the largest
// scale per kv head (v_smax, zeroed before).  grid (B * nblk, Hkv).  A warp
// takes rows warp, warp + 4, ... (4 columns per lane) and keeps them (as
// bf16) from the load to the codes; the codes go through a shared-memory
// tile so that each column of 128 keys is written contiguously.
__global__ void __launch_bounds__(kRows) quant_v_kernel(const QuantParams p) {
  constexpr int kPitch = kRows + 4;               // bytes per column row in the transpose
  constexpr int kRowsPerWarp = kRows / 4;
  __shared__ float red[4];
  __shared__ __align__(16) uint8_t tile[kD * kPitch];
  const int g = blockIdx.y;
  const int bi = blockIdx.x;
  const int b = bi / p.nblk;
  const int i = bi % p.nblk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  long long seq0;
  int L;
  if (!block_bounds(p, b, &seq0, &L)) {
    if (threadIdx.x == 0) record_status(p.status, FA_ERR_CU_SEQLENS);
    return;
  }
  const int r0 = kRows * i;
  const int rows = max(0, min(kRows, L - r0));
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(p.v);
  for (int w = threadIdx.x; w < kD * kPitch / 4; w += kRows) reinterpret_cast<uint32_t*>(tile)[w] = 0u;
  uint2 raw[kRowsPerWarp];
#pragma unroll
  for (int j = 0; j < kRowsPerWarp; ++j) {
    const int r = warp + 4 * j;
    raw[j] = r < rows ? *reinterpret_cast<const uint2*>(x + ((seq0 + r0 + r) * p.Hkv + g) * kD + 4 * lane)
                      : make_uint2(0u, 0u);
  }
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < kRowsPerWarp; ++j) {
    const float a0 = __uint_as_float(raw[j].x << 16), a1 = __uint_as_float(raw[j].x & 0xFFFF0000u);
    const float a2 = __uint_as_float(raw[j].y << 16), a3 = __uint_as_float(raw[j].y & 0xFFFF0000u);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(a2), fabsf(a3))));
  }
  const float amax = block_amax(m, red);          // also orders the zero fill before the codes
  float scale, inv;
  block_scales(amax, &scale, &inv);
  if (threadIdx.x == 0) {
    p.v_scale[(long long)g * p.B * p.nblk + bi] = scale;
    if (rows > 0) atomicMax(reinterpret_cast<unsigned int*>(p.v_smax + g), __float_as_uint(scale));
  }
#pragma unroll
  for (int j = 0; j < kRowsPerWarp; ++j) {
    const int r = warp + 4 * j;
    if (r >= rows) break;
    const float a0 = __uint_as_float(raw[j].x << 16), a1 = __uint_as_float(raw[j].x & 0xFFFF0000u);
    const float a2 = __uint_as_float(raw[j].y << 16), a3 = __uint_as_float(raw[j].y & 0xFFFF0000u);
    const uint32_t c = e4m3x2(a0 * inv, a1 * inv) | (e4m3x2(a2 * inv, a3 * inv) << 16);
#pragma unroll
    for (int e = 0; e < 4; ++e) tile[(4 * lane + e) * kPitch + r] = (uint8_t)(c >> (8 * e));
  }
  __syncthreads();
  // column c of this block: 128 key codes, one 4-byte word per lane
  uint8_t* dst = p.v8t + (long long)g * kD * p.vt_stride + (long long)bi * kRows;
  for (int c = warp; c < kD; c += 4)
    *reinterpret_cast<uint32_t*>(dst + (long long)c * p.vt_stride + 4 * lane) =
        *reinterpret_cast<const uint32_t*>(tile + c * kPitch + 4 * lane);
}

}  // namespace

int launch_fp8_quantize(const QuantParams& p, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cudaError_t e = cudaMemsetAsync(p.v_smax, 0, sizeof(float) * p.Hkv, stream);
  if (e != cudaSuccess) return (int)e;
  const unsigned nb = (unsigned)(p.B * p.nblk);
  quant_qk_kernel<<<dim3(nb, p.Hq + p.Hkv), kRows, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  quant_v_kernel<<<dim3(nb, p.Hkv), kRows, 0, stream>>>(p);
  return (int)cudaGetLastError();
}

}  // namespace fa
