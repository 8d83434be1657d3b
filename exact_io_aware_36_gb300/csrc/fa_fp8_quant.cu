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
// division amax / 448, the division x / scale (IEEE, round to nearest), and
// the conversion to e4m3 (round to nearest even, saturated).
//
// One block of 128 threads per (head, sequence block); a row of d = 128 is one
// warp, 4 columns per lane: butterfly strides 1 and 2 inside a lane, 4 .. 64
// across lanes by shuffles.  Two passes over the rows (the maximum, then the
// codes) recompute the transform instead of holding the block.
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

// Row `row` (token) of head h: this lane's 4 columns, optionally sign-flipped
// and transformed by the butterfly.
template <bool TRANSFORM>
__device__ __forceinline__ void load_row(const __nv_bfloat16* x, int H, long long tok, int h,
                                         const float (&sg)[4], float (&v)[4]) {
  const int lane = threadIdx.x & 31;
  const uint2 raw = *reinterpret_cast<const uint2*>(x + (tok * H + h) * kD + 4 * lane);
  v[0] = __uint_as_float(raw.x << 16);
  v[1] = __uint_as_float(raw.x & 0xFFFF0000u);
  v[2] = __uint_as_float(raw.y << 16);
  v[3] = __uint_as_float(raw.y & 0xFFFF0000u);
  if constexpr (TRANSFORM) {
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] *= sg[e];
    // stride 1: (0,1), (2,3);  stride 2: (0,2), (1,3)
    float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2;
    v[1] = a1 + a3;
    v[2] = a0 - a2;
    v[3] = a1 - a3;
    // strides 4 .. 64: column c = 4 lane + e pairs with c ^ stride, in lane ^ (stride / 4)
#pragma unroll
    for (int sl = 1; sl < 32; sl <<= 1) {
      const bool upper = (lane & sl) != 0;          // this lane holds the (a, b) pair's b
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float o = __shfl_xor_sync(0xffffffffu, v[e], sl);
        v[e] = upper ? o - v[e] : v[e] + o;
      }
    }
  }
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

// Q or K: codes [T, H, 128] and scales [H, B * nblk].  grid (B * nblk, H).
template <bool TRANSFORM>
__global__ void __launch_bounds__(kRows) quant_rows_kernel(const QuantParams p, const __nv_bfloat16* x,
                                                           int H, uint8_t* codes, float* scales) {
  __shared__ float red[4];
  const int h = blockIdx.y;
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
  float* sc_out = scales + (long long)h * p.B * p.nblk + bi;
  const int r0 = kRows * i;
  if (r0 >= L) {
    if (threadIdx.x == 0) *sc_out = 1.f;
    return;
  }
  const int rows = min(kRows, L - r0);
  float sg[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) sg[e] = TRANSFORM ? __ldg(p.signs + 4 * lane + e) : 1.f;
  float m = 0.f;
  for (int r = warp; r < rows; r += 4) {
    float v[4];
    load_row<TRANSFORM>(x, H, seq0 + r0 + r, h, sg, v);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
  }
  const float amax = block_amax(m, red);
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  if (threadIdx.x == 0) *sc_out = scale;
  for (int r = warp; r < rows; r += 4) {
    float v[4];
    const long long tok = seq0 + r0 + r;
    load_row<TRANSFORM>(x, H, tok, h, sg, v);
    const uint32_t c01 = e4m3x2(__fdiv_rn(v[0], scale), __fdiv_rn(v[1], scale));
    const uint32_t c23 = e4m3x2(__fdiv_rn(v[2], scale), __fdiv_rn(v[3], scale));
    *reinterpret_cast<uint32_t*>(codes + (tok * H + h) * kD + 4 * lane) = c01 | (c23 << 16);
  }
}

// V: codes transposed into [Hkv, 128, B * nblk * 128], scales, and the largest
// scale per kv head (v_smax, zeroed before).  grid (B * nblk, Hkv).
__global__ void __launch_bounds__(kRows) quant_v_kernel(const QuantParams p) {
  constexpr int kPitch = kRows + 4;               // bytes per column row in the transpose
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
  const float sg[4] = {1.f, 1.f, 1.f, 1.f};
  for (int w = threadIdx.x; w < kD * kPitch / 4; w += kRows) reinterpret_cast<uint32_t*>(tile)[w] = 0u;
  float m = 0.f;
  for (int r = warp; r < rows; r += 4) {
    float v[4];
    load_row<false>(x, p.Hkv, seq0 + r0 + r, g, sg, v);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
  }
  const float amax = block_amax(m, red);          // also orders the zero fill before the codes
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  if (threadIdx.x == 0) {
    p.v_scale[(long long)g * p.B * p.nblk + bi] = scale;
    if (rows > 0) atomicMax(reinterpret_cast<unsigned int*>(p.v_smax + g), __float_as_uint(scale));
  }
  for (int r = warp; r < rows; r += 4) {
    float v[4];
    load_row<false>(x, p.Hkv, seq0 + r0 + r, g, sg, v);
    const uint32_t c01 = e4m3x2(__fdiv_rn(v[0], scale), __fdiv_rn(v[1], scale));
    const uint32_t c23 = e4m3x2(__fdiv_rn(v[2], scale), __fdiv_rn(v[3], scale));
    const uint32_t c = c01 | (c23 << 16);
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
  quant_rows_kernel<true><<<dim3(nb, p.Hq), kRows, 0, stream>>>(
      p, static_cast<const __nv_bfloat16*>(p.q), p.Hq, p.q8, p.q_scale);
  quant_rows_kernel<true><<<dim3(nb, p.Hkv), kRows, 0, stream>>>(
      p, static_cast<const __nv_bfloat16*>(p.k), p.Hkv, p.k8, p.k_scale);
  quant_v_kernel<<<dim3(nb, p.Hkv), kRows, 0, stream>>>(p);
  return (int)cudaGetLastError();
}

}  // namespace fa
