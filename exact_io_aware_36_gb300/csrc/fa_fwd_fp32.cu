// fa_fwd_fp32.cu -- fp32 forward for exact attention on CUDA cores.
//
// Tensor-core TF32 cannot hold a 1e-5 absolute error on O, so the fp32
// forward multiplies in fp32 FMAs.  It is the same tiled method as the bf16
// kernel ("FlashAttention: Faster Attention Without Dropping a Single
// Interaction", Key design 2: the running max m and sum l merged per key
// tile), at a scale where latency, not throughput, matters.
//
// One warp owns one query row.  Keys are visited in tiles of 32: lane j
// computes the full dot product of the row with key j, the warp merges the
// tile's max and exponential sum into (m, l), and every lane accumulates its
// share of the d output columns (columns lane, lane + 32, ...).  Scores live
// in the base-2 domain: x = s * scale * log2(e) + bias * log2(e).
#include <cuda_runtime.h>
#include <math.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxD = 128;
constexpr int kCols = kMaxD / 32;

__global__ void __launch_bounds__(kWarps * 32)
fwd_fp32_kernel(AttnParams p) {
  __shared__ float q_s[kWarps][kMaxD];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.z;
  const int h = blockIdx.y;
  const int g = h / p.group;
  const int d = p.d;

  long long seq0;
  int L;
  if (p.cu_seqlens) {
    const int c0 = p.cu_seqlens[b];
    const int c1 = p.cu_seqlens[b + 1];
    if ((b == 0 && c0 != 0) || c1 < c0 || (long long)c1 > p.T || c1 - c0 > p.N) {
      if (threadIdx.x == 0) record_status(p.status, FA_ERR_CU_SEQLENS);
      return;
    }
    seq0 = c0;
    L = c1 - c0;
  } else {
    seq0 = (long long)b * p.N;
    L = p.N;
  }
  const int row = blockIdx.x * kWarps + warp;
  if (row >= L) return;

  const float* Q = static_cast<const float*>(p.q);
  const float* K = static_cast<const float*>(p.k);
  const float* V = static_cast<const float*>(p.v);
  const long long tq = seq0 + row;
  for (int c = lane; c < d; c += 32) q_s[warp][c] = Q[(tq * p.Hq + h) * d + c];
  __syncwarp();

  const float c2 = p.scale_log2;
  const float slope2 = p.alibi ? p.alibi[h] * kLog2e : 0.f;
  const int n_keys = p.causal ? row + 1 : L;
  const int key_lo = p.causal ? max(0, row - p.window) : 0;   // sliding-window band start

  float m = -INFINITY;
  float l = 0.f;
  float acc[kCols];
#pragma unroll
  for (int i = 0; i < kCols; ++i) acc[i] = 0.f;

  for (int k0 = key_lo; k0 < n_keys; k0 += 32) {
    const int j = k0 + lane;
    float x = -INFINITY;
    if (j < n_keys) {
      const float* kr = K + ((seq0 + j) * p.Hkv + g) * d;
      float s = 0.f;
      for (int c = 0; c < d; ++c) s = fmaf(q_s[warp][c], kr[c], s);
      x = s * c2;
      if (p.alibi) x += slope2 * (float)(j - row);
    }
    float tile_max = x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tile_max = fmaxf(tile_max, __shfl_xor_sync(0xffffffffu, tile_max, o));
    const float m_new = fmaxf(m, tile_max);
    const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - m_new);
    const float pj = (j < n_keys) ? exp2f(x - m_new) : 0.f;
    float psum = pj;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
    l = l * alpha + psum;
    m = m_new;
#pragma unroll
    for (int i = 0; i < kCols; ++i) acc[i] *= alpha;
    const int n_in = min(32, n_keys - k0);
    for (int jj = 0; jj < n_in; ++jj) {
      const float pb = __shfl_sync(0xffffffffu, pj, jj);
      const float* vr = V + ((seq0 + k0 + jj) * p.Hkv + g) * d;
#pragma unroll
      for (int i = 0; i < kCols; ++i) {
        const int c = lane + 32 * i;
        if (c < d) acc[i] = fmaf(pb, vr[c], acc[i]);
      }
    }
  }

  float* O = static_cast<float*>(p.o);
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int i = 0; i < kCols; ++i) {
    const int c = lane + 32 * i;
    if (c < d) O[(tq * p.Hq + h) * d + c] = acc[i] * inv_l;
  }
  if (lane == 0) p.lse[(long long)h * p.T + tq] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

}  // namespace

int launch_fwd_fp32(const AttnParams& p, void* stream) {
  dim3 grid((p.N + kWarps - 1) / kWarps, p.Hq, p.B);
  fwd_fp32_kernel<<<grid, kWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return (int)cudaGetLastError();
}

}  // namespace fa
