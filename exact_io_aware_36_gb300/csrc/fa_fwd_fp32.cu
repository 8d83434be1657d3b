// fa_fwd_fp32.cu -- fp32 forward for exact attention on CUDA cores.
//
// Tensor-core TF32 cannot hold a 1e-5 absolute error on O, so the fp32
// forward multiplies in fp32 FMAs.  It is the same tiled method as the bf16
// kernel ("FlashAttention: Faster Attention Without Dropping a Single
// Interaction", Key design 2: the running max m and sum l merged per key
// tile), at a scale where latency, not throughput, matters.
//
// One warp owns one query row.  Keys are visited in tiles of 32 staged in
// shared memory: lane j computes the full dot product of the row with key j,
// the warp merges the tile's max and exponential sum into (m, l), and every
// lane accumulates its share of the d output columns (columns lane,
// lane + 32, ...).  Scores live in the base-2 domain:
// x = s * scale * log2(e) + bias * log2(e).
#include <cuda_runtime.h>
#include <math.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxD = 128;
constexpr int kCols = kMaxD / 32;
constexpr int kTile = 32;                           // keys per tile
constexpr int kKStride = kMaxD + 1;                 // lane j reads K row j: no bank conflicts
constexpr int kPer = kTile * kMaxD / kThreads;      // tile elements per thread and tensor
static_assert(kPer == (kTile / kWarps) * kCols, "loader layout");

// One block owns kWarps consecutive query rows of one (sequence, head), one
// warp per row.  The block walks the union of its rows' key ranges in tiles
// of 32 keys: each tile of K and V is loaded by all threads with coalesced
// loads (the next tile's loads are issued into registers before the current
// tile is computed), so a tile costs one memory round trip rather than one
// per element.
__global__ void __launch_bounds__(kThreads)
fwd_fp32_kernel(AttnParams p) {
  __shared__ float q_s[kWarps][kMaxD];
  __shared__ float k_s[kTile][kKStride];
  __shared__ float v_s[kTile][kMaxD];
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
  const int row0 = blockIdx.x * kWarps;
  if (row0 >= L) return;                              // uniform over the block
  const int row = row0 + warp;
  const bool active = row < L;                        // warps past the end only help load

  const float* Q = static_cast<const float*>(p.q);
  const float* K = static_cast<const float*>(p.k);
  const float* V = static_cast<const float*>(p.v);
  const long long tq = seq0 + row;
  for (int c = lane; c < d; c += 32) q_s[warp][c] = active ? Q[(tq * p.Hq + h) * d + c] : 0.f;

  const float c2 = p.scale_log2;
  const float slope2 = p.alibi ? p.alibi[h] * kLog2e : 0.f;
  // This row sees keys [key_lo, n_keys); the block walks [blk_lo, blk_hi).
  const int n_keys = p.causal ? row + 1 : L;
  const int key_lo = p.causal ? max(0, row - p.window) : 0;   // sliding-window band start
  const int blk_lo = p.causal ? max(0, row0 - p.window) : 0;
  const int blk_hi = p.causal ? min(row0 + kWarps, L) : L;

  // Warp w loads tile rows w, w + 4, ...; lane l columns l, l + 32, ...
  // (one contiguous key row per warp instruction, no index division).
  constexpr int kRowsPerWarp = kTile / kWarps;
  float kr[kPer], vr[kPer];
  auto load_tile = [&](int k0) {
    const int nk = min(kTile, blk_hi - k0);
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int jj = warp + kWarps * r;
      const long long off = ((seq0 + k0 + jj) * p.Hkv + g) * d;
#pragma unroll
      for (int i = 0; i < kCols; ++i) {
        const int c = lane + 32 * i;
        kr[r * kCols + i] = 0.f;
        vr[r * kCols + i] = 0.f;
        if (jj < nk && c < d) {
          kr[r * kCols + i] = __ldg(K + off + c);
          vr[r * kCols + i] = __ldg(V + off + c);
        }
      }
    }
  };
  auto store_tile = [&]() {
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int jj = warp + kWarps * r;
#pragma unroll
      for (int i = 0; i < kCols; ++i) {
        const int c = lane + 32 * i;
        if (c < d) {
          k_s[jj][c] = kr[r * kCols + i];
          v_s[jj][c] = vr[r * kCols + i];
        }
      }
    }
  };

  float m = -INFINITY;
  float l = 0.f;
  float acc[kCols];
#pragma unroll
  for (int i = 0; i < kCols; ++i) acc[i] = 0.f;

  if (blk_lo < blk_hi) load_tile(blk_lo);
  for (int k0 = blk_lo; k0 < blk_hi; k0 += kTile) {
    __syncthreads();                                  // the previous tile is consumed
    store_tile();
    __syncthreads();
    if (k0 + kTile < blk_hi) load_tile(k0 + kTile);   // in flight while this tile is computed
    const int j = k0 + lane;
    const bool valid = active && j >= key_lo && j < n_keys;
    float x = -INFINITY;
    if (valid) {
      // four partial sums break the dependent FMA chain
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
      int c = 0;
      for (; c + 4 <= d; c += 4) {
        s0 = fmaf(q_s[warp][c], k_s[lane][c], s0);
        s1 = fmaf(q_s[warp][c + 1], k_s[lane][c + 1], s1);
        s2 = fmaf(q_s[warp][c + 2], k_s[lane][c + 2], s2);
        s3 = fmaf(q_s[warp][c + 3], k_s[lane][c + 3], s3);
      }
      for (; c < d; ++c) s0 = fmaf(q_s[warp][c], k_s[lane][c], s0);
      x = ((s0 + s1) + (s2 + s3)) * c2;
      if (p.alibi) x += slope2 * (float)(j - row);
    }
    float tile_max = x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tile_max = fmaxf(tile_max, __shfl_xor_sync(0xffffffffu, tile_max, o));
    const float m_new = fmaxf(m, tile_max);
    const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - m_new);
    const float pj = valid ? exp2f(x - m_new) : 0.f;
    float psum = pj;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
    l = l * alpha + psum;
    m = m_new;
#pragma unroll
    for (int i = 0; i < kCols; ++i) acc[i] *= alpha;
    const int n_in = min(kTile, blk_hi - k0);
#pragma unroll 8
    for (int jj = 0; jj < n_in; ++jj) {
      const float pb = __shfl_sync(0xffffffffu, pj, jj);
#pragma unroll
      for (int i = 0; i < kCols; ++i) {
        const int c = lane + 32 * i;
        if (c < d) acc[i] = fmaf(pb, v_s[jj][c], acc[i]);
      }
    }
  }
  if (!active) return;

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
  fwd_fp32_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return (int)cudaGetLastError();
}

}  // namespace fa
