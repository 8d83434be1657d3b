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
// One persistent kernel, one pass over each input: a CTA takes items
// (128-row block, head) of Q, K and V in turn, each staged in shared memory
// by TMA while the items before it are processed.  Q and K: one thread per
// row, the butterfly in registers.  V: one thread per head-dim column, so
// that its transposed codes (keys contiguous) are written as one run.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "fa_host_util.h"
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
// 128 bytes per row.
// Persistent: a CTA takes items (block of 128 rows, head; Q heads, then K
// heads, all heads of one row block before the next) and keeps kQkStages
// of them in flight in shared memory: each is loaded by TMA as two boxes of
// 128 rows x 64 columns (128-byte swizzle, so that the threads reading one
// row each hit distinct banks), and the next items' loads run while this
// one is transformed.
constexpr int kQkStages = 3;
constexpr int kBox = kRows * 64 * 2;              // one box: 128 rows x 64 columns, bf16
constexpr int kQkSmem = kQkStages * 2 * kBox + 1024;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// V, one item: codes transposed into [Hkv, 128, B * nblk * 128] (keys
// contiguous per head-dim column), the block's scale, and the largest scale
// per kv head (v_smax, zeroed before; as an unsigned maximum of the
// non-negative floats' bits).  Thread c takes column c of the staged tile
// (128 keys, read down the rows of the swizzled boxes) and writes its 128
// codes as one contiguous run; rows past the sequence end give code 0.
__device__ __forceinline__ void quant_v_column(const QuantParams& p, const uint8_t* tile, int bi, int g,
                                               int rows, float* red) {
  const int c = threadIdx.x;
  // element (r, c): box c / 64, row r, 16-byte chunk ((c % 64) / 8) ^ (r % 8), lane c % 8
  const uint8_t* colp = tile + (c / 64) * kBox + (c % 8) * 2;
  const int ch = (c % 64) / 8;
  uint32_t pk[kRows / 2];                          // rows 2i (low half) and 2i + 1 (high half), bf16
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < kRows / 2; ++i) {
    const int r = 2 * i;
    const uint32_t lo = r < rows ? *reinterpret_cast<const uint16_t*>(colp + r * 128 + ((ch ^ (r & 7)) << 4)) : 0u;
    const uint32_t hi = r + 1 < rows
        ? *reinterpret_cast<const uint16_t*>(colp + (r + 1) * 128 + ((ch ^ ((r + 1) & 7)) << 4)) : 0u;
    pk[i] = lo | (hi << 16);
    m = fmax3(m, fabsf(__uint_as_float(lo << 16)), fabsf(__uint_as_float(hi << 16)));
  }
  const float amax = block_amax(m, red);           // also: every thread has read the tile
  float scale, inv;
  block_scales(amax, &scale, &inv);
  if (threadIdx.x == 0) {
    p.v_scale[(long long)g * p.B * p.nblk + bi] = scale;
    if (rows > 0) atomicMax(reinterpret_cast<unsigned int*>(p.v_smax + g), __float_as_uint(scale));
  }
  uint4* dst = reinterpret_cast<uint4*>(p.v8t + ((long long)g * kD + c) * p.vt_stride + (long long)bi * kRows);
#pragma unroll
  for (int j = 0; j < kRows / 16; ++j) {           // 16 keys per store
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t a = pk[8 * j + 2 * e], b = pk[8 * j + 2 * e + 1];
      w[e] = e4m3x2(__uint_as_float(a << 16) * inv, __uint_as_float(a & 0xFFFF0000u) * inv) |
             (e4m3x2(__uint_as_float(b << 16) * inv, __uint_as_float(b & 0xFFFF0000u) * inv) << 16);
    }
    dst[j] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__global__ void __launch_bounds__(kRows, 2)
quant_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
             const __grid_constant__ CUtensorMap tmv, const QuantParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ uint64_t full[kQkStages];
  __shared__ float red2[2][4];                     // by item parity: no barrier before its reuse
  __shared__ __align__(16) float sg[kD];
  __shared__ int abort_flag;
  const int tid = threadIdx.x;
  const int nb = p.B * p.nblk;
  const int HH = p.Hq + 2 * p.Hkv;
  const long long nitems = (long long)nb * HH;
  if (tid == 0) {
    for (int s = 0; s < kQkStages; ++s) mbar_init(&full[s], 1);
    abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmq);
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  sg[tid] = __ldg(p.signs + tid);
  __syncthreads();
  const WaitCtx wc{&abort_flag, p.status};

  // Item u: row block bi = u / HH of head y = u % HH (y < Hq: Q, then K,
  // then V).  Returns
  // false for a malformed cu_seqlens (recorded); rows <= 0 past a short
  // sequence's end.
  auto item = [&](long long u, int* bi, int* y, long long* seq0, int* rows) -> bool {
    *bi = (int)(u / HH);
    *y = (int)(u % HH);
    int L;
    if (!block_bounds(p, *bi / p.nblk, seq0, &L)) return false;
    *rows = min(kRows, L - kRows * (*bi % p.nblk));
    return true;
  };
  // Thread 0: load item u into stage s (an item without rows only completes
  // the stage's phase).
  auto issue = [&](long long u, int s) {
    int bi, y, rows;
    long long seq0;
    const bool ok = item(u, &bi, &y, &seq0, &rows);
    if (!ok || rows <= 0) {
      mbar_arrive(&full[s]);
      return;
    }
    const CUtensorMap* m = y < p.Hq ? &tmq : y < p.Hq + p.Hkv ? &tmk : &tmv;
    const int h = y < p.Hq ? y : y < p.Hq + p.Hkv ? y - p.Hq : y - p.Hq - p.Hkv;
    const int z = (int)(seq0 + kRows * (bi % p.nblk));
    mbar_arrive_expect_tx(&full[s], 2 * kBox);
    tma_load_3d(smem + s * 2 * kBox, m, 0, h, z, &full[s]);
    tma_load_3d(smem + s * 2 * kBox + kBox, m, 64, h, z, &full[s]);
  };
  if (tid == 0)
    for (int s = 0; s < kQkStages; ++s)
      if (blockIdx.x + (long long)s * gridDim.x < nitems) issue(blockIdx.x + (long long)s * gridDim.x, s);

  int k = 0;
  for (long long u = blockIdx.x; u < nitems; u += gridDim.x, ++k) {
    const int s = k % kQkStages;
    // every thread leaves together if any warp's wait gave up
    if (__syncthreads_or(!wait_warp(&full[s], (k / kQkStages) & 1, wc))) break;
    // Past that barrier every thread is done with the previous item's stage:
    // it takes the item kQkStages after that one.
    if (tid == 0 && k > 0) {
      const long long un = u + (long long)(kQkStages - 1) * gridDim.x;
      if (un < nitems) issue(un, (k - 1) % kQkStages);
    }
    float* red = red2[k & 1];
    int bi, y, rows = 0;
    long long seq0 = 0;
    if (!item(u, &bi, &y, &seq0, &rows) && tid == 0) record_status(p.status, FA_ERR_CU_SEQLENS);
    if (rows <= 0 && y < p.Hq + p.Hkv) {           // Q / K block past its sequence's end: scale 1, no codes
      if (tid == 0) *((y < p.Hq ? p.q_scale : p.k_scale) + (long long)(y < p.Hq ? y : y - p.Hq) * nb + bi) = 1.f;
      continue;
    }
    if (y >= p.Hq + p.Hkv) {                       // V: this thread's column of the tile
      quant_v_column(p, smem + s * 2 * kBox, bi, y - p.Hq - p.Hkv, rows, red);
      continue;
    }
    const bool isq = y < p.Hq;
    const int h = isq ? y : y - p.Hq;
    const int H = isq ? p.Hq : p.Hkv;
    const int r0 = kRows * (bi % p.nblk);
    const int r = tid;
    const bool valid = r < rows;
    // The row as 64 packed pairs (columns 2i, 2i + 1): every add, subtract
    // and multiply below is the same IEEE float32 operation on each half.
    uint64_t v[kD / 2];
    if (valid) {
      // chunk c of this row: box c / 8, 16-byte column chunk (c % 8) ^ (r % 8)
      const uint8_t* rowp = smem + s * 2 * kBox + r * 128;
#pragma unroll
      for (int c = 0; c < kD / 8; ++c) {
        const uint4 raw = *reinterpret_cast<const uint4*>(rowp + (c / 8) * kBox + (((c % 8) ^ (r & 7)) << 4));
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) v[4 * c + e] = f2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
      }
    } else {
#pragma unroll
      for (int c = 0; c < kD / 2; ++c) v[c] = 0;
    }
    const uint64_t* sg2 = reinterpret_cast<const uint64_t*>(sg);
#pragma unroll
    for (int c = 0; c < kD / 2; ++c) v[c] = fmul2(v[c], sg2[c]);
    // stride 1: within each pair
#pragma unroll
    for (int c = 0; c < kD / 2; ++c) {
      float a, bb;
      f2split(v[c], a, bb);
      v[c] = f2(a + bb, a - bb);
    }
#pragma unroll
    for (int st = 0; st < 6; ++st) {               // strides 2, 4, ..., 64: hp pairs apart
      const int hp = 1 << st;
#pragma unroll
      for (int kk = 0; kk < kD / 4; ++kk) {        // pair kk: (c, c + hp)
        const int c = (kk / hp) * 2 * hp + kk % hp;
        const uint64_t a = v[c], bb = v[c + hp];
        v[c] = fadd2(a, bb);
        v[c + hp] = fsub2(a, bb);
      }
    }
    float m = 0.f;
#pragma unroll
    for (int c = 0; c < kD / 2; ++c) {
      float a, bb;
      f2split(v[c], a, bb);
      m = fmax3(m, fabsf(a), fabsf(bb));
    }
    const float amax = block_amax(m, red);
    float scale, inv;
    block_scales(amax, &scale, &inv);
    if (tid == 0) *((isq ? p.q_scale : p.k_scale) + (long long)h * nb + bi) = scale;
    if (valid) {
      uint8_t* codes = (isq ? p.q8 : p.k8) + ((seq0 + r0 + r) * H + h) * kD;
      const uint64_t inv2 = f2(inv, inv);
#pragma unroll
      for (int c = 0; c < kD / 2; c += 8) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x0, x1, x2, x3;
          f2split(fmul2(v[c + 2 * e], inv2), x0, x1);
          f2split(fmul2(v[c + 2 * e + 1], inv2), x2, x3);
          w[e] = e4m3x2(x0, x1) | (e4m3x2(x2, x3) << 16);
        }
        reinterpret_cast<uint4*>(codes)[c / 8] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  // After an abort, loads still in flight must land before shared memory
  // goes away: every item issued but not consumed (items k .. k + S - 2;
  // item k + S - 1 was to be issued by the item that gave up).
  for (int j = 0; j + 1 < kQkStages; ++j) {
    const long long u = blockIdx.x + (long long)(k + j) * gridDim.x;
    if (u < nitems) wait_warp_drain(&full[(k + j) % kQkStages], ((k + j) / kQkStages) & 1);
  }
}

}  // namespace

int launch_fp8_quantize(const QuantParams& p, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cudaError_t e = cudaMemsetAsync(p.v_smax, 0, sizeof(float) * p.Hkv, stream);
  if (e != cudaSuccess) return (int)e;
  const unsigned nb = (unsigned)(p.B * p.nblk);
  CUtensorMap tq, tk, tv;
  int r = make_tmap_bf16_3d(&tq, p.q, kD, p.Hq, p.T, kRows);
  if (!r) r = make_tmap_bf16_3d(&tk, p.k, kD, p.Hkv, p.T, kRows);
  if (!r) r = make_tmap_bf16_3d(&tv, p.v, kD, p.Hkv, p.T, kRows);
  if (!r) r = set_max_dynamic_smem(reinterpret_cast<const void*>(quant_kernel), kQkSmem);
  int nsm = 0;
  if (!r) r = sm_count(&nsm);
  if (r) return r;
  const long long nitems = (long long)nb * (p.Hq + 2 * p.Hkv);
  quant_kernel<<<(unsigned)std::min<long long>(nitems, 2LL * nsm), kRows, kQkSmem, stream>>>(tq, tk, tv, p);
  return (int)cudaGetLastError();
}

}  // namespace fa
