// fa_decode_bf16.cu -- split-KV decode over a KV cache for sm_103a.
//
// Method: the q_len newest tokens of each sequence attend causally to the
// sequence's cached keys ("FlashAttention: Faster Attention Without Dropping
// a Single Interaction", Long context and inference: small-query decode over
// a growing cache).  The keys of one (sequence, kv head) are cut into chunks;
// each block reduces one chunk to a partial state (m, l, O) per query row,
// and a combine kernel merges the chunks with Key design 2's rule:
//     m = max_s m_s,  l = sum_s 2^(m_s - m) l_s,  O = sum_s 2^(m_s - m) O_s / l
// (log2 units; O_s unnormalised), LSE = (m + log2 l) ln 2.
//
// The work reads every cached key and value once and does R = group * q_len
// (<= 16) rows of arithmetic per key: it is bound by HBM, not by math, so it
// runs on the CUDA cores in fp32 (packed f32x2 FMAs) and spends its effort on
// the memory side: TMA streams 64-key tiles of K and V (128-byte swizzle)
// through a 3-stage mbarrier ring, two blocks share an SM, and the chunk size
// gives each SM several blocks.
//
// Block (288 threads): warp 8 issues the TMA loads; each of warps 0-7 owns
// 8 keys of every tile and runs its own online softmax over them, with no
// block-wide barrier in the loop:
//   S        lane (key kq, column quarter cq) dots its key with the R
//            pre-scaled query rows over its quarter; a 4-lane butterfly
//            completes the sums; bias and mask applied.
//   softmax  row max and sum over the warp's 8 keys by 3-step butterflies;
//            (m, l) per row in registers; P of the 8 keys to a small
//            per-warp buffer in shared memory.
//   PV       lane owns d / 32 columns of O for all rows: O = alpha O + P V.
// At the end of the chunk the 8 warps' states are merged (the same merge
// rule) through the then idle K/V ring into the block's partial state.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_host_util.h"
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kComputeThreads = 256;
constexpr int kThreads = kComputeThreads + 32;
constexpr int kLoadWarp = 8;
constexpr int kTileKeys = 64;
constexpr int kStages = 3;
constexpr uint32_t kBarCompute = 1;   // named barrier of warps 0-7

template <int D, int RM>
struct DecCfg {
  static constexpr int NB = D / 64;
  static constexpr int BOX = kTileKeys * 64 * 2;    // 64 keys x 64 columns
  static constexpr int TILE = NB * BOX;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + kStages * TILE;
  static constexpr int Q_OFF = V_OFF + kStages * TILE;           // fp32 [RM][D]
  static constexpr int P_OFF = Q_OFF + RM * D * 4;               // fp32 [8 warps][RM][8]
  static constexpr int ROW_OFF = P_OFF + 8 * RM * 8 * 4;          // int pos[RM], float slope2[RM]
  static constexpr int BAR_OFF = (ROW_OFF + 2 * RM * 4 + 15) / 16 * 16;
  static constexpr int SMEM_BYTES = BAR_OFF + 64 + 1024;
};

struct DecBars {
  uint64_t full[kStages], empty[kStages];
  int abort_flag;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// RM: rows per block rounded up to a power of two (p.R <= RM are real).
// Two blocks share an SM, except at 16 rows, whose accumulators need the
// registers of one.
template <int D, int RM>
__global__ void __launch_bounds__(kThreads, RM >= 16 ? 1 : 2)
decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const DecodeParams p) {
  using C = DecCfg<D, RM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  DecBars* bars = reinterpret_cast<DecBars*>(smem + C::BAR_OFF);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // block = (sequence b, kv head g, chunk s), chunk fastest
  const int s = (int)(blockIdx.x % (unsigned)p.nsplit);
  const int bg = (int)(blockIdx.x / (unsigned)p.nsplit);
  const int g = bg % p.Hkv;
  const int b = bg / p.Hkv;
  const int L = p.seqlens ? __ldg(p.seqlens + b) : p.S_max;
  if (L < p.q_len || L > p.S_max) {
    if (threadIdx.x == 0) record_status(p.status, FA_ERR_CU_SEQLENS);
    return;
  }
  const int k0 = s * p.chunk;
  if (k0 >= L) return;                          // past this cache's end: no partial
  const int k1 = min(k0 + p.chunk, L);
  const int W = p.window;
  const int pos0 = L - p.q_len;                 // position of query row 0
  const int kmin = max(k0, pos0 - W);           // lowest key any row of the block sees
  const int R = p.R;
  float* po = p.part_o + (long long)blockIdx.x * R * D;
  float* pml = p.part_ml + (long long)blockIdx.x * R * 3;
  if (kmin >= k1) {                             // chunk below every row's window: empty state
    for (int i = threadIdx.x; i < R * D; i += blockDim.x) po[i] = 0.f;
    if (threadIdx.x < R) {
      pml[3 * threadIdx.x] = -INFINITY;
      pml[3 * threadIdx.x + 1] = 0.f;
      pml[3 * threadIdx.x + 2] = 0.f;
    }
    return;
  }
  const int n = (k1 - kmin + kTileKeys - 1) / kTileKeys;

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&bars->full[st], 1);
      mbar_init(&bars->empty[st], kComputeThreads / 32);
    }
    bars->abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  const WaitCtx wc{&bars->abort_flag, p.status};

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    int issued = 0;
    for (int j = 0; j < n; ++j) {
      const int st = j % kStages;
      if (!wait_warp(&bars->empty[st], ((j / kStages) & 1) ^ 1, wc)) break;
      if (lane == 0) {
        const int row = b * p.S_max + kmin + kTileKeys * j;
        mbar_arrive_expect_tx(&bars->full[st], 2 * C::TILE);
#pragma unroll
        for (int bx = 0; bx < C::NB; ++bx) {
          tma_load_3d(smem + C::K_OFF + st * C::TILE + bx * C::BOX, &tmK, bx * 64, g, row, &bars->full[st]);
          tma_load_3d(smem + C::V_OFF + st * C::TILE + bx * C::BOX, &tmV, bx * 64, g, row, &bars->full[st]);
        }
      }
      __syncwarp();
      issued = j + 1;
    }
    // Loads in flight must land before this block's shared memory goes away.
    for (int j = max(0, issued - kStages); j < issued; ++j)
      wait_warp_drain(&bars->full[j % kStages], (j / kStages) & 1);
    return;
  }

  // --------------------------------------------------------------- compute
  const int t = threadIdx.x;
  float* qs = reinterpret_cast<float*>(smem + C::Q_OFF);
  int* rpos = reinterpret_cast<int*>(smem + C::ROW_OFF);
  float* rslope = reinterpret_cast<float*>(smem + C::ROW_OFF + RM * 4);
  // Query rows r = qi * group + hg (query token qi of this sequence, head
  // g * group + hg), pre-scaled by scale * log2(e); rows R..RM-1 are zero.
  for (int e = t; e < RM * (D / 8); e += kComputeThreads) {
    const int r = e / (D / 8);
    const int c8 = e % (D / 8);
    float f[8];
    if (r < R) {
      const int qi = r / p.group;
      const int h = g * p.group + r % p.group;
      const uint4 raw = *reinterpret_cast<const uint4*>(
          static_cast<const __nv_bfloat16*>(p.q) + (((long long)b * p.q_len + qi) * p.Hq + h) * D + c8 * 8);
      const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w4[i] << 16) * p.scale_log2;
        f[2 * i + 1] = __uint_as_float(w4[i] & 0xFFFF0000u) * p.scale_log2;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = 0.f;
    }
    float4* dst = reinterpret_cast<float4*>(qs + r * D + c8 * 8);
    dst[0] = make_float4(f[0], f[1], f[2], f[3]);
    dst[1] = make_float4(f[4], f[5], f[6], f[7]);
  }
  if (t < RM) {
    const int r = t < R ? t : 0;
    rpos[t] = pos0 + r / p.group;
    rslope[t] = p.alibi ? __ldg(p.alibi + g * p.group + r % p.group) * kLog2e : 0.f;
  }
  named_bar_sync(kBarCompute, kComputeThreads);

  // Warp w owns keys 8w .. 8w+7 of every tile and keeps its own (m, l, O)
  // for all rows; lane = (key kq, column quarter cq) for S, and lane owns
  // columns CPL * lane .. for O.
  constexpr int CPL = D / 32;
  const int kq = lane >> 2;
  const int cq = lane & 3;
  const int krow = 8 * warp + kq;
  float* pw = reinterpret_cast<float*>(smem + C::P_OFF) + warp * RM * 8;   // P of the warp, [RM][8]
  float m_r[RM], l_r[RM];
  uint64_t o2[RM][CPL / 2];
#pragma unroll
  for (int r = 0; r < RM; ++r) {
    m_r[r] = -INFINITY;
    l_r[r] = 0.f;
#pragma unroll
    for (int c = 0; c < CPL / 2; ++c) o2[r][c] = f2(0.f, 0.f);
  }
  const int col = CPL * lane;                  // first column of this lane's O
  const int vbox = col >> 6;
  const int vbyte = (col & 63) * 2;

  bool ok = true;
  for (int j = 0; j < n; ++j) {
    const int st = j % kStages;
    if (!(ok = wait_warp(&bars->full[st], (j / kStages) & 1, wc))) break;
    // ------------------------------------------- S = (q c2) . k (+ bias)
    const uint8_t* kt = smem + C::K_OFF + st * C::TILE;
    uint64_t acc[RM];
#pragma unroll
    for (int r = 0; r < RM; ++r) acc[r] = f2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
      const int c0 = 8 * cq + 32 * i;
      const int box = c0 >> 6;
      const int chunk = (c0 & 63) >> 3;
      const uint4 kv = *reinterpret_cast<const uint4*>(kt + box * C::BOX + krow * 128 + ((chunk ^ (krow & 7)) << 4));
      const uint64_t k01 = f2(__uint_as_float(kv.x << 16), __uint_as_float(kv.x & 0xFFFF0000u));
      const uint64_t k23 = f2(__uint_as_float(kv.y << 16), __uint_as_float(kv.y & 0xFFFF0000u));
      const uint64_t k45 = f2(__uint_as_float(kv.z << 16), __uint_as_float(kv.z & 0xFFFF0000u));
      const uint64_t k67 = f2(__uint_as_float(kv.w << 16), __uint_as_float(kv.w & 0xFFFF0000u));
#pragma unroll
      for (int r = 0; r < RM; ++r) {
        const float4 qa = *reinterpret_cast<const float4*>(qs + r * D + c0);
        const float4 qb = *reinterpret_cast<const float4*>(qs + r * D + c0 + 4);
        acc[r] = ffma2(f2(qa.x, qa.y), k01, acc[r]);
        acc[r] = ffma2(f2(qa.z, qa.w), k23, acc[r]);
        acc[r] = ffma2(f2(qb.x, qb.y), k45, acc[r]);
        acc[r] = ffma2(f2(qb.z, qb.w), k67, acc[r]);
      }
    }
    const int key = kmin + kTileKeys * j + krow;
    // ------------------- online softmax over the warp's 8 keys, per row
#pragma unroll
    for (int r = 0; r < RM; ++r) {
      float a0, a1;
      f2split(acc[r], a0, a1);
      float x = a0 + a1;
      x += __shfl_xor_sync(0xffffffffu, x, 1);
      x += __shfl_xor_sync(0xffffffffu, x, 2);
      const int pos = rpos[r];
      x = fmaf(rslope[r], (float)(key - pos), x);
      if (r >= R || key >= k1 || key > pos || key < pos - W) x = -INFINITY;
      float mx = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float mn = fmaxf(m_r[r], mx);
      float alpha = 1.f, pr = 0.f;
      if (mn != -INFINITY) {            // else nothing visible to this row yet
        alpha = ex2_approx(m_r[r] - mn);
        pr = ex2_approx(x - mn);
      }
      float ps = pr + __shfl_xor_sync(0xffffffffu, pr, 4);
      ps += __shfl_xor_sync(0xffffffffu, ps, 8);
      ps += __shfl_xor_sync(0xffffffffu, ps, 16);
      l_r[r] = fmaf(l_r[r], alpha, ps);
      m_r[r] = mn;
      if (cq == 0) pw[r * 8 + kq] = pr;
#pragma unroll
      for (int c = 0; c < CPL / 2; ++c) o2[r][c] = fmul2(o2[r][c], f2(alpha, alpha));
    }
    __syncwarp();
    // ------------------------------------------------------ O += P V
    const uint8_t* vt = smem + C::V_OFF + st * C::TILE;
#pragma unroll
    for (int k4 = 0; k4 < 8; k4 += 4) {
      float4 p4[RM];
#pragma unroll
      for (int r = 0; r < RM; ++r) p4[r] = *reinterpret_cast<const float4*>(pw + r * 8 + k4);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int vr = 8 * warp + k4 + u;
        const uint8_t* vrow = vt + vbox * C::BOX + vr * 128 + (((vbyte >> 4) ^ (vr & 7)) << 4) + (vbyte & 15);
        uint64_t v2[CPL / 2];
        if (CPL == 4) {
          const uint2 w = *reinterpret_cast<const uint2*>(vrow);
          v2[0] = f2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u));
          v2[CPL / 2 - 1] = f2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
        } else {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(vrow);
          v2[0] = f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
        }
#pragma unroll
        for (int r = 0; r < RM; ++r) {
          const float pu = u == 0 ? p4[r].x : u == 1 ? p4[r].y : u == 2 ? p4[r].z : p4[r].w;
#pragma unroll
          for (int c = 0; c < CPL / 2; ++c) o2[r][c] = ffma2(f2(pu, pu), v2[c], o2[r][c]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->empty[st]);
  }
  // ------------------------------------- merge the 8 warps' partial states
  // Every load issued was for a tile all warps consumed, so the K/V ring is
  // idle once all warps are here and holds the exchange.
  if (named_bar_any(kBarCompute, kComputeThreads, !ok)) return;
  float* ow = reinterpret_cast<float*>(smem + C::K_OFF);           // [8][RM][D]
  float* mlw = ow + 8 * RM * D;                                      // [8][RM][2]
#pragma unroll
  for (int r = 0; r < RM; ++r) {
    if (r < R) {
#pragma unroll
      for (int c = 0; c < CPL / 2; ++c) {
        float a0, a1;
        f2split(o2[r][c], a0, a1);
        *reinterpret_cast<float2*>(ow + (warp * RM + r) * D + col + 2 * c) = make_float2(a0, a1);
      }
      if (lane == 0) {
        mlw[(warp * RM + r) * 2] = m_r[r];
        mlw[(warp * RM + r) * 2 + 1] = l_r[r];
      }
    }
  }
  named_bar_sync(kBarCompute, kComputeThreads);
  for (int e = t; e < R * D; e += kComputeThreads) {
    const int r = e / D;
    const int c = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < 8; ++w2) M = fmaxf(M, mlw[(w2 * RM + r) * 2]);
    float o = 0.f, l = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < 8; ++w2) {
      const float mw = mlw[(w2 * RM + r) * 2];
      const float wt = mw == -INFINITY ? 0.f : ex2_approx(mw - M);
      o = fmaf(wt, ow[(w2 * RM + r) * D + c], o);
      l = fmaf(wt, mlw[(w2 * RM + r) * 2 + 1], l);
    }
    po[r * D + c] = o;
    if (c == 0) {
      pml[3 * r] = M;
      pml[3 * r + 1] = l;      // P in fp32: the product used exactly these weights
      pml[3 * r + 2] = l;
    }
  }
}

// ---------------------------------------------------------------------------
// d = 128: the two products on the tensor cores, in transposed form so that
// the keys, not the few query rows, fill the 128-row M of tcgen05:
//   S^T(j) = K_j Q^T    M 128 keys, N 16 (query rows, zero-padded), K d
//   O^T   += V_j^T P^T   M 128 head dims, N 16, K 128 keys (A = V_j as an
//                        MN-major operand, B = P from shared memory)
// Block (192 threads): warp 5 TMA, warp 4 MMA (one lane), warps 0-3 the
// softmax with one key of the tile per thread.  The reference max of every
// row is raised speculatively: a tile whose scores stay within tau of it
// (the common case) needs no max at all; otherwise the block takes the exact
// tile max (one vote and one exchange) and rescales its O^T rows in TMEM
// once the previous product is complete.  P goes to shared memory in bf16;
// the block's partial state is (m, l, l~) with l the exact sum of P and l~ the
// sum of the rounded P the product used.
// TMEM: S^T buffers at columns 0 and 16, O^T at 32 (16 columns each).
namespace tc {

constexpr int kThreads = 192;
constexpr int kMmaWarp = 4;
constexpr int kLoadWarp = 5;
constexpr int kStages = 3;
constexpr int kN = 16;                              // query rows per block, padded
constexpr float kTau = 8.0f;
constexpr int BOX = 128 * 64 * 2;                   // 128 keys x 64 head dims
constexpr int TILE = 2 * BOX;                       // 128 keys x 128 head dims
constexpr int QBOX = kN * 128;                      // 16 rows x 64 head dims (bf16)
constexpr int PBOX = kN * 128;                      // 16 rows x 64 keys (bf16)
constexpr int K_OFF = 0;
constexpr int V_OFF = K_OFF + kStages * TILE;
constexpr int Q_OFF = V_OFF + kStages * TILE;       // 2 boxes
constexpr int P_OFF = Q_OFF + 2 * QBOX;             // 2 buffers x 2 boxes
constexpr int RED_OFF = P_OFF + 4 * PBOX;           // float [8][16]: per-warp row maxima / sums
constexpr int ROW_OFF = RED_OFF + 8 * kN * 4;       // int pos[16], float slope2[16]
constexpr int BAR_OFF = ROW_OFF + 2 * kN * 4;
constexpr int SMEM_BYTES = BAR_OFF + 128 + 1024;
constexpr uint32_t S_COL = 0, O_COL = 32;

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], p_full[2];
  uint64_t pv_done[2];       // PV(j) completes pv_done[j & 1]: waited in order, no phase skipped
  uint64_t o_done;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 128, "barrier block");

__global__ void __launch_bounds__(kThreads, 1)
decode_split_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  Bars* bars = reinterpret_cast<Bars*>(smem + BAR_OFF);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int s = (int)(blockIdx.x % (unsigned)p.nsplit);
  const int bg = (int)(blockIdx.x / (unsigned)p.nsplit);
  const int g = bg % p.Hkv;
  const int b = bg / p.Hkv;
  const int L = p.seqlens ? __ldg(p.seqlens + b) : p.S_max;
  if (L < p.q_len || L > p.S_max) {
    if (threadIdx.x == 0) record_status(p.status, FA_ERR_CU_SEQLENS);
    return;
  }
  const int k0 = s * p.chunk;
  if (k0 >= L) return;                          // past this cache's end: no partial
  const int k1 = min(k0 + p.chunk, L);
  const int W = p.window;
  const int pos0 = L - p.q_len;
  const int kmin = max(k0, pos0 - W);
  const int R = p.R;
  float* po = p.part_o + (long long)blockIdx.x * R * D;
  float* pml = p.part_ml + (long long)blockIdx.x * R * 3;
  if (kmin >= k1) {                             // chunk below every row's window: empty state
    for (int i = threadIdx.x; i < R * D; i += blockDim.x) po[i] = 0.f;
    if (threadIdx.x < R) {
      pml[3 * threadIdx.x] = -INFINITY;
      pml[3 * threadIdx.x + 1] = 0.f;
      pml[3 * threadIdx.x + 2] = 0.f;
    }
    return;
  }
  const int n = (k1 - kmin + 127) / 128;

  int* rpos = reinterpret_cast<int*>(smem + ROW_OFF);
  float* rslope = reinterpret_cast<float*>(smem + ROW_OFF + kN * 4);
  float* red = reinterpret_cast<float*>(smem + RED_OFF);
  // Q rows R..15 are zero (the TMA box fills rows 0..R-1 only)
  for (int i = threadIdx.x; i < 2 * QBOX / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem + Q_OFF)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x < kN) {
    const int r = threadIdx.x < R ? threadIdx.x : 0;
    rpos[threadIdx.x] = pos0 + r / p.group;
    rslope[threadIdx.x] = p.alibi ? __ldg(p.alibi + g * p.group + r % p.group) * kLog2e : 0.f;
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 4);
    }
    mbar_init(&bars->pv_done[0], 1);
    mbar_init(&bars->pv_done[1], 1);
    mbar_init(&bars->o_done, 1);
    bars->abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtx wc{&bars->abort_flag, p.status};

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      // the block's R rows: q_len tokens x group heads, row r = qi * group + hg
      mbar_arrive_expect_tx(&bars->q_full, 2 * R * 128);
      for (int bx = 0; bx < 2; ++bx)
        tma_load_3d(smem + Q_OFF + bx * QBOX, &tmQ, bx * 64, g * p.group, b * p.q_len, &bars->q_full);
    }
    __syncwarp();
    int issued = 0;
    for (int j = 0; j < n; ++j) {
      const int st = j % kStages;
      if (!wait_warp(&bars->kv_empty[st], ((j / kStages) & 1) ^ 1, wc)) break;
      if (lane == 0) {
        const int row = b * p.S_max + kmin + 128 * j;
        mbar_arrive_expect_tx(&bars->kv_full[st], 2 * TILE);
        for (int bx = 0; bx < 2; ++bx) {
          tma_load_3d(smem + K_OFF + st * TILE + bx * BOX, &tmK, bx * 64, g, row, &bars->kv_full[st]);
          tma_load_3d(smem + V_OFF + st * TILE + bx * BOX, &tmV, bx * 64, g, row, &bars->kv_full[st]);
        }
      }
      __syncwarp();
      issued = j + 1;
    }
    wait_warp_drain(&bars->q_full, 0);
    for (int j = max(0, issued - kStages); j < issued; ++j)
      wait_warp_drain(&bars->kv_full[j % kStages], (j / kStages) & 1);
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t ID_S = idesc_bf16_f32(128, kN, 0, 0);   // K and Q K-major
    constexpr uint32_t ID_O = idesc_bf16_f32(128, kN, 1, 0);   // V^T MN-major, P K-major
    const uint32_t sQ = smem_u32(smem + Q_OFF);
    const uint32_t sK = smem_u32(smem + K_OFF);
    const uint32_t sV = smem_u32(smem + V_OFF);
    const uint32_t sP = smem_u32(smem + P_OFF);
    auto issue_s = [&](int j) {
      const uint32_t kb = sK + (j % kStages) * TILE;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t offk = (kk >> 2) * BOX + (kk & 3) * 32;
        const uint32_t offq = (kk >> 2) * QBOX + (kk & 3) * 32;
        mma_ss(tmem + S_COL + 16 * (j & 1), smem_desc_sw128(kb + offk, 16, 1024),
               smem_desc_sw128(sQ + offq, 16, 1024), ID_S, kk > 0 ? 1u : 0u);
      }
      mma_commit(&bars->s_full[j & 1]);
    };
    bool ok = wait_warp(&bars->q_full, 0, wc);
    for (int j = 0; ok && j < 2 && j < n; ++j) {
      if (!(ok = wait_warp(&bars->kv_full[j % kStages], (j / kStages) & 1, wc))) break;
      tc_fence_after();
      if (lane == 0) issue_s(j);
      __syncwarp();
    }
    for (int j = 0; ok && j < n; ++j) {
      const int st = j % kStages;
      if (!(ok = wait_warp(&bars->p_full[j & 1], (j >> 1) & 1, wc))) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t vb = sV + st * TILE;
        const uint32_t pb = sP + (j & 1) * 2 * PBOX;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)          // K = 128 keys, 16 per MMA
          mma_ss(tmem + O_COL, smem_desc_sw128(vb + kk * 2048, BOX, 1024),
                 smem_desc_sw128(pb + (kk >> 2) * PBOX + (kk & 3) * 32, 16, 1024), ID_O,
                 (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->pv_done[j & 1]);
        mma_commit(&bars->kv_empty[st]);
      }
      __syncwarp();
      // S^T(j+2) over S buffer j&1, which the softmax of tile j has released
      const int nx = j + 2;
      if (nx < n) {
        if (!(ok = wait_warp(&bars->kv_full[nx % kStages], (nx / kStages) & 1, wc))) break;
        tc_fence_after();
        if (lane == 0) issue_s(nx);
        __syncwarp();
      }
    }
    if (lane == 0) mma_commit(&bars->o_done);
    __syncwarp();
    wait_warp_drain(&bars->o_done, 0);
  } else {
    // ------------------------------------------------------------- softmax
    const int t = threadIdx.x;                  // key of the tile; head dim of O^T
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
    const float c2 = p.scale_log2;
    float m_ref[kN], l_t[kN], lr_t[kN];
#pragma unroll
    for (int r = 0; r < kN; ++r) {
      m_ref[r] = -INFINITY;
      l_t[r] = 0.f;
      lr_t[r] = 0.f;
    }
    int pv_waited = 0;                          // PV completions waited, in order
    bool ok = true;
    // Wait until PV(upto) has completed, taking every PV in order.  PV(k)
    // signals pv_done[k & 1]; PV(k + 2) needs P(k + 2), which is written only
    // after PV(k) was waited here, so a barrier never runs a phase ahead.
    auto ensure_pv = [&](int upto) {
      while (ok && pv_waited <= upto) {
        ok = wait_warp(&bars->pv_done[pv_waited & 1], (pv_waited >> 1) & 1, wc);
        ++pv_waited;
      }
    };
    for (int j = 0; j < n; ++j) {
      ok = wait_warp(&bars->s_full[j & 1], (j >> 1) & 1, wc);
      float x[kN];
      bool need = false;
      if (ok) {
        tc_fence_after();
        uint32_t sv[kN];
        tmem_ld16(lane_base + S_COL + 16 * (j & 1), sv);
        tmem_wait_ld();
        reg_fence16(sv);
        const int key = kmin + 128 * j + t;
#pragma unroll
        for (int r = 0; r < kN; ++r) {
          const int pos = rpos[r];
          float xr = fmaf(__uint_as_float(sv[r]), c2, rslope[r] * (float)(key - pos));
          if (r >= R || key >= k1 || key > pos || key < pos - W) xr = -INFINITY;
          x[r] = xr;
          need |= xr > m_ref[r] + kTau;         // also true on a row's first visible key
        }
      }
      // every softmax warp learns whether any gave up, and whether any row
      // must raise its reference
      if (named_bar_any(1, 128, !ok)) {
        ok = false;
        break;
      }
      if (named_bar_any(1, 128, need)) {
        // exact tile max per row: warp butterflies, then across the 4 warps
#pragma unroll
        for (int r = 0; r < kN; ++r) {
          float mr = x[r];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, o));
          if (lane == 0) red[warp * kN + r] = mr;
        }
        named_bar_sync(1, 128);
        float alpha[kN];
        bool any_raise = false;
#pragma unroll
        for (int r = 0; r < kN; ++r) {
          const float tm = fmaxf(fmaxf(red[r], red[kN + r]), fmaxf(red[2 * kN + r], red[3 * kN + r]));
          const float mn = fmaxf(m_ref[r], tm);
          alpha[r] = (mn == -INFINITY || mn == m_ref[r]) ? 1.f : ex2_approx(m_ref[r] - mn);
          any_raise |= mn != m_ref[r] && j > 0;
          m_ref[r] = mn;
          l_t[r] *= alpha[r];
          lr_t[r] *= alpha[r];
        }
        named_bar_sync(1, 128);                 // red[] is reused by the next tile
        if (any_raise) {                        // uniform over the block
          ensure_pv(j - 1);                     // O^T holds PV(0..j-1) complete
          uint32_t o[kN];
          tmem_ld16(lane_base + O_COL, o);
          tmem_wait_ld();
          reg_fence16(o);
#pragma unroll
          for (int r = 0; r < kN; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
          tmem_st16(lane_base + O_COL, o);
          tmem_wait_st();
        }
      }
      // P = 2^(x - m): bf16 to shared memory as the B operand of O^T (row r,
      // key t: box t / 64, 16-byte chunk (t % 64) / 8 swizzled by r % 8)
      ensure_pv(j - 2);                         // P buffer j&1 was read by PV(j-2)
      uint8_t* pbuf = smem + P_OFF + (j & 1) * 2 * PBOX + (t >> 6) * PBOX;
      const int kc = (t & 63) >> 3;
      const int kb2 = (t & 7) * 2;
#pragma unroll
      for (int r = 0; r < kN; ++r) {
        const float pr = m_ref[r] == -INFINITY ? 0.f : ex2_approx(x[r] - m_ref[r]);
        const __nv_bfloat16 pb = __float2bfloat16_rn(pr);
        l_t[r] += pr;
        lr_t[r] += __bfloat162float(pb);
        *reinterpret_cast<__nv_bfloat16*>(pbuf + (r >> 3) * 1024 + (r & 7) * 128 +
                                           ((kc ^ (r & 7)) << 4) + kb2) = pb;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[j & 1]);
    }
    // ------------------------------------------------- partial state
    if (ok) ok = wait_warp(&bars->o_done, 0, wc);
    if (named_bar_any(1, 128, !ok)) {
      ok = false;
    } else {
      tc_fence_after();
      uint32_t o[kN];
      tmem_ld16(lane_base + O_COL, o);
      tmem_wait_ld();
      reg_fence16(o);
#pragma unroll
      for (int r = 0; r < kN; ++r)
        if (r < R) po[r * D + t] = __uint_as_float(o[r]);
      // l and l~ of each row: sums over the 128 key lanes (warp butterflies,
      // then the four warps' partial sums through shared memory)
      float mrow = -INFINITY;
#pragma unroll
      for (int r = 0; r < kN; ++r) {
        float a = l_t[r], c = lr_t[r];
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) {
          a += __shfl_xor_sync(0xffffffffu, a, o2);
          c += __shfl_xor_sync(0xffffffffu, c, o2);
        }
        if (lane == 0) {
          red[warp * kN + r] = a;
          red[(4 + warp) * kN + r] = c;
        }
        if (r == t) mrow = m_ref[r];
      }
      named_bar_sync(1, 128);
      if (t < R) {
        pml[3 * t] = mrow;
        pml[3 * t + 1] = red[t] + red[kN + t] + red[2 * kN + t] + red[3 * kN + t];
        pml[3 * t + 2] = red[4 * kN + t] + red[5 * kN + t] + red[6 * kN + t] + red[7 * kN + t];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

int launch(const DecodeParams& p, cudaStream_t stream) {
  if (const int ea = set_max_dynamic_smem(reinterpret_cast<const void*>(decode_split_tc_kernel), SMEM_BYTES)) return ea;
  CUtensorMap tq, tk, tv;
  const long long rows = (long long)p.B * p.S_max;
  int r = make_tmap_bf16_3d_box(&tq, p.q, 128, p.Hq, (long long)p.B * p.q_len, p.group, p.q_len);
  if (!r) r = make_tmap_bf16_3d(&tk, p.k, 128, p.Hkv, rows, 128);
  if (!r) r = make_tmap_bf16_3d(&tv, p.v, 128, p.Hkv, rows, 128);
  if (r) return r;
  const long long grid = (long long)p.B * p.Hkv * p.nsplit;
  decode_split_tc_kernel<<<(unsigned)grid, kThreads, SMEM_BYTES, stream>>>(tq, tk, tv, p);
  return (int)cudaGetLastError();
}

}  // namespace tc

// One warp per output row (query token, head): merge the chunks' partial
// states, write O and LSE.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeParams p) {
  const long long wid = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long rows = (long long)p.B * p.q_len * p.Hq;
  if (wid >= rows) return;
  const int h = (int)(wid % p.Hq);
  const int tq = (int)(wid / p.Hq);               // query token b * q_len + qi
  const int b = tq / p.q_len;
  const int qi = tq % p.q_len;
  const int L = p.seqlens ? __ldg(p.seqlens + b) : p.S_max;
  if (L < p.q_len || L > p.S_max) return;         // reported by the split kernel
  const int g = h / p.group;
  const int r = qi * p.group + h % p.group;
  const int ns = (L + p.chunk - 1) / p.chunk;
  const long long u0 = ((long long)b * p.Hkv + g) * p.nsplit;
  float M = -INFINITY;
  for (int s = lane; s < ns; s += 32) M = fmaxf(M, p.part_ml[((u0 + s) * p.R + r) * 3]);
  M = warp_max(M);
  constexpr int PER = D / 32;
  float o[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) o[i] = 0.f;
  float lsum = 0.f, lrsum = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float* ml = p.part_ml + ((u0 + s) * p.R + r) * 3;
    const float ms = ml[0];
    if (ms == -INFINITY) continue;                // chunk with nothing visible
    const float wgt = ex2_approx(ms - M);
    lsum = fmaf(wgt, ml[1], lsum);
    lrsum = fmaf(wgt, ml[2], lrsum);
    const float* src = p.part_o + ((u0 + s) * p.R + r) * D;
#pragma unroll
    for (int i = 0; i < PER; ++i) o[i] = fmaf(wgt, src[lane + 32 * i], o[i]);
  }
  // O is normalised by the weights its product used; LSE by the exact sum
  const float inv = lrsum > 0.f ? 1.f / lrsum : 0.f;
  const long long orow = ((long long)tq * p.Hq + h) * D;
  if (p.o_f32) {
#pragma unroll
    for (int i = 0; i < PER; ++i) static_cast<float*>(p.o)[orow + lane + 32 * i] = o[i] * inv;
  } else {
#pragma unroll
    for (int i = 0; i < PER; ++i)
      static_cast<__nv_bfloat16*>(p.o)[orow + lane + 32 * i] = __float2bfloat16_rn(o[i] * inv);
  }
  if (lane == 0)
    p.lse[(long long)h * p.B * p.q_len + tq] = lsum > 0.f ? (M + lg2_approx(lsum)) * kLn2 : -INFINITY;
}

template <int D, int RM>
int launch_split(const DecodeParams& p, cudaStream_t stream) {
  using C = DecCfg<D, RM>;
  auto kern = decode_split_kernel<D, RM>;
  if (const int ea = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES)) return ea;
  CUtensorMap tk, tv;
  const long long rows = (long long)p.B * p.S_max;
  int r = make_tmap_bf16_3d(&tk, p.k, D, p.Hkv, rows, kTileKeys);
  if (!r) r = make_tmap_bf16_3d(&tv, p.v, D, p.Hkv, rows, kTileKeys);
  if (r) return r;
  const long long grid = (long long)p.B * p.Hkv * p.nsplit;
  kern<<<(unsigned)grid, kThreads, C::SMEM_BYTES, stream>>>(tk, tv, p);
  return (int)cudaGetLastError();
}

template <int D>
int launch_d(const DecodeParams& p, cudaStream_t stream) {
  int r;
  if (D == 128) r = tc::launch(p, stream);
  else if (p.R <= 1) r = launch_split<D, 1>(p, stream);
  else if (p.R <= 2) r = launch_split<D, 2>(p, stream);
  else if (p.R <= 4) r = launch_split<D, 4>(p, stream);
  else if (p.R <= 8) r = launch_split<D, 8>(p, stream);
  else r = launch_split<D, 16>(p, stream);
  if (r) return r;
  const long long rows = (long long)p.B * p.q_len * p.Hq;
  decode_combine_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(p);
  return (int)cudaGetLastError();
}

}  // namespace

int launch_decode_bf16(const DecodeParams& p, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  return p.d == 128 ? launch_d<128>(p, stream) : launch_d<64>(p, stream);
}

}  // namespace fa
