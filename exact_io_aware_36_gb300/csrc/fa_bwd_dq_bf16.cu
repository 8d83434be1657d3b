// fa_bwd_dq_bf16.cu -- dQ of exact attention without atomics, for sm_103a.
//
// Method ("FlashAttention: Faster Attention Without Dropping a Single
// Interaction", Key design 3): with the forward's LSE and D_i = dO_i . O_i,
// the row i of dQ needs only its own query row and the key/value tiles it
// meets: P_ij = exp(S_ij - LSE_i), dP_ij = dO_i . v_j,
// dS_ij = P_ij (dP_ij - D_i), dQ_i = scale * sum_j dS_ij k_j.  This kernel
// owns 128 query rows and walks their key tiles in a fixed order, keeping
// dQ in TMEM, so dq is the same bit for bit on every run.  It is the
// deterministic backward's replacement for the dQ accumulation of the dK/dV
// kernel (the same page, Limitations: a slower deterministic backward is an
// option); it costs two extra MMAs per pair (S and dP are recomputed here).
//
// GB300 mapping (one CTA per SM, 192 threads, one block = 128 query rows of
// one head of one sequence):
//   warp 5     TMA producer: Q and dO once; K_j and V_j (64 keys) into a
//              ring of stages with full/empty mbarriers.
//   warp 4     MMA issuer (one lane), per key tile j:
//                S(j)  = Q K_j^T    (M 128, N 64, K d; both K-major)
//                dP(j) = dO V_j^T   (same shape)
//                dQ   += dS(j) K_j  (A = dS from TMEM, B = K_j MN-major)
//              issued as S/dP(0), S/dP(1), then dQ(j), S/dP(j+2), ...
//   warps 0-3  one TMEM lane = one query row: P and dS of the tile's 64
//              keys in fp32; dS goes back to TMEM as bf16 over its S columns.
// TMEM: S buffers at 0 / 64, dP buffers at 128 / 192, dQ at [256, 256 + d).
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_host_util.h"
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 192;
constexpr int kMmaWarp = 4;
constexpr int kLoadWarp = 5;

template <int D>
struct DqCfg {
  static constexpr int NB = D / 64;
  static constexpr int STAGES = D == 128 ? 4 : 8;
  static constexpr int Q_BOX = 128 * 64 * 2;      // 128 rows x 64 columns
  static constexpr int Q_TILE = NB * Q_BOX;
  static constexpr int KV_BOX = 64 * 64 * 2;      // 64 keys x 64 columns
  static constexpr int KV_TILE = NB * KV_BOX;
  static constexpr int Q_OFF = 0;
  static constexpr int DO_OFF = Q_OFF + Q_TILE;
  static constexpr int K_OFF = DO_OFF + Q_TILE;
  static constexpr int V_OFF = K_OFF + STAGES * KV_TILE;
  static constexpr int BAR_OFF = V_OFF + STAGES * KV_TILE;
  static constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per block");
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DQ_COL = 256;   // S, dP: + 64 * buffer
};

struct DqBars {
  uint64_t q_full;
  uint64_t kv_full[8], kv_empty[8];
  uint64_t sdp_full[2];
  uint64_t ds_ready[2];
  uint64_t dq_done;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(DqBars) <= 256, "barrier block");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// BAND: causal band (sliding window p.window); only with CAUSAL.
template <int D, bool CAUSAL, bool ALIBI, bool BAND>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
              const AttnParams p) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  DqBars* bars = reinterpret_cast<DqBars*>(smem + C::BAR_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // 1-D grid, query block slowest: under a causal mask the blocks far down
  // the sequence (most key tiles) start first.
  const int nqb = (p.N + 127) / 128;
  const int hb = (int)(blockIdx.x % (unsigned)(p.Hq * p.B));
  const int qslot = (int)(blockIdx.x / (unsigned)(p.Hq * p.B));
  const int h = hb % p.Hq;
  const int b = hb / p.Hq;
  const int qb = CAUSAL ? nqb - 1 - qslot : qslot;
  long long seq0;
  int L;
  if (!seq_bounds(p, b, &seq0, &L)) {
    if (threadIdx.x == 0) record_status(p.status, FA_ERR_CU_SEQLENS);
    return;
  }
  const int m0 = qb * 128;
  if (m0 >= L) return;
  // Key tiles of 64 this block meets: all without a mask; under the causal
  // mask up to its last row, and with a window w from row m0 - w on.
  const int W = p.window;
  const int rows_end = min(m0 + 128, L);
  const int lo = BAND ? max(0, m0 - W) / 64 : 0;
  const int hi = CAUSAL ? (rows_end - 1) / 64 : (L - 1) / 64;
  const int n = hi - lo + 1;                       // >= 1

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->sdp_full[i], 1);
      mbar_init(&bars->ds_ready[i], 4);
    }
    mbar_init(&bars->dq_done, 1);
    bars->abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtx wc{&bars->abort_flag, p.status};

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    const int kvh = h / p.group;
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(&bars->q_full, 2 * C::Q_TILE);
#pragma unroll
      for (int bx = 0; bx < C::NB; ++bx) {
        tma_load_3d(smem + C::Q_OFF + bx * C::Q_BOX, &tmQ, bx * 64, h, (int)(seq0 + m0), &bars->q_full);
        tma_load_3d(smem + C::DO_OFF + bx * C::Q_BOX, &tmdO, bx * 64, h, (int)(seq0 + m0), &bars->q_full);
      }
    }
    __syncwarp();
    int issued = 0;
    for (int j = 0; j < n; ++j) {
      const int st = j % C::STAGES;
      if (!wait_warp(&bars->kv_empty[st], ((j / C::STAGES) & 1) ^ 1, wc)) break;
      if (lane == 0) {
        const int row = (int)(seq0 + 64 * (lo + j));
        mbar_arrive_expect_tx(&bars->kv_full[st], 2 * C::KV_TILE);
#pragma unroll
        for (int bx = 0; bx < C::NB; ++bx) {
          tma_load_3d(smem + C::K_OFF + st * C::KV_TILE + bx * C::KV_BOX, &tmK, bx * 64, kvh, row,
                      &bars->kv_full[st]);
          tma_load_3d(smem + C::V_OFF + st * C::KV_TILE + bx * C::KV_BOX, &tmV, bx * 64, kvh, row,
                      &bars->kv_full[st]);
        }
      }
      __syncwarp();
      issued = j + 1;
    }
    // Loads in flight must land before this CTA's shared memory goes away.
    wait_warp_drain(&bars->q_full, 0);
    for (int j = max(0, issued - C::STAGES); j < issued; ++j)
      wait_warp_drain(&bars->kv_full[j % C::STAGES], (j / C::STAGES) & 1);
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t ID_S = idesc_bf16_f32(128, 64, 0, 0);    // S, dP
    constexpr uint32_t ID_DQ = idesc_bf16_f32(128, D, 0, 1);    // dQ (A from TMEM)
    const uint32_t sQ = smem_u32(smem + C::Q_OFF);
    const uint32_t sdO = smem_u32(smem + C::DO_OFF);
    const uint32_t sK = smem_u32(smem + C::K_OFF);
    const uint32_t sV = smem_u32(smem + C::V_OFF);
    // Base descriptors, built once; each MMA's operand is an offset from them.
    const uint64_t qdesc = smem_desc_sw128(sQ, 16, 1024), odesc = smem_desc_sw128(sdO, 16, 1024);
    const uint64_t kdesc0 = smem_desc_sw128(sK, 16, 1024), vdesc0 = smem_desc_sw128(sV, 16, 1024);
    const uint64_t kmn0 = smem_desc_sw128(sK, C::KV_BOX, 1024);
    auto issue_sdp = [&](int j) {
      const int st = j % C::STAGES;
      const uint32_t buf = (uint32_t)(j & 1);
      const uint64_t kd = desc_add(kdesc0, st * C::KV_TILE), vd = desc_add(vdesc0, st * C::KV_TILE);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(tmem + C::S_COL + 64 * buf, desc_add(qdesc, (kk >> 2) * C::Q_BOX + (kk & 3) * 32),
               desc_add(kd, (kk >> 2) * C::KV_BOX + (kk & 3) * 32), ID_S, kk > 0 ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(tmem + C::DP_COL + 64 * buf, desc_add(odesc, (kk >> 2) * C::Q_BOX + (kk & 3) * 32),
               desc_add(vd, (kk >> 2) * C::KV_BOX + (kk & 3) * 32), ID_S, kk > 0 ? 1u : 0u);
      mma_commit(&bars->sdp_full[buf]);
    };
    bool ok = wait_warp(&bars->q_full, 0, wc);
    for (int j = 0; ok && j < 2 && j < n; ++j) {
      if (!(ok = wait_warp(&bars->kv_full[j % C::STAGES], (j / C::STAGES) & 1, wc))) break;
      tc_fence_after();
      if (lane == 0) issue_sdp(j);
      __syncwarp();
    }
    for (int j = 0; ok && j < n; ++j) {
      const int st = j % C::STAGES;
      const uint32_t buf = (uint32_t)(j & 1);
      if (!(ok = wait_warp(&bars->ds_ready[buf], (j >> 1) & 1, wc))) break;
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)   // dQ += dS K   (K = 64 keys, 16 per MMA)
          mma_ts(tmem + C::DQ_COL, tmem + C::S_COL + 64 * buf + 8 * kk,
                 desc_add(kmn0, st * C::KV_TILE + kk * 2048), ID_DQ, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars->kv_empty[st]);
      }
      __syncwarp();
      // S/dP(j+2) reuse the columns of step j: the compute warps are done
      // with them (ds_ready), and dQ(j) reads its dS first (MMAs run in
      // issue order).
      const int nx = j + 2;
      if (nx < n) {
        if (!(ok = wait_warp(&bars->kv_full[nx % C::STAGES], (nx / C::STAGES) & 1, wc))) break;
        tc_fence_after();
        if (lane == 0) issue_sdp(nx);
        __syncwarp();
      }
    }
    if (lane == 0) mma_commit(&bars->dq_done);
    __syncwarp();
    // Tensor-core work must be finished before the TMEM is released.
    wait_warp_drain(&bars->dq_done, 0);
  } else {
    // ------------------------------------------------------------- compute
    const int r = 32 * warp + lane;
    const int row = m0 + r;                     // query row within the sequence
    const bool valid = row < L;
    const long long tok = seq0 + row;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
    // log2-domain row statistics; a row past the sequence end gets +inf, so
    // its P and dS are exactly 0
    const float L2 = valid ? __ldg(p.lse + (long long)h * p.T + tok) * kLog2e : INFINITY;
    const float Dv = valid ? __ldg(p.D + (long long)h * p.T + tok) : 0.f;
    const float slope2 = ALIBI ? __ldg(p.alibi + h) * kLog2e : 0.f;
    const uint64_t c2p = f2(p.scale_log2, p.scale_log2);
    const uint64_t dvp = f2(Dv, Dv);
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const uint32_t buf = (uint32_t)(j & 1);
      if (!(ok = wait_warp(&bars->sdp_full[buf], (j >> 1) & 1, wc))) break;
      tc_fence_after();
      const int n0 = 64 * (lo + j);
      const bool need_mask = (CAUSAL && n0 + 63 > m0) || (BAND && n0 < m0 + 127 - W) || (n0 + 64 > L);
      // x = s * scale * log2(e) + slope2 * (key - row) - L2
      const float base = ALIBI ? fmaf(slope2, (float)(n0 - row), -L2) : -L2;
      const uint32_t tS = lane_base + C::S_COL + 64 * buf;
      const uint32_t tP = lane_base + C::DP_COL + 64 * buf;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {    // 32 keys at a time
        uint32_t sv[32], dp[32];
        tmem_ld32(tS + 32 * half, sv);
        tmem_ld32(tP + 32 * half, dp);
        tmem_wait_ld();
        reg_fence32(sv);
        reg_fence32(dp);
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int cc = 32 * half + 2 * c;      // key within the tile
          const uint64_t bias = ALIBI ? f2(fmaf(slope2, (float)cc, base), fmaf(slope2, (float)(cc + 1), base))
                                      : f2(base, base);
          float x0, x1;
          f2split(ffma2(f2(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])), c2p, bias), x0, x1);
          float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          if (need_mask) {
            const int key = n0 + cc;
            if (key >= L || (CAUSAL && key > row) || (BAND && key < row - W)) p0 = 0.f;
            if (key + 1 >= L || (CAUSAL && key + 1 > row) || (BAND && key + 1 < row - W)) p1 = 0.f;
          }
          const uint64_t ds = fmul2(f2(p0, p1), fsub2(f2(__uint_as_float(dp[2 * c]), __uint_as_float(dp[2 * c + 1])), dvp));
          float d0, d1;
          f2split(ds, d0, d1);
          pk[c] = pack_bf16x2(d0, d1);
        }
        tmem_st16(tS + 16 * half, pk);           // dS (bf16) over consumed S columns
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ds_ready[buf]);
    }
    // ------------------------------------------------------------ epilogue
    if (ok) ok = wait_warp(&bars->dq_done, 0, wc);
    if (ok) {
      tc_fence_after();
      const float sc = p.scale;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.dq) + (tok * p.Hq + h) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(lane_base + C::DQ_COL + c0, rr);
        tmem_wait_ld();
        reg_fence32(rr);
        uint32_t pkd[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pkd[e] = pack_bf16x2(__uint_as_float(rr[2 * e]) * sc, __uint_as_float(rr[2 * e + 1]) * sc);
        if (valid) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) d4[v4] = make_uint4(pkd[4 * v4], pkd[4 * v4 + 1], pkd[4 * v4 + 2], pkd[4 * v4 + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool ALIBI, bool BAND>
int launch_impl(const AttnParams& p, cudaStream_t stream) {
  using C = DqCfg<D>;
  auto kern = bwd_dq_kernel<D, CAUSAL, ALIBI, BAND>;
  if (const int ea = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES)) return ea;
  CUtensorMap tq, tk, tv, tdo;
  int r = make_tmap_bf16_3d(&tq, p.q, D, p.Hq, p.T, 128);
  if (!r) r = make_tmap_bf16_3d(&tdo, p.dO, D, p.Hq, p.T, 128);
  if (!r) r = make_tmap_bf16_3d(&tk, p.k, D, p.Hkv, p.T, 64);
  if (!r) r = make_tmap_bf16_3d(&tv, p.v, D, p.Hkv, p.T, 64);
  if (r) return r;
  dim3 grid((unsigned)(((p.N + 127) / 128) * p.Hq * p.B));
  kern<<<grid, kThreads, C::SMEM_BYTES, stream>>>(tq, tk, tv, tdo, p);
  return (int)cudaGetLastError();
}

template <int D>
int launch_masks(const AttnParams& p, cudaStream_t stream) {
  const bool alibi = p.alibi != nullptr;
  if (p.causal && p.window != kNoWindow)
    return alibi ? launch_impl<D, true, true, true>(p, stream) : launch_impl<D, true, false, true>(p, stream);
  if (p.causal)
    return alibi ? launch_impl<D, true, true, false>(p, stream) : launch_impl<D, true, false, false>(p, stream);
  return alibi ? launch_impl<D, false, true, false>(p, stream) : launch_impl<D, false, false, false>(p, stream);
}

}  // namespace

int launch_bwd_dq_bf16(const AttnParams& p, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  return p.d == 128 ? launch_masks<128>(p, stream) : launch_masks<64>(p, stream);
}

}  // namespace fa
