// fa_fwd_bf16.cu -- tensor-core forward of exact attention for sm_103a.
//
// Method ("FlashAttention: Faster Attention Without Dropping a Single
// Interaction"): Key design 1 (tiles of Q, K, V staged on chip; S and P never
// leave the SM), Key design 2 (running max m and sum l merged tile by tile,
// the output accumulator rescaled when m grows; FA2's L = m + log l saved per
// row), Key design 4 (FA2's sequence-parallel work items; FA3-style
// asynchrony: producer, MMA, softmax and correction roles).
//
// Persistent: one CTA per SM.  A work item is (query block of 256 rows,
// query head, sequence), two query tiles of 128 rows.  Items are numbered
// with the query block slowest (under the causal mask the blocks far down a
// sequence, which see the most key tiles, come first) and the heads of one
// sequence adjacent (a GQA group's query heads share their K/V in L2).  CTA c
// takes, in round r, item r * G + c on even rounds and r * G + G - 1 - c on
// odd ones (G CTAs): a longest-first snake that evens out the CTAs' loads
// without a counter in device memory.  Every role walks the same item list,
// so no item index is passed between them.  All rings, barrier phases and
// TMEM buffers continue across items: the next item's Q and K/V loads and its
// first products overlap the previous item's last products and epilogue.
//
// Roles (CORR = false: 384 threads, warps 10 and 11 idle; CORR = true: 512
// threads):
//   warp 9     TMA producer: per item Q0 / Q1 (each once its buffer's last
//              S product is done), then per step j one slot holding K_j and
//              V_{j-1} (128-byte swizzle) under one full / empty barrier pair.
//   warp 8     MMA issuer (one lane): S_t = Q_t K_j^T into TMEM (both operands
//              K-major in shared memory), O_t += P_t V_j with P_t read from
//              TMEM and V_j MN-major in shared memory.  Per step j the stream
//              is PV0(j-1), S0(j), PV1(j-1), S1(j): the softmax of one tile
//              overlaps the tensor work of the other.
//   warps 0-3  softmax of query tile 0 (one TMEM lane = one query row)
//   warps 4-7  softmax of query tile 1
//   warps 12-15 (CORR) correction warpgroup: rescales O rows in TMEM when a
//              softmax warp raised its reference max, and runs the epilogue
//              (O / l, LSE, stores) while the softmax warps go on with the
//              next item.  Without CORR the softmax warps do both.
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
// P_t (bf16, two per 32-bit column) overwrites the first 64 columns of S_t.
//
// Softmax in base 2: x = s * scale * log2(e) (+ slope * log2(e) * (j - i)),
// p = 2^(x - m_ref).  The reference max m_ref is only raised when a tile's
// max exceeds it by more than kTau = 8 (lazy rescale): the result is the same
// for any reference, and p stays <= 2^8.  When it is raised, the O row is
// rescaled in TMEM before PV_t(j) is issued; that is safe then because the
// commit that published S_t(j) also covers PV_t(j-1).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "fa_host_util.h"
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

#ifndef FA_FWD_CORRECTION_WARPS
#define FA_FWD_CORRECTION_WARPS 0
#endif


constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kCorrWarp0 = 12;
constexpr float kTau = 8.0f;
constexpr float kSpecSum = 256.0f;   // 2^kTau

// Register limits per thread.  The softmax warpgroups raise theirs (a row of
// S lives in registers), the warpgroup of the MMA and producer warps (warps
// 8-11) lowers its, and so does the correction warpgroup under CORR.  The
// limits of a CTA's warpgroups must add up to at most what it is launched
// with: 3 x 168 for 384 threads, 4 x 128 for 512.
constexpr uint32_t kRegsCtl = 56;
constexpr uint32_t kRegsSoftmax3 = 224;                       // without CORR
constexpr uint32_t kRegsSoftmax4 = 176, kRegsCorr = 104;      // with CORR
static_assert(2 * kRegsSoftmax3 + kRegsCtl <= 3 * 168, "register split (384 threads)");
static_assert(2 * kRegsSoftmax4 + kRegsCorr + kRegsCtl <= 4 * 128, "register split (512 threads)");

template <int D, bool CORR>
struct FwdCfg {
  static constexpr int NB = D / 64;                 // 64-column boxes per row
  static constexpr int BOX_BYTES = 128 * 64 * 2;    // one 128 x 64 bf16 box
  static constexpr int TILE_BYTES = NB * BOX_BYTES; // one 128 x D tile
  static constexpr int NS = D == 128 ? 2 : 5;      // slots (K_j, V_{j-1})
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + 2 * TILE_BYTES;
  static constexpr int V_OFF = K_OFF + NS * TILE_BYTES;
  // CORR: row stats and alphas handed to the correction warpgroup.
  static constexpr int STAT_OFF = V_OFF + NS * TILE_BYTES;
  static constexpr int STAT_BYTES = CORR ? 2 * 128 * 4 * 4 : 0;
  static constexpr int BAR_OFF = STAT_OFF + STAT_BYTES;
  static constexpr int SMEM_BYTES = BAR_OFF + 512 + 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static constexpr uint32_t S_COL0 = 0, S_COL1 = 128;
  static constexpr uint32_t O_COL0 = 256, O_COL1 = 256 + D;
};

struct FwdBars {
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[8], kv_empty[8];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done[2], o_free[2];
  uint64_t corr_req[2][4], corr_done[2][4];   // CORR: requests of softmax warp (t, q)
  uint64_t mma_drain;
  int req_kind[2][4];                          // 0: rescale, 1: epilogue
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(FwdBars) <= 512, "barrier block");

// Per-row data the softmax warps hand to the correction warpgroup, [tile][row]:
// m (log2 units), l (exact sum), lr (sum of the bf16-rounded p), alpha.
struct RowStats {
  float m[2][128], l[2][128], lr[2][128], alpha[2][128];
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// One work item: query rows [m0, m0 + 256) of head h of sequence b.  Query
// tile t (rows m0 + 128 t ...) needs kv tiles lo[t] .. hi[t]; the K/V stream
// covers lo[0] .. hi[1] in steps 0 .. nkv_max (the last step only has V),
// and tile t is active on steps [k0[t], k0[t] + nkv[t]).  With ALiBi the
// tiles go from the diagonal backwards: the positive slope makes scores grow
// toward the diagonal, so the first tile holds (nearly) the row max and the
// lazy rescale almost never fires.
struct FwdItem {
  int h, b, m0, L;
  long long seq0;
  bool tile1;
  int lo[2], hi[2], nkv[2], k0[2], nkv_max;
};

template <bool CAUSAL, bool ALIBI, bool BAND>
__device__ __forceinline__ int fwd_item(const AttnParams& p, int idx, FwdItem& it) {
  // returns 1: work, 0: empty (a block past the sequence end), -1: malformed
  const int nqb = (p.N + 255) / 256;
  const int hb = idx % (p.Hq * p.B);
  const int qslot = idx / (p.Hq * p.B);
  it.h = hb % p.Hq;
  it.b = hb / p.Hq;
  const int qb = CAUSAL ? nqb - 1 - qslot : qslot;
  if (!seq_bounds(p, it.b, &it.seq0, &it.L)) return -1;
  it.m0 = qb * 256;
  if (it.m0 >= it.L) return 0;
  it.tile1 = it.m0 + 128 < it.L;
  const int W = p.window;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r0 = it.m0 + 128 * t;
    const int rows_end = min(r0 + 128, it.L);
    it.lo[t] = BAND ? max(0, r0 - W) / 128 : 0;
    it.hi[t] = CAUSAL ? (rows_end - 1) / 128 : (it.L - 1) / 128;
    it.nkv[t] = it.hi[t] - it.lo[t] + 1;
  }
  if (!it.tile1) {
    it.nkv[1] = 0;
    it.lo[1] = it.lo[0];
    it.hi[1] = it.hi[0];
  }
  it.nkv_max = it.hi[1] - it.lo[0] + 1;
  it.k0[0] = ALIBI ? it.hi[1] - it.hi[0] : 0;
  it.k0[1] = ALIBI ? 0 : it.lo[1] - it.lo[0];
  return 1;
}

template <bool ALIBI>
__device__ __forceinline__ int kv_tile(const FwdItem& it, int k) {
  return ALIBI ? it.hi[1] - k : it.lo[0] + k;
}

// Item index of round r for this CTA (snake order); >= nitems when done.
__device__ __forceinline__ int item_of_round(int r) {
  const int G = (int)gridDim.x;
  return r * G + ((r & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
}

// Epilogue of one query row: O = acc / lr from TMEM columns tO.., LSE from
// (m, l); writes the row's O (fp32 or bf16) and LSE.  Loads O in two halves
// of D / 2 columns; after the second load the TMEM columns are no longer
// needed and `release` runs (o_free).  Warp-collective (TMEM loads).
template <int D, typename Release>
__device__ __forceinline__ void epilogue_row(const AttnParams& p, uint32_t tO, bool valid,
                                             long long tok, int h, float m, float l, float lr,
                                             Release release) {
  const float inv = lr > 0.f ? 1.f / lr : 0.f;
#pragma unroll 1
  for (int half = 0; half < 2; ++half) {
    uint32_t o[D / 2];
#pragma unroll
    for (int c = 0; c < D / 2; c += 32) tmem_ld32(tO + half * (D / 2) + c, o + c);
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < D / 2; c += 32) reg_fence32(o + c);
    if (half == 1) release();
    const int c0 = half * (D / 2);
    if (valid) {
      if (p.o_f32) {
        float4* O = reinterpret_cast<float4*>(static_cast<float*>(p.o) + (tok * p.Hq + h) * D + c0);
#pragma unroll
        for (int v4 = 0; v4 < D / 8; ++v4)
          O[v4] = make_float4(__uint_as_float(o[4 * v4]) * inv, __uint_as_float(o[4 * v4 + 1]) * inv,
                              __uint_as_float(o[4 * v4 + 2]) * inv, __uint_as_float(o[4 * v4 + 3]) * inv);
      } else {
        uint4* O = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + (tok * p.Hq + h) * D + c0);
#pragma unroll
        for (int v4 = 0; v4 < D / 16; ++v4)
          O[v4] = make_uint4(pack_bf16x2(__uint_as_float(o[8 * v4]) * inv, __uint_as_float(o[8 * v4 + 1]) * inv),
                             pack_bf16x2(__uint_as_float(o[8 * v4 + 2]) * inv, __uint_as_float(o[8 * v4 + 3]) * inv),
                             pack_bf16x2(__uint_as_float(o[8 * v4 + 4]) * inv, __uint_as_float(o[8 * v4 + 5]) * inv),
                             pack_bf16x2(__uint_as_float(o[8 * v4 + 6]) * inv, __uint_as_float(o[8 * v4 + 7]) * inv));
      }
    }
  }
  if (valid) p.lse[(long long)h * p.T + tok] = l > 0.f ? (m + lg2_approx(l)) * kLn2 : -INFINITY;
}

// O row (D columns at tO) *= alpha, in TMEM.  Warp-collective.
template <int D>
__device__ __forceinline__ void rescale_row(uint32_t tO, float alpha) {
#pragma unroll 1
  for (int c0 = 0; c0 < D; c0 += 16) {
    uint32_t o[16];
    tmem_ld16(tO + c0, o);
    tmem_wait_ld();
    reg_fence16(o);
#pragma unroll
    for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
    tmem_st16(tO + c0, o);
  }
}

// BAND: causal band (sliding window p.window); only with CAUSAL.
// CORR: the correction warpgroup owns O's rescaling and the epilogue.
template <int D, bool CAUSAL, bool ALIBI, bool BAND, bool CORR>
__global__ void __launch_bounds__(CORR ? 512 : 384, 1)
fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const AttnParams p, const int nitems) {
  using C = FwdCfg<D, CORR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + C::BAR_OFF);
  RowStats* stats = reinterpret_cast<RowStats*>(smem + C::STAT_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->q_full[t], 1);
      mbar_init(&bars->q_empty[t], 1);
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 4);
      mbar_init(&bars->o_done[t], 1);
      mbar_init(&bars->o_free[t], 4);
      for (int q = 0; q < 4; ++q) {
        mbar_init(&bars->corr_req[t][q], 1);
        mbar_init(&bars->corr_done[t][q], 1);
      }
    }
    for (int s = 0; s < 8; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->mma_drain, 1);
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
  // Bounded wait, inlined: code under a changed register limit holds no calls.
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool { return wait_warp_inl(bar, parity, wc); };

  // Each warpgroup sets its register limit at the head of its role's branch
  // (the limits then hold for the code each branch holds).
  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    regs_lower<kRegsCtl>();
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    bool ok = true;
    int n = 0;                 // items done (both tiles' Q buffers cycle per item)
    int g = 0;                 // K/V steps issued over all items
    for (int r = 0; ok; ++r) {
      const int idx = item_of_round(r);
      if (idx >= nitems) break;
      FwdItem it;
      const int kind = fwd_item<CAUSAL, ALIBI, BAND>(p, idx, it);
      if (kind < 0 && lane == 0) record_status(p.status, FA_ERR_CU_SEQLENS);
      if (kind <= 0) continue;
      const int kvh = it.h / p.group;
      // Q_t once the previous item's last S_t product has read its buffer
      // (an item without tile 1 still passes its phase through, empty).
      for (int t = 0; t < 2; ++t) {
        if (n > 0 && !(ok = wait(&bars->q_empty[t], (n - 1) & 1))) break;
        if (lane == 0) {
          const bool has = t == 0 || it.tile1;
          mbar_arrive_expect_tx(&bars->q_full[t], has ? C::TILE_BYTES : 0);
          if (has)
#pragma unroll
            for (int bx = 0; bx < C::NB; ++bx)
              tma_load_3d(smem + C::Q_OFF + t * C::TILE_BYTES + bx * C::BOX_BYTES, &tmQ, bx * 64, it.h,
                          (int)(it.seq0 + it.m0 + 128 * t), &bars->q_full[t]);
        }
        __syncwarp();
      }
      if (!ok) break;
      for (int j = 0; j <= it.nkv_max; ++j, ++g) {  // step j's slot: K_j and V_{j-1}
        const int sl = g % C::NS;
        if (g >= C::NS && !(ok = wait(&bars->kv_empty[sl], ((g / C::NS) - 1) & 1))) break;
        if (lane == 0) {
          const bool has_k = j < it.nkv_max, has_v = j >= 1;
          mbar_arrive_expect_tx(&bars->kv_full[sl], (has_k + has_v) * C::TILE_BYTES);
#pragma unroll
          for (int bx = 0; bx < C::NB; ++bx) {
            if (has_k)
              tma_load_3d(smem + C::K_OFF + sl * C::TILE_BYTES + bx * C::BOX_BYTES, &tmK, bx * 64, kvh,
                          (int)(it.seq0 + 128 * kv_tile<ALIBI>(it, j)), &bars->kv_full[sl]);
            if (has_v)
              tma_load_3d(smem + C::V_OFF + sl * C::TILE_BYTES + bx * C::BOX_BYTES, &tmV, bx * 64, kvh,
                          (int)(it.seq0 + 128 * kv_tile<ALIBI>(it, j - 1)), &bars->kv_full[sl]);
          }
        }
        __syncwarp();
      }
      ++n;
    }
    // Loads in flight must land before this CTA's shared memory goes away.
    if (n > 0) {
      wait_warp_drain(&bars->q_full[0], (n - 1) & 1);
      wait_warp_drain(&bars->q_full[1], (n - 1) & 1);
    }
    for (int s = max(0, g - C::NS); s < g; ++s) wait_warp_drain(&bars->kv_full[s % C::NS], (s / C::NS) & 1);
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    regs_lower<kRegsCtl>();
    constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, 0, 0);
    constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, 0, 1);
    const uint32_t sQ = smem_u32(smem + C::Q_OFF);
    const uint32_t sK = smem_u32(smem + C::K_OFF);
    const uint32_t sV = smem_u32(smem + C::V_OFF);
    const uint32_t colS[2] = {C::S_COL0, C::S_COL1};
    const uint32_t colO[2] = {C::O_COL0, C::O_COL1};
    // Base descriptors, built once; each MMA's operand is an offset from them.
    const uint64_t qdesc[2] = {smem_desc_sw128(sQ, 16, 1024), smem_desc_sw128(sQ + C::TILE_BYTES, 16, 1024)};
    const uint64_t kdesc0 = smem_desc_sw128(sK, 16, 1024);
    const uint64_t vdesc0 = smem_desc_sw128(sV, C::BOX_BYTES, 1024);
    bool ok = true;
    int n = 0, g = 0;
    int cs[2] = {0, 0};        // S_t products issued (s_full / p_full phases)
    int nt[2] = {0, 0};        // items in which tile t was active (o_done / o_free phases)
    for (int r = 0; ok; ++r) {
      const int idx = item_of_round(r);
      if (idx >= nitems) break;
      FwdItem it;
      if (fwd_item<CAUSAL, ALIBI, BAND>(p, idx, it) <= 0) continue;
      bool q_waited[2] = {false, false};
      const int cs0[2] = {cs[0], cs[1]};               // this item's first S_t product
      for (int j = 0; ok && j <= it.nkv_max; ++j, ++g) {
        const int sl = g % C::NS;                       // K_j and V_{j-1}
        const uint64_t kdesc = desc_add(kdesc0, sl * C::TILE_BYTES);
        const uint64_t vdesc = desc_add(vdesc0, sl * C::TILE_BYTES);
        // TMA data needs no tcgen05 fence: the MMAs read it once the
        // transaction count of the slot's barrier has completed.
        if (!(ok = wait(&bars->kv_full[sl], (g / C::NS) & 1))) break;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int jl = j - 1 - it.k0[t];              // tile t's local PV step
          if (j >= 1 && jl >= 0 && jl < it.nkv[t]) {
            if (!(ok = wait(&bars->p_full[t], (cs0[t] + jl) & 1))) break;
            // The item's first PV_t overwrites O_t: the previous item's
            // epilogue must have read it.
            if (jl == 0 && nt[t] > 0 && !(ok = wait(&bars->o_free[t], (nt[t] - 1) & 1))) break;
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
              for (int kk = 0; kk < 128 / 16; ++kk)
                mma_ts(tmem + colO[t], tmem + colS[t] + kk * 8, desc_add(vdesc, kk * 2048), IDESC_O,
                       (jl > 0 || kk > 0) ? 1u : 0u);
              if (jl == it.nkv[t] - 1) mma_commit(&bars->o_done[t]);
            }
            __syncwarp();
          }
          const int js = j - it.k0[t];                  // tile t's local S step
          if (js >= 0 && js < it.nkv[t]) {
            if (!q_waited[t]) {
              if (!(ok = wait(&bars->q_full[t], n & 1))) break;
              q_waited[t] = true;
            }
            if (lane == 0) {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
                mma_ss(tmem + colS[t], desc_add(qdesc[t], off), desc_add(kdesc, off), IDESC_S, kk > 0 ? 1u : 0u);
              }
              mma_commit(&bars->s_full[t]);
              if (js == it.nkv[t] - 1) mma_commit(&bars->q_empty[t]);
            }
            __syncwarp();
            ++cs[t];
          }
        }
        if (!ok) break;
        if (lane == 0) mma_commit(&bars->kv_empty[sl]);
        __syncwarp();
      }
      if (!ok) break;
      // An item without tile 1 passes its Q phases through: the producer
      // waits on q_empty[1] once per item.
      if (!it.tile1) {
        if (!(ok = wait(&bars->q_full[1], n & 1))) break;
        if (lane == 0) mbar_arrive(&bars->q_empty[1]);
        __syncwarp();
      }
      for (int t = 0; t < 2; ++t) nt[t] += it.nkv[t] > 0;
      ++n;
    }
    // Tensor-core work must be finished before the TMEM is released.
    if (lane == 0) mma_commit(&bars->mma_drain);
    __syncwarp();
    wait_warp_drain(&bars->mma_drain, 0);
  } else if (warp < 8) {
    // ------------------------------------------------------------- softmax
    if constexpr (CORR) regs_raise<kRegsSoftmax4>();
    else regs_raise<kRegsSoftmax3>();
    const int t = warp >> 2;
    const int q4 = warp & 3;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q4) << 16);
    const uint32_t tS = lane_base + (t ? C::S_COL1 : C::S_COL0);
    const uint32_t tO = lane_base + (t ? C::O_COL1 : C::O_COL0);
    const float c2 = p.scale_log2;
    bool ok = true;
    int cs = 0;                // S_t products consumed (s_full / p_full phases)
    int nt = 0;                // items in which this tile was active
    int nreq = 0;              // CORR: requests sent to correction warp (t, q4)
    const int r_in_tile = 32 * q4 + lane;
    // CORR: before a new request, the previous one must have been taken
    // (its data read), so the request barrier never runs two phases ahead.
    auto request_slot_free = [&]() -> bool {
      return nreq == 0 || wait(&bars->corr_done[t][q4], (nreq - 1) & 1);
    };
    for (int r = 0; ok; ++r) {
      const int idx = item_of_round(r);
      if (idx >= nitems) break;
      int h, L, nsteps, kv_first, r0;
      long long seq0;
      {
        FwdItem it;
        if (fwd_item<CAUSAL, ALIBI, BAND>(p, idx, it) <= 0) continue;
        if (it.nkv[t] == 0) continue;                   // uniform over the tile's warps
        h = it.h;
        L = it.L;
        seq0 = it.seq0;
        nsteps = it.nkv[t];
        kv_first = kv_tile<ALIBI>(it, it.k0[t]);        // the tile's first kv tile
        r0 = it.m0 + 128 * t;
      }
      const int row = r0 + r_in_tile;                   // row within the sequence
      float slope2 = 0.f;
      if (ALIBI) slope2 = __ldg(p.alibi + h) * kLog2e;
      float m_ref = -INFINITY;
      float l = 0.f;     // sum of p in fp32: gives the LSE
      float lr = 0.f;    // sum of the bf16-rounded p the PV MMA sees: normalises O
      for (int j = 0; j < nsteps; ++j, ++cs) {          // j: this tile's local step
        if (!(ok = wait(&bars->s_full[t], cs & 1))) break;
        tc_fence_after();
        uint32_t s[128];
        tmem_ld32(tS + 0, s);
        tmem_ld32(tS + 32, s + 32);
        tmem_ld32(tS + 64, s + 64);
        tmem_ld32(tS + 96, s + 96);
        tmem_wait_ld();
        reg_fence32(s);
        reg_fence32(s + 32);
        reg_fence32(s + 64);
        reg_fence32(s + 96);
        const int n0 = 128 * (ALIBI ? kv_first - j : kv_first + j);
        const int W = p.window;
        const bool need_mask = (CAUSAL && n0 + 127 > r0) || (BAND && n0 < r0 + 127 - W) || (n0 + 128 > L);
        // Masked scores become -inf (raw scores stay in s; the scale and the
        // ALiBi bias are applied where they are consumed).  A row can meet a
        // tile that is wholly outside its band; its scores are then all -inf,
        // its p all 0, and its state unchanged.
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            const int key = n0 + c;
            if (key >= L || (CAUSAL && key > row) || (BAND && key < row - W)) s[c] = __float_as_uint(-INFINITY);
          }
        }
        // ALiBi bias of column c in log2 units: slope2 * (n0 + c - row).
        const float base = ALIBI ? slope2 * (float)(n0 - row) : 0.f;
        // p = 2^(x - m) with packed f32x2 scale-and-subtract and MUFU exp2;
        // P is stored to TMEM as produced; returns the tile's sums of the
        // exact p and of the bf16-rounded p the PV MMA sees.
        const uint64_t c2p = f2(c2, c2);
        auto exp_pass = [&](float mb, float& ts, float& tsr) {
          const uint64_t nmb = f2(-mb, -mb);
          const uint64_t step = f2(2.f * slope2, 2.f * slope2);
          uint64_t acc[2] = {0, 0}, accr[2] = {0, 0};
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t pk[16];
            // ALiBi: bias - m for the pair (c, c+1), exact at the chunk start
            // and advanced by 2 * slope2 per pair (16 steps at most).
            uint64_t bm = ALIBI ? f2(fmaf(slope2, (float)(32 * ch), base - mb),
                                     fmaf(slope2, (float)(32 * ch + 1), base - mb))
                                : nmb;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const uint64_t xy = f2(__uint_as_float(s[32 * ch + 2 * c]), __uint_as_float(s[32 * ch + 2 * c + 1]));
              const uint64_t e = ffma2(xy, c2p, bm);
              if (ALIBI) bm = fadd2(bm, step);
              float e0, e1;
              f2split(e, e0, e1);
              const float p0 = ex2_approx(e0);
              const float p1 = ex2_approx(e1);
              acc[c & 1] = fadd2(acc[c & 1], f2(p0, p1));
              pk[c] = pack_bf16x2(p0, p1);
              accr[c & 1] = fadd2(accr[c & 1], f2(__uint_as_float(pk[c] << 16),
                                                   __uint_as_float(pk[c] & 0xFFFF0000u)));
            }
            tmem_st16(tS + 16 * ch, pk);
          }
          float a0, a1, b0, b1;
          f2split(fadd2(acc[0], acc[1]), a0, a1);
          f2split(fadd2(accr[0], accr[1]), b0, b1);
          ts = a0 + a1;
          tsr = b0 + b1;
        };
        // Speculative pass: once a row has a reference max, compute P with it
        // directly.  If the tile's sum of p is at most 2^tau, no p exceeds
        // 2^tau, i.e. no score exceeds the reference by more than tau, so no
        // raise is due and the pass is exactly what the full path would
        // produce.
        float ts = 0.f, tsr = 0.f;
        bool full = __any_sync(0xffffffffu, m_ref == -INFINITY);
        bool spec_over = false;     // this row's speculative sum exceeded 2^tau
        bool raised = false;        // this warp moved a row's reference (j > 0)
        float alpha = 1.f;
        if (!full) {
          exp_pass(m_ref, ts, tsr);
          spec_over = !(ts <= kSpecSum);                      // also catches inf / nan
          full = __any_sync(0xffffffffu, spec_over);
          if (full) tmem_wait_st();
        }
        if (full) {
          float mx[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) mx[i] = -INFINITY;
          if (ALIBI) {       // max of s * c2 + bias
#pragma unroll
            for (int c = 0; c < 128; c += 8)
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int cc = c + 2 * i;
                mx[i] = fmax3(mx[i], fmaf(__uint_as_float(s[cc]), c2, fmaf(slope2, (float)cc, base)),
                              fmaf(__uint_as_float(s[cc + 1]), c2, fmaf(slope2, (float)(cc + 1), base)));
              }
          } else {
#pragma unroll
            for (int c = 0; c < 128; c += 8)
#pragma unroll
              for (int i = 0; i < 4; ++i)
                mx[i] = fmax3(mx[i], __uint_as_float(s[c + 2 * i]), __uint_as_float(s[c + 2 * i + 1]));
          }
          float xmax = fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]);
          if (!ALIBI) xmax *= c2;
          // Lazy rescale: raise the reference when the max grew past tau, and
          // also when this row's speculative sum overflowed (its max then
          // exceeds the reference; without the raise every later tile of a
          // row whose reference came from a few keys would fail the
          // speculation again).  Either choice of reference gives the same
          // result.
          const bool raise = xmax > m_ref + kTau || spec_over;
          const float m_new = raise ? xmax : m_ref;
          alpha = raise ? ex2_approx(m_ref - m_new) : 1.f;
          l *= alpha;
          lr *= alpha;
          raised = j > 0 && __any_sync(0xffffffffu, raise);
          if (!CORR && raised) rescale_row<D>(tO, alpha);
          m_ref = m_new;
          exp_pass(m_ref == -INFINITY ? 0.f : m_ref, ts, tsr);
        }
        l += ts;
        lr += tsr;
        if (CORR && raised) {
          // The correction warp rescales these rows of O and then passes
          // p_full on in this warp's place.
          if (!(ok = request_slot_free())) break;
          stats->alpha[t][r_in_tile] = alpha;
          if (lane == 0) bars->req_kind[t][q4] = 0;
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->corr_req[t][q4]);
          ++nreq;
        } else {
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->p_full[t]);
        }
      }
      // ---------------------------------------------------------- epilogue
      if constexpr (CORR) {
        if (!ok) break;
        if (!(ok = request_slot_free())) break;
        stats->m[t][r_in_tile] = m_ref;
        stats->l[t][r_in_tile] = l;
        stats->lr[t][r_in_tile] = lr;
        if (lane == 0) bars->req_kind[t][q4] = 1;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->corr_req[t][q4]);
        ++nreq;
      } else {
        if (ok) ok = wait(&bars->o_done[t], nt & 1);
        if (ok) tc_fence_after();
        if (!ok) break;
        epilogue_row<D>(p, tO, row < L, seq0 + row, h, m_ref, l, lr, [&] {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->o_free[t]);
        });
      }
      ++nt;
    }
  } else if (CORR && warp >= kCorrWarp0) {
    // ---------------------------------------------------------- correction
    regs_lower<kRegsCorr>();
    // Warp q serves the requests of softmax warps (0, q) and (1, q), which
    // own the same TMEM lanes: rescales of O rows while an item runs, then
    // the item's epilogue.  Requests of the two tiles interleave in time, so
    // the warp polls both barriers.
    const int q4 = warp & 3;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q4) << 16);
    const int r_in_tile = 32 * q4 + lane;
    bool ok = true;
    int nreq[2] = {0, 0};      // requests taken per tile
    int nt[2] = {0, 0};        // epilogues done per tile
    int rr[2] = {0, 0};        // next round to look at per tile
    bool pending[2] = {false, false};   // epilogue requested, waiting for o_done
    float em[2] = {0.f, 0.f}, el[2] = {0.f, 0.f}, elr[2] = {0.f, 0.f};
    long long e_seq0[2] = {0, 0};       // the item each tile's next epilogue is for
    int e_row[2] = {0, 0}, e_L[2] = {0, 0}, e_h[2] = {0, 0};
    bool has[2] = {false, false};
    // next item in which tile t is active, from round rr[t] on
    auto advance = [&](int t) {
      has[t] = false;
      while (true) {
        const int idx = item_of_round(rr[t]);
        if (idx >= nitems) return;
        ++rr[t];
        FwdItem it;
        if (fwd_item<CAUSAL, ALIBI, BAND>(p, idx, it) <= 0) continue;
        if (it.nkv[t] == 0) continue;
        e_seq0[t] = it.seq0;
        e_row[t] = it.m0 + 128 * t + r_in_tile;
        e_L[t] = it.L;
        e_h[t] = it.h;
        has[t] = true;
        return;
      }
    };
    advance(0);
    advance(1);
    // Nothing here blocks on one tile while the other may need service: an
    // epilogue whose products are not done yet is left pending and polled.
    uint64_t idle_since = 0;
    while (ok && (has[0] || has[1])) {
      bool any = false;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (!has[t]) continue;
        const uint32_t tO = lane_base + (t ? C::O_COL1 : C::O_COL0);
        if (pending[t]) {
          if (!__all_sync(0xffffffffu, mbar_try_wait(&bars->o_done[t], nt[t] & 1))) continue;
          any = true;
          tc_fence_after();
          epilogue_row<D>(p, tO, e_row[t] < e_L[t], e_seq0[t] + e_row[t], e_h[t], em[t], el[t], elr[t], [&] {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->o_free[t]);
          });
          pending[t] = false;
          ++nt[t];
          advance(t);
          continue;
        }
        if (!__all_sync(0xffffffffu, mbar_try_wait(&bars->corr_req[t][q4], nreq[t] & 1))) continue;
        any = true;
        tc_fence_after();
        const int kind = bars->req_kind[t][q4];
        if (kind == 0) {                        // rescale, then pass p_full on
          const float alpha = stats->alpha[t][r_in_tile];
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->corr_done[t][q4]);
          rescale_row<D>(tO, alpha);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->p_full[t]);
        } else {                                // epilogue of the tile's item
          em[t] = stats->m[t][r_in_tile];
          el[t] = stats->l[t][r_in_tile];
          elr[t] = stats->lr[t][r_in_tile];
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->corr_done[t][q4]);
          pending[t] = true;
        }
        ++nreq[t];
      }
      if (any) {
        idle_since = 0;
      } else {
        // Back off, so the polling does not take issue slots from the
        // softmax warps that share this SM's schedulers.
        __nanosleep(128);
        // Nothing ready: bounded like every other wait (the limit turns a
        // lost request into an error status instead of a hang).
        int bad = 0;
        if (lane == 0) {
          const uint64_t now = globaltimer_ns();
          if (idle_since == 0) idle_since = now;
          if (bars->abort_flag) bad = 1;
          else if (now - idle_since > kWaitLimitNs) {
            bars->abort_flag = 1;
            record_status(p.status, FA_ERR_DEVICE_TIMEOUT);
            bad = 1;
          }
        }
        idle_since = __shfl_sync(0xffffffffu, idle_since, 0);
        if (__shfl_sync(0xffffffffu, bad, 0)) ok = false;
      }
    }
  } else if (warp < 12) {
    regs_lower<kRegsCtl>();           // warps 10, 11: no role
  }
  // Every warpgroup returns to the launch limit before the common tail.
  if constexpr (CORR) {
    if (warp < 8) regs_lower<128>();
    else regs_raise<128>();
  } else {
    if (warp < 8) regs_lower<168>();
    else regs_raise<168>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool ALIBI, bool BAND, bool CORR>
int launch_impl(const AttnParams& p, cudaStream_t stream) {
  using C = FwdCfg<D, CORR>;
  auto kern = fwd_bf16_kernel<D, CAUSAL, ALIBI, BAND, CORR>;
  if (const int ea = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES)) return ea;
  // The warpgroups' raised register limits draw on what the CTA is launched
  // with (threads x registers per thread); a build that allocated fewer
  // would leave a raise waiting forever, so it is refused here instead.
  static int regs_ok = -1;
  if (regs_ok < 0) {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, reinterpret_cast<const void*>(kern)) != cudaSuccess)
      return (int)cudaErrorInvalidDeviceFunction;
    regs_ok = a.numRegs >= (CORR ? 128 : 168);
  }
  if (!regs_ok) return (int)cudaErrorInvalidConfiguration;
  CUtensorMap tq, tk, tv;
  int r = make_tmap_bf16_3d(&tq, p.q, D, p.Hq, p.T, 128);
  if (!r) r = make_tmap_bf16_3d(&tk, p.k, D, p.Hkv, p.T, 128);
  if (!r) r = make_tmap_bf16_3d(&tv, p.v, D, p.Hkv, p.T, 128);
  if (r) return r;
  const long long nitems = (long long)((p.N + 255) / 256) * p.Hq * p.B;
  int nsm = 0;
  if (const int es = sm_count(&nsm)) return es;
  const unsigned grid = (unsigned)std::min<long long>(nitems, nsm);
  kern<<<grid, CORR ? 512 : 384, C::SMEM_BYTES, stream>>>(tq, tk, tv, p, (int)nitems);
  return (int)cudaGetLastError();
}

template <int D, bool CORR>
int launch_masks(const AttnParams& p, cudaStream_t stream) {
  const bool alibi = p.alibi != nullptr;
  if (p.causal && p.window != kNoWindow)
    return alibi ? launch_impl<D, true, true, true, CORR>(p, stream)
                 : launch_impl<D, true, false, true, CORR>(p, stream);
  if (p.causal)
    return alibi ? launch_impl<D, true, true, false, CORR>(p, stream)
                 : launch_impl<D, true, false, false, CORR>(p, stream);
  return alibi ? launch_impl<D, false, true, false, CORR>(p, stream)
               : launch_impl<D, false, false, false, CORR>(p, stream);
}

}  // namespace

int launch_fwd_bf16_persistent(const AttnParams& p, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  constexpr bool kCorr = FA_FWD_CORRECTION_WARPS != 0;
  return p.d == 128 ? launch_masks<128, kCorr>(p, stream) : launch_masks<64, kCorr>(p, stream);
}

// Which forward runs.  The persistent kernel saves a CTA launch, its set-up
// and the wait for its first loads per work item, and overlaps an item's
// epilogue with the next item's loads and products; that pays where items
// are short.  Where items average more than 16 kv steps (dense causal
// sequences of N > 3840; wide bands) one CTA per query block with a
// TMA-store epilogue is faster (same-box A/B, TFLOP/s, persistent / per
// block: N = 16384 1304 / 1414; N = 8192 with GQA and ALiBi 1133 / 1254;
// N = 4096 1084 - 1091 / 1098; N = 2048 879 / 841; packed lengths of
// 128-4096 951 / 922; N = 1024, d = 64 346 / 332).
int launch_fwd_bf16(const AttnParams& p, void* stream) {
  // Average kv steps of a dense batch's query blocks of 256 rows: N / 256 + 1
  // under the causal mask, N / 128 without, at most (w + 256) / 128 + 1 in a
  // band of width w.  Packed batches always go to the persistent kernel.
  long long steps = p.causal ? p.N / 256 + 1 : (p.N + 127) / 128;
  if (p.causal && p.window != kNoWindow) steps = std::min<long long>(steps, (p.window + 256) / 128 + 1);
  const bool long_items = p.cu_seqlens == nullptr && steps > 16;
  return long_items ? launch_fwd_bf16_block(p, stream) : launch_fwd_bf16_persistent(p, stream);
}

}  // namespace fa
