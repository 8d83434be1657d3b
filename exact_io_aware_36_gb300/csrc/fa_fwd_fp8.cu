// fa_fwd_fp8.cu -- FP8 (e4m3) forward of attention for sm_103a.
//
// Method ("FlashAttention: Faster Attention Without Dropping a Single
// Interaction", FA3: per-block quantization with the incoherent Hadamard
// transform; not exact): the inputs are the codes and per-block scales that
// fa_fp8_quantize writes; the online softmax is that of the bf16 forward
// (Key design 2, base-2 exponentials with a lazily raised reference max), and
// both products run on the tensor cores as kind::f8f6f4 with fp32
// accumulation:
//   S(j)  = Q8 K8_j^T, scaled per tile by scale * s_q * s_k(j) / d (the 1/d
//           undoes the unnormalised Hadamard: (QDH)(KDH)^T = d QK^T);
//   O    += P8 V8_j: P = 2^(x - m) times r(j) = s_v(j) / s_v,max (<= 1, so
//           one V scale per kv head, s_v,max, serves all tiles), rounded to
//           e4m3; O = s_v,max * acc / l~ with l~ the sum of the rounded
//           P / r(j), the weights the product actually used.
// LSE uses the exact sum of P.
//
// GB300 mapping as the bf16 forward (one CTA per SM, 320 threads, two query
// tiles of 128 rows, warp 9 TMA, warp 8 MMA, warps 0-7 softmax), with:
//   - Q8, K8 tiles of 128 rows x 128 bytes (one 128-byte swizzle span), V as
//     its transposed codes (128 head dims x 128 keys), so both products read
//     K-major operands from shared memory;
//   - P8 written by the softmax warps to shared memory (128 rows x 128 keys,
//     swizzled, two buffers per tile) instead of TMEM, as the A operand of
//     the PV product.  With P out of the S columns, S_t(j + 1) goes to the
//     tensor cores as soon as the softmax has read S_t(j) (s_free), not after
//     PV_t(j): the next scores are ready when the softmax finishes a tile, so
//     the two tiles' softmax warps run back to back instead of waiting for
//     PV + S each step.  P buffer b is reused two steps later, after
//     PV_t(j - 2) is done (pv_done[t][b]); p_full is per buffer too, because
//     the softmax can finish step j + 1 before PV_t(j) is issued;
//   - 4 slots of 16 KB K and 16 KB V: slot j holds K_j and V_{j-1}, the
//     operands of step j's products S_t(j) and PV_t(j-1), under one full and
//     one empty barrier (one wait and one release per step for the MMA warp).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_host_util.h"
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 320;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr float kTau = 8.0f;
constexpr float kSpecSum = 256.0f;   // 2^kTau
constexpr int kD = 128;

struct Cfg {
  static constexpr int TILE = 128 * 128;           // 128 rows x 128 bytes
  static constexpr int NS = 4;                     // slots (K_j, V_{j-1})
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + 2 * TILE;
  static constexpr int V_OFF = K_OFF + NS * TILE;
  static constexpr int P_OFF = V_OFF + NS * TILE;   // [tile][buffer] P codes
  static constexpr int BAR_OFF = P_OFF + 4 * TILE;
  static constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per block");
  // The epilogue stages both tiles' O (fp32 at most) in the K/V slots.
  static_assert(2 * 128 * kD * 4 <= P_OFF - K_OFF, "O staging must fit the K/V slots");
  static constexpr uint32_t S_COL0 = 0, S_COL1 = 128;
  static constexpr uint32_t O_COL0 = 256, O_COL1 = 384;
};

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[8], kv_empty[8];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2][2], pv_done[2][2];     // [tile][P buffer]
  uint64_t o_done;
  uint32_t tmem_base;
  int abort_flag;
};

// kind::f8f6f4 instruction descriptor: D f32, A and B e4m3, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Two e4m3 codes of (lo, hi), lo in the low byte; and back to f32 (exact).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Sum of the four e4m3 values of a 32-bit word, as f16x2 (pairs of the word's
// bytes 0 + 2 and 1 + 3; e4m3 values are exact in f16).
__device__ __forceinline__ uint32_t e4m3x4_sum_h2(uint32_t w) {
  uint32_t a, b, r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(a) : "h"((uint16_t)(w & 0xFFFFu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(b) : "h"((uint16_t)(w >> 16)));
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint64_t h2_to_f2(uint32_t h2) {
  float lo, hi;
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi) : "r"(h2));
  return f2(lo, hi);
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <bool CAUSAL, bool ALIBI, bool BAND>
__global__ void __launch_bounds__(kThreads, 1)
fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
               const AttnParams p) {
  using C = Cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  Bars* bars = reinterpret_cast<Bars*>(smem + C::BAR_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // 1-D grid, query block slowest: longest-first under a causal mask.
  const int nqb = (p.N + 255) / 256;
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
  const int m0 = qb * 256;
  if (m0 >= L) return;
  const bool tile1 = m0 + 128 < L;
  const int W = p.window;
  int lo[2], hi[2], nkv[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r0 = m0 + 128 * t;
    const int rows_end = min(r0 + 128, L);
    lo[t] = BAND ? max(0, r0 - W) / 128 : 0;
    hi[t] = CAUSAL ? (rows_end - 1) / 128 : (L - 1) / 128;
    nkv[t] = hi[t] - lo[t] + 1;
  }
  if (!tile1) {
    nkv[1] = 0;
    lo[1] = lo[0];
    hi[1] = hi[0];
  }
  const int nkv_max = hi[1] - lo[0] + 1;
  constexpr bool REV = ALIBI;                    // diagonal-first with ALiBi
  auto kvj = [&](int k) { return REV ? hi[1] - k : lo[0] + k; };
  const int k0[2] = {REV ? hi[1] - hi[0] : 0, REV ? 0 : lo[1] - lo[0]};
  const int kvh = h / p.group;
  const long long nbt = (long long)p.B * p.nblk;  // blocks per head

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->s_free[t], 4);
      for (int bf = 0; bf < 2; ++bf) {
        mbar_init(&bars->p_full[t][bf], 4);
        mbar_init(&bars->pv_done[t][bf], 1);
      }
    }
    mbar_init(&bars->o_done, 1);
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
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int ntiles = tile1 ? 2 : 1;
      mbar_arrive_expect_tx(&bars->q_full, ntiles * C::TILE);
      for (int t = 0; t < ntiles; ++t)
        tma_load_3d(smem + C::Q_OFF + t * C::TILE, &tmQ, 0, h, (int)(seq0 + m0 + 128 * t), &bars->q_full);
    }
    __syncwarp();
    int issued = 0;
    for (int j = 0; j <= nkv_max; ++j) {      // step j: its slot holds K_j and V_{j-1}
      const int sl = j % C::NS;
      if (!wait_warp(&bars->kv_empty[sl], ((j / C::NS) & 1) ^ 1, wc)) break;
      if (lane == 0) {
        const bool has_k = j < nkv_max, has_v = j >= 1;
        mbar_arrive_expect_tx(&bars->kv_full[sl], (has_k + has_v) * C::TILE);
        if (has_k)
          tma_load_3d(smem + C::K_OFF + sl * C::TILE, &tmK, 0, kvh, (int)(seq0 + 128 * kvj(j)), &bars->kv_full[sl]);
        // transposed V codes: x = key column of block (b, kvj), always a multiple of 128
        if (has_v)
          tma_load_3d(smem + C::V_OFF + sl * C::TILE, &tmV, (int)(((long long)b * p.nblk + kvj(j - 1)) * 128), 0,
                      kvh, &bars->kv_full[sl]);
      }
      __syncwarp();
      issued = j + 1;
    }
    wait_warp_drain(&bars->q_full, 0);
    for (int j = max(0, issued - C::NS); j < issued; ++j)
      wait_warp_drain(&bars->kv_full[j % C::NS], (j / C::NS) & 1);
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t IDESC = idesc_e4m3_f32(128, 128);   // S and O: M = N = 128
    const uint32_t sQ = smem_u32(smem + C::Q_OFF);
    const uint32_t sK = smem_u32(smem + C::K_OFF);
    const uint32_t sV = smem_u32(smem + C::V_OFF);
    const uint32_t sP = smem_u32(smem + C::P_OFF);
    // Base descriptors, built once; each MMA's operand is an offset from them.
    const uint64_t qdesc = smem_desc_sw128(sQ, 16, 1024), pdesc = smem_desc_sw128(sP, 16, 1024);
    const uint64_t kdesc0 = smem_desc_sw128(sK, 16, 1024), vdesc0 = smem_desc_sw128(sV, 16, 1024);
    const uint32_t colS[2] = {C::S_COL0, C::S_COL1};
    const uint32_t colO[2] = {C::O_COL0, C::O_COL1};
    bool ok = wait_warp(&bars->q_full, 0, wc);
    for (int j = 0; ok && j <= nkv_max; ++j) {
      const int sl = j % C::NS;                        // K_j and V_{j-1}
      const uint64_t kdesc = desc_add(kdesc0, sl * C::TILE), vdesc = desc_add(vdesc0, sl * C::TILE);
      // TMA data needs no tcgen05 fence: the MMAs read it once the
      // transaction count of the slot's barrier has completed.
      if (!(ok = wait_warp(&bars->kv_full[sl], (j / C::NS) & 1, wc))) break;
      // S_t(j) first, each once the softmax has read S_t(j - 1) ...
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int jl = j - k0[t];                      // tile t's local step
        if (jl >= 0 && jl < nkv[t]) {
          if (jl >= 1) {
            if (!(ok = wait_warp(&bars->s_free[t], (jl - 1) & 1, wc))) break;
            tc_fence_after();
          }
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)             // 32 head dims per MMA
              mma_ss_f8(tmem + colS[t], desc_add(qdesc, t * C::TILE + kk * 32), desc_add(kdesc, kk * 32), IDESC,
                        kk > 0 ? 1u : 0u);
            mma_commit(&bars->s_full[t]);
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      // ... then PV_t(j - 1) once its P is in shared memory
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int jl = j - 1 - k0[t];
        if (jl >= 0 && jl < nkv[t]) {
          const int bf = jl & 1;
          if (!(ok = wait_warp(&bars->p_full[t][bf], (jl >> 1) & 1, wc))) break;
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)             // 32 keys per MMA
              mma_ss_f8(tmem + colO[t], desc_add(pdesc, (2 * t + bf) * C::TILE + kk * 32), desc_add(vdesc, kk * 32),
                        IDESC, (jl > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&bars->pv_done[t][bf]);
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(&bars->kv_empty[sl]);
      __syncwarp();
    }
    if (lane == 0) mma_commit(&bars->o_done);
    __syncwarp();
    wait_warp_drain(&bars->o_done, 0);
  } else {
    // ------------------------------------------------------------- softmax
    const int t = warp >> 2;
    // this tile's step range as scalars (a runtime index into the arrays
    // would put them in local memory)
    const int nkv_t = t ? nkv[1] : nkv[0];
    const int k0_t = t ? k0[1] : k0[0];
    const int q4 = warp & 3;
    const int rr = 32 * q4 + lane;                     // row within the tile
    const int row = m0 + 128 * t + rr;                 // row within the sequence
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q4) << 16);
    const uint32_t tS = lane_base + (t ? C::S_COL1 : C::S_COL0);
    const uint32_t tO = lane_base + (t ? C::O_COL1 : C::O_COL0);
    uint8_t* prow0 = smem + C::P_OFF + 2 * t * C::TILE + rr * 128;   // buffer 0; buffer 1 is + TILE
    const float vmax = __ldg(p.v_smax + kvh);
    // (a CTA without a second tile reads no scale for it)
    const float sq = nkv_t > 0 ? __ldg(p.q_scale + (long long)h * nbt + (long long)b * p.nblk + 2 * qb + t) : 1.f;
    const float c2q = p.scale_log2 * sq * (1.0f / kD);
    float slope2 = 0.f;
    if (ALIBI) slope2 = __ldg(p.alibi + h) * kLog2e;
    float m_ref = -INFINITY;
    float l = 0.f;     // sum of P (exact): gives the LSE
    float lr = 0.f;    // sum of the rounded P / r: the weights the P V product used
    bool ok = true;
    for (int j = 0; j < nkv_t; ++j) {
      if (!(ok = wait_warp(&bars->s_full[t], j & 1, wc))) break;
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
      // S_t(j) is in registers: the tensor cores may write S_t(j + 1)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free[t]);
      // P buffer j % 2 was last read by PV_t(j - 2)
      uint8_t* prow = prow0 + (j & 1) * C::TILE;
      if (j >= 2) {
        if (!(ok = wait_warp(&bars->pv_done[t][j & 1], ((j - 2) >> 1) & 1, wc))) break;
      }
      const int kt = kvj(k0_t + j);
      const int n0 = 128 * kt;
      const long long blk = (long long)kvh * nbt + (long long)b * p.nblk + kt;
      const float c2 = c2q * __ldg(p.k_scale + blk);
      const float sv = __ldg(p.v_scale + blk);
      const float inv_rj = vmax / sv;                  // 1 / r(j), r(j) <= 1
      const float lg_rj = lg2_approx(sv) - lg2_approx(vmax);   // log2 r(j), folded into the bias
      const int r0 = m0 + 128 * t;
      const bool need_mask = (CAUSAL && n0 + 127 > r0) || (BAND && n0 < r0 + 127 - W) || (n0 + 128 > L);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int key = n0 + c;
          if (key >= L || (CAUSAL && key > row) || (BAND && key < row - W)) s[c] = __float_as_uint(-INFINITY);
        }
      }
      const float base = ALIBI ? slope2 * (float)(n0 - row) : 0.f;
      const uint64_t c2p = f2(c2, c2);
      // P = 2^(x - mb) (exact sum ts), P r -> e4m3 codes to shared memory
      // (row rr, 16-byte chunks swizzled by rr & 7); tsr sums the rounded
      // values the product sees
      // P' = 2^(x - mb + log2 r) = P r is computed directly (exact sum ts of P
      // from it), rounded to e4m3 and stored to shared memory (row rr, 16-byte
      // chunks swizzled by rr & 7); tsr sums the rounded values / r, the
      // weights the product sees (per 16-key chunk in f16x2, where e4m3
      // values and their small sums are exact or within 2^-11).
      auto exp_pass = [&](float mb, float& ts, float& tsr) {
        const float off = lg_rj - mb;
        const uint64_t nmb = f2(off, off);
        const uint64_t step = f2(2.f * slope2, 2.f * slope2);
        uint64_t acc[2] = {0, 0}, accr = 0;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {               // 16 keys per chunk
          uint64_t bm = ALIBI ? f2(fmaf(slope2, (float)(16 * ch), base + off),
                                   fmaf(slope2, (float)(16 * ch + 1), base + off))
                              : nmb;
          uint32_t pk[4];
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {             // 4 keys per 32-bit word
            uint32_t w = 0;
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
              const int cc = 16 * ch + 4 * c4 + 2 * hlf;
              const uint64_t xy = f2(__uint_as_float(s[cc]), __uint_as_float(s[cc + 1]));
              const uint64_t e = ffma2(xy, c2p, bm);
              if (ALIBI) bm = fadd2(bm, step);
              float e0, e1;
              f2split(e, e0, e1);
              const float p0 = ex2_approx(e0);
              const float p1 = ex2_approx(e1);
              acc[hlf] = fadd2(acc[hlf], f2(p0, p1));
              w |= e4m3x2(p0, p1) << (16 * hlf);
            }
            pk[c4] = w;
          }
          *reinterpret_cast<uint4*>(prow + ((ch ^ (rr & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          const uint32_t h = hadd2(hadd2(e4m3x4_sum_h2(pk[0]), e4m3x4_sum_h2(pk[1])),
                                   hadd2(e4m3x4_sum_h2(pk[2]), e4m3x4_sum_h2(pk[3])));
          accr = fadd2(accr, h2_to_f2(h));
        }
        float a0, a1, b0, b1;
        f2split(fadd2(acc[0], acc[1]), a0, a1);
        f2split(accr, b0, b1);
        ts = (a0 + a1) * inv_rj;
        tsr = (b0 + b1) * inv_rj;
      };
      float ts = 0.f, tsr = 0.f;
      bool full = __any_sync(0xffffffffu, m_ref == -INFINITY);
      bool spec_over = false;
      if (!full) {
        exp_pass(m_ref, ts, tsr);
        spec_over = !(ts <= kSpecSum);
        full = __any_sync(0xffffffffu, spec_over);
      }
      if (full) {
        float mx[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) mx[i] = -INFINITY;
        if (ALIBI) {
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
        // raise past tau, or when this row's speculative sum overflowed
        const bool raise = xmax > m_ref + kTau || spec_over;
        const float m_new = raise ? xmax : m_ref;
        const float alpha = raise ? ex2_approx(m_ref - m_new) : 1.f;
        l *= alpha;
        lr *= alpha;
        if (j > 0 && __any_sync(0xffffffffu, raise)) {
          // O must hold PV_t(j - 1) before it is rescaled
          if (!(ok = wait_warp(&bars->pv_done[t][(j - 1) & 1], ((j - 1) >> 1) & 1, wc))) break;
          tc_fence_after();
#pragma unroll 1
          for (int cb = 0; cb < kD; cb += 16) {
            uint32_t o[16];
            tmem_ld16(tO + cb, o);
            tmem_wait_ld();
            reg_fence16(o);
#pragma unroll
            for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tmem_st16(tO + cb, o);
          }
        }
        m_ref = m_new;
        exp_pass(m_ref == -INFINITY ? 0.f : m_ref, ts, tsr);
      }
      l += ts;
      lr += tsr;
      tmem_wait_st();
      fence_proxy_async_smem();                       // P codes visible to the tensor cores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[t][j & 1]);
    }
    // ------------------------------------------------------------ epilogue
    // O and LSE as in the bf16 forward: a tile whose 128 rows all lie in the
    // sequence is staged in the K/V slots in the TMA box layout and written
    // by TMA stores; a tile crossing the sequence end keeps per-thread
    // stores of its valid rows.
    if (nkv_t > 0) {                          // uniform over the tile's warps
      if (ok) ok = wait_warp(&bars->o_done, 0, wc);
      const bool full_tile = m0 + 128 * t + 128 <= L;
      const int r = 32 * q4 + lane;            // row within the tile
      const int esz = p.o_f32 ? 4 : 2;
      uint8_t* stg = smem + C::K_OFF + t * (128 * kD * 4);
      const bool valid = row < L;
      const float inv = lr > 0.f ? vmax / lr : 0.f;
      const long long tok = seq0 + row;
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int cb = 0; cb < kD; cb += 32) {
          uint32_t o[32];
          tmem_ld32(tO + cb, o);
          tmem_wait_ld();
          reg_fence32(o);
          if (p.o_f32) {
            float4 v[8];
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              v[v4] = make_float4(__uint_as_float(o[4 * v4]) * inv, __uint_as_float(o[4 * v4 + 1]) * inv,
                                  __uint_as_float(o[4 * v4 + 2]) * inv, __uint_as_float(o[4 * v4 + 3]) * inv);
            if (full_tile) {
              uint8_t* rowp = stg + (cb / 32) * 16384 + r * 128;
#pragma unroll
              for (int cc = 0; cc < 8; ++cc) *reinterpret_cast<float4*>(rowp + ((cc ^ (r & 7)) << 4)) = v[cc];
            } else if (valid) {
              float* O = static_cast<float*>(p.o) + (tok * p.Hq + h) * kD + cb;
#pragma unroll
              for (int v4 = 0; v4 < 8; ++v4) reinterpret_cast<float4*>(O)[v4] = v[v4];
            }
          } else {
            uint32_t pkd[16];
#pragma unroll
            for (int c = 0; c < 16; ++c)
              pkd[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv);
            if (full_tile) {
              uint8_t* rowp = stg + (cb / 64) * 16384 + r * 128;
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                *reinterpret_cast<uint4*>(rowp + ((((cb % 64) / 8 + cc) ^ (r & 7)) << 4)) =
                    make_uint4(pkd[4 * cc], pkd[4 * cc + 1], pkd[4 * cc + 2], pkd[4 * cc + 3]);
            } else if (valid) {
              __nv_bfloat16* O = static_cast<__nv_bfloat16*>(p.o) + (tok * p.Hq + h) * kD + cb;
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4)
                reinterpret_cast<uint4*>(O)[v4] = make_uint4(pkd[4 * v4], pkd[4 * v4 + 1], pkd[4 * v4 + 2], pkd[4 * v4 + 3]);
            }
          }
        }
        if (valid)
          p.lse[(long long)h * p.T + tok] = l > 0.f ? (m_ref + lg2_approx(l)) * kLn2 : -INFINITY;
      }
      if (full_tile) {
        // Every warp of the tile reaches this barrier (also after an abort);
        // the stores go out only if all four staged their rows.
        fence_proxy_async_smem();
        const bool any_bad = named_bar_any(1 + t, 128, !ok);
        if (!any_bad && q4 == 0 && lane == 0) {
          const int boxes = (kD * esz) / 128;
          for (int bx = 0; bx < boxes; ++bx)
            tma_store_3d(&tmO, stg + bx * 16384, bx * (128 / esz), h, (int)(seq0 + m0 + 128 * t));
          bulk_commit_group();
          bulk_wait_group0();                  // shared memory must outlive the stores
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

template <bool CAUSAL, bool ALIBI, bool BAND>
int launch_impl(const AttnParams& p, cudaStream_t stream) {
  auto kern = fwd_fp8_kernel<CAUSAL, ALIBI, BAND>;
  if (const int ea = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), Cfg::SMEM_BYTES)) return ea;
  CUtensorMap tq, tk, tv;
  int r = make_tmap_u8_3d(&tq, p.q, kD, p.Hq, p.T, kD, (long long)kD * p.Hq, 128, 1, 128);
  if (!r) r = make_tmap_u8_3d(&tk, p.k, kD, p.Hkv, p.T, kD, (long long)kD * p.Hkv, 128, 1, 128);
  if (!r) r = make_tmap_u8_3d(&tv, p.v, p.vt_stride, kD, p.Hkv, p.vt_stride, p.vt_stride * kD, 128, 128, 1);
  CUtensorMap to;
  if (!r) r = p.o_f32 ? make_tmap_f32_3d(&to, p.o, kD, p.Hq, p.T, 128) : make_tmap_bf16_3d(&to, p.o, kD, p.Hq, p.T, 128);
  if (r) return r;
  dim3 grid((unsigned)(((p.N + 255) / 256) * p.Hq * p.B));
  kern<<<grid, kThreads, Cfg::SMEM_BYTES, stream>>>(tq, tk, tv, to, p);
  return (int)cudaGetLastError();
}

}  // namespace

int launch_fwd_fp8(const AttnParams& p, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const bool alibi = p.alibi != nullptr;
  if (p.causal && p.window != kNoWindow)
    return alibi ? launch_impl<true, true, true>(p, stream) : launch_impl<true, false, true>(p, stream);
  if (p.causal)
    return alibi ? launch_impl<true, true, false>(p, stream) : launch_impl<true, false, false>(p, stream);
  return alibi ? launch_impl<false, true, false>(p, stream) : launch_impl<false, false, false>(p, stream);
}

}  // namespace fa
