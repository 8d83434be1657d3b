// fa_fwd_bf16_block.cu -- tensor-core forward of exact attention for sm_103a,
// one CTA per query block (the forward for long dense sequences; the
// persistent kernel in fa_fwd_bf16.cu takes the others).
//
// Method ("FlashAttention: Faster Attention Without Dropping a Single
// Interaction"): Key design 1 (tiles of Q, K, V staged on chip; S and P never
// leave the SM), Key design 2 (running max m and sum l merged tile by tile,
// the output accumulator rescaled when m grows; FA2's L = m + log l saved per
// row), Key design 4 (FA3-style asynchrony: producer and consumer roles).
//
// GB300 mapping (one CTA per SM, 384 threads, 2 query tiles of 128 rows):
//   warp 9     TMA producer: Q0/Q1 once, then per step j one slot holding
//              K_j and V_{j-1} (128-byte swizzle), with one full and one
//              empty mbarrier per slot.  Step j's products are S_t(j), which
//              reads K_j, and PV_t(j-1), which reads V_{j-1}; both are done
//              when the slot is released, so pairing the two tiles this way
//              holds neither back, and the MMA warp has one wait and one
//              release per step.
//   warp 8     MMA issuer (one lane): S_t = Q_t K_j^T into TMEM (both
//              operands K-major in shared memory), then O_t += P_t V_j with
//              P_t read from TMEM and V_j MN-major in shared memory.
//   warps 0-3  softmax of query tile 0 (one TMEM lane = one query row)
//   warps 4-7  softmax of query tile 1
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
// P_t (bf16, two per 32-bit column) overwrites the first 64 columns of S_t.
// The MMA stream per key tile j is PV0(j-1), S0(j), PV1(j-1), S1(j), so the
// softmax of one tile overlaps the tensor work of the other.
//
// Softmax in base 2: x = s * scale * log2(e) (+ slope * log2(e) * (j - i)),
// p = 2^(x - m_ref).  The reference max m_ref is only raised when a tile's
// max exceeds it by more than kTau = 8 (lazy rescale): the result is the same
// for any reference, and p stays <= 2^8.  When it is raised, the owning
// thread rescales its O row in TMEM; this is safe then because the commit
// that published S_t(j) also covers PV_t(j-1).
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_host_util.h"

namespace fa {
namespace {

constexpr int kThreads = 384;     // warps 10, 11 have no role: they complete warpgroup 2
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
// Register limits per thread after the role split (setmaxnreg): the two
// softmax warpgroups take what warpgroup 2 (producer, MMA issuer, two idle
// warps) gives back from the 168 registers every thread is launched with.
constexpr uint32_t kRegsCtl = 56;
constexpr uint32_t kRegsSoftmax = 224;
static_assert(2 * kRegsSoftmax + kRegsCtl <= 3 * 168, "register split (384 threads)");
constexpr float kTau = 8.0f;
constexpr float kSpecSum = 256.0f;   // 2^kTau

template <int D>
struct FwdCfg {
  static constexpr int NB = D / 64;                 // 64-column boxes per row
  static constexpr int BOX_BYTES = 128 * 64 * 2;    // one 128 x 64 bf16 box
  static constexpr int TILE_BYTES = NB * BOX_BYTES; // one 128 x D tile
  static constexpr int NS = D == 128 ? 2 : 5;      // slots (K_j, V_{j-1})
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + 2 * TILE_BYTES;
  static constexpr int V_OFF = K_OFF + NS * TILE_BYTES;
  static constexpr int BAR_OFF = V_OFF + NS * TILE_BYTES;
  static constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per block");
  // The epilogue stages both tiles' O (fp32 at most) in the K/V slots.
  static_assert(2 * 128 * D * 4 <= BAR_OFF - K_OFF, "O staging must fit the K/V slots");
  static constexpr uint32_t S_COL0 = 0, S_COL1 = 128;
  static constexpr uint32_t O_COL0 = 256, O_COL1 = 256 + D;
};

struct FwdBars {
  uint64_t q_full;
  uint64_t kv_full[8], kv_empty[8];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// BAND: causal band (sliding window p.window); only with CAUSAL.
template <int D, bool CAUSAL, bool ALIBI, bool BAND>
__global__ void __launch_bounds__(kThreads, 1)
fwd_bf16_block_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                const AttnParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + C::BAR_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // 1-D grid, query block slowest: with a causal mask the blocks far down
  // the sequence (most K/V tiles) are all launched first, across every head
  // and sequence, so the SMs are loaded longest-first and the tail is short.
  const int nqb = (p.N + 255) / 256;
  const int hb = (int)(blockIdx.x % (unsigned)(p.Hq * p.B));
  const int qslot = (int)(blockIdx.x / (unsigned)(p.Hq * p.B));
  const int h = hb % p.Hq;
  const int b = hb / p.Hq;
  const int qb = CAUSAL ? nqb - 1 - qslot : qslot;

  long long seq0;
  int L;
  if (p.cu_seqlens) {
    const int c0 = __ldg(p.cu_seqlens + b);
    const int c1 = __ldg(p.cu_seqlens + b + 1);
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
  const int m0 = qb * 256;
  if (m0 >= L) return;                       // uniform: nothing to do
  const bool tile1 = m0 + 128 < L;
  // Query tile t (rows [r0, r0 + 128)) needs kv tiles lo[t] .. hi[t]: all of
  // them without a mask; under the causal mask those up to the diagonal, and
  // with a sliding window w only those from row r0 - w on.
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
  // The K/V stream covers kv tiles lo[0] .. hi[1] (tile 1's range starts and
  // ends no earlier than tile 0's, and the two overlap or touch).  Step k
  // visits kv tile kvj(k).  With ALiBi the tiles go from the diagonal
  // backwards: the positive slope makes scores grow toward the diagonal, so
  // the first tile holds (nearly) the row max and the lazy rescale almost
  // never fires.  Tile t is active on steps [k0[t], k0[t] + nkv[t]).
  const int nkv_max = hi[1] - lo[0] + 1;
  constexpr bool REV = ALIBI;
  auto kvj = [&](int k) { return REV ? hi[1] - k : lo[0] + k; };
  const int k0[2] = {REV ? hi[1] - hi[0] : 0, REV ? 0 : lo[1] - lo[0]};

  // The producer's lane initialises the barriers and starts the Q load and
  // the first slots' K/V loads at once; the TMEM allocation and the CTA-wide
  // sync run while those loads are in flight.
  const int kvh = h / p.group;
  auto issue_slot = [&](int j) {                // step j's slot: K_j and V_{j-1}
    const int sl = j % C::NS;
    const bool has_k = j < nkv_max, has_v = j >= 1;
    mbar_arrive_expect_tx(&bars->kv_full[sl], (has_k + has_v) * C::TILE_BYTES);
#pragma unroll
    for (int bx = 0; bx < C::NB; ++bx) {
      if (has_k)
        tma_load_3d(smem + C::K_OFF + sl * C::TILE_BYTES + bx * C::BOX_BYTES, &tmK, bx * 64, kvh,
                    (int)(seq0 + 128 * kvj(j)), &bars->kv_full[sl]);
      if (has_v)
        tma_load_3d(smem + C::V_OFF + sl * C::TILE_BYTES + bx * C::BOX_BYTES, &tmV, bx * 64, kvh,
                    (int)(seq0 + 128 * kvj(j - 1)), &bars->kv_full[sl]);
    }
  };
  const int early = min(C::NS, nkv_max + 1);    // slots filled before the sync
  if (warp == kLoadWarp && lane == 0) {
    mbar_init(&bars->q_full, 1);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 4);
    }
    mbar_init(&bars->o_done, 1);
    bars->abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    const int ntiles = tile1 ? 2 : 1;
    mbar_arrive_expect_tx(&bars->q_full, ntiles * C::TILE_BYTES);
    for (int t = 0; t < ntiles; ++t)
#pragma unroll
      for (int bx = 0; bx < C::NB; ++bx)
        tma_load_3d(smem + C::Q_OFF + t * C::TILE_BYTES + bx * C::BOX_BYTES, &tmQ, bx * 64, h,
                    (int)(seq0 + m0 + 128 * t), &bars->q_full);
    for (int j = 0; j < early; ++j) issue_slot(j);
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

  // Every wait below is inlined: code under a raised register limit can hold
  // no calls.
  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    regs_lower<kRegsCtl>();
    int issued = early;               // slots whose loads were issued
    for (int j = early; j <= nkv_max; ++j) {
      const int sl = j % C::NS;
      if (!wait_warp_inl(&bars->kv_empty[sl], ((j / C::NS) & 1) ^ 1, wc)) break;
      if (lane == 0) issue_slot(j);
      __syncwarp();
      issued = j + 1;
    }
    // Loads in flight must land before this CTA's shared memory goes away.
    wait_warp_drain(&bars->q_full, 0);
    for (int j = max(0, issued - C::NS); j < issued; ++j)
      wait_warp_drain(&bars->kv_full[j % C::NS], (j / C::NS) & 1);
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
    bool ok = wait_warp_inl(&bars->q_full, 0, wc);
    for (int j = 0; ok && j <= nkv_max; ++j) {
      const int sl = j % C::NS;                       // K_j and V_{j-1}
      const uint64_t kdesc = desc_add(kdesc0, sl * C::TILE_BYTES);
      const uint64_t vdesc = desc_add(vdesc0, sl * C::TILE_BYTES);
      // TMA data needs no tcgen05 fence: the MMAs read it once the
      // transaction count of the slot's barrier has completed.
      if (!(ok = wait_warp_inl(&bars->kv_full[sl], (j / C::NS) & 1, wc))) break;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (j >= 1 && j - 1 >= k0[t] && j - 1 < k0[t] + nkv[t]) {
          if (!(ok = wait_warp_inl(&bars->p_full[t], (j - 1 - k0[t]) & 1, wc))) break;
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < 128 / 16; ++kk)
              mma_ts(tmem + colO[t], tmem + colS[t] + kk * 8, desc_add(vdesc, kk * 2048), IDESC_O,
                     (j - 1 > k0[t] || kk > 0) ? 1u : 0u);
          }
          __syncwarp();
        }
        if (j >= k0[t] && j < k0[t] + nkv[t]) {
          if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
              mma_ss(tmem + colS[t], desc_add(qdesc[t], off), desc_add(kdesc, off), IDESC_S, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bars->s_full[t]);
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
    // Tensor-core work must be finished before the TMEM is released.
    wait_warp_drain(&bars->o_done, 0);
  } else if (warp < 8) {
    // ------------------------------------------------------------- softmax
    regs_raise<kRegsSoftmax>();
    const int t = warp >> 2;
    const int q4 = warp & 3;
    const int row = m0 + 128 * t + 32 * q4 + lane;       // row within the sequence
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q4) << 16);
    const uint32_t tS = lane_base + (t ? C::S_COL1 : C::S_COL0);
    const uint32_t tO = lane_base + (t ? C::O_COL1 : C::O_COL0);
    const float c2 = p.scale_log2;
    float slope2 = 0.f;
    if (ALIBI) slope2 = __ldg(p.alibi + h) * kLog2e;
    float m_ref = -INFINITY;
    float l = 0.f;     // sum of p in fp32: gives the LSE
    float lr = 0.f;    // sum of the bf16-rounded p the PV MMA sees: normalises O
    bool ok = true;
    for (int j = 0; j < nkv[t]; ++j) {        // j: this tile's local step
      if (!(ok = wait_warp_inl(&bars->s_full[t], j & 1, wc))) break;
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
      const int n0 = 128 * kvj(k0[t] + j);
      const int r0 = m0 + 128 * t;
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
      // directly.  If the tile's sum of p is at most 2^tau, no p exceeds 2^tau,
      // i.e. no score exceeds the reference by more than tau, so no raise is
      // due and the pass is exactly what the full path would produce.
      float ts = 0.f, tsr = 0.f;
      bool full = __any_sync(0xffffffffu, m_ref == -INFINITY);
      bool spec_over = false;     // this row's speculative sum exceeded 2^tau
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
        const float alpha = raise ? ex2_approx(m_ref - m_new) : 1.f;
        l *= alpha;
        lr *= alpha;
        if (j > 0 && __any_sync(0xffffffffu, raise)) {
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
        m_ref = m_new;
        exp_pass(m_ref == -INFINITY ? 0.f : m_ref, ts, tsr);
      }
      l += ts;
      lr += tsr;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[t]);
    }
    // ------------------------------------------------------------ epilogue
    // O = acc / l~ per row and LSE.  A tile whose 128 rows all lie in the
    // sequence is staged in shared memory (the K/V slots, free once every
    // product is done) in the TMA box layout (128-byte rows, 16-byte chunks
    // swizzled by row) and written by TMA stores: whole rows at a time
    // instead of 32 scattered 16-byte pieces per warp instruction.  A tile
    // that crosses the sequence end keeps per-thread stores of its valid
    // rows (a box would overwrite the next sequence's rows).
    if (nkv[t] > 0) {                          // uniform over the tile's warps
      if (ok) ok = wait_warp_inl(&bars->o_done, 0, wc);
      const bool full_tile = m0 + 128 * t + 128 <= L;
      const int r = 32 * q4 + lane;            // row within the tile
      const int esz = p.o_f32 ? 4 : 2;
      uint8_t* stg = smem + C::K_OFF + t * (128 * D * 4);
      const bool valid = row < L;
      const float inv = lr > 0.f ? 1.f / lr : 0.f;
      const long long tok = seq0 + row;
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c0, o);
          tmem_wait_ld();
          reg_fence32(o);
          if (p.o_f32) {
            float4 v[8];
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              v[v4] = make_float4(__uint_as_float(o[4 * v4]) * inv, __uint_as_float(o[4 * v4 + 1]) * inv,
                                  __uint_as_float(o[4 * v4 + 2]) * inv, __uint_as_float(o[4 * v4 + 3]) * inv);
            if (full_tile) {                   // box c0 / 32: this row's 128 bytes
              uint8_t* rowp = stg + (c0 / 32) * 16384 + r * 128;
#pragma unroll
              for (int cc = 0; cc < 8; ++cc) *reinterpret_cast<float4*>(rowp + ((cc ^ (r & 7)) << 4)) = v[cc];
            } else if (valid) {
              float* O = static_cast<float*>(p.o) + (tok * p.Hq + h) * D + c0;
#pragma unroll
              for (int v4 = 0; v4 < 8; ++v4) reinterpret_cast<float4*>(O)[v4] = v[v4];
            }
          } else {
            uint32_t pkd[16];
#pragma unroll
            for (int c = 0; c < 16; ++c)
              pkd[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv, __uint_as_float(o[2 * c + 1]) * inv);
            if (full_tile) {                   // box c0 / 64: chunks (c0 % 64) / 8 .. + 3 of this row
              uint8_t* rowp = stg + (c0 / 64) * 16384 + r * 128;
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                *reinterpret_cast<uint4*>(rowp + ((((c0 % 64) / 8 + cc) ^ (r & 7)) << 4)) =
                    make_uint4(pkd[4 * cc], pkd[4 * cc + 1], pkd[4 * cc + 2], pkd[4 * cc + 3]);
            } else if (valid) {
              __nv_bfloat16* O = static_cast<__nv_bfloat16*>(p.o) + (tok * p.Hq + h) * D + c0;
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4)
                reinterpret_cast<uint4*>(O)[v4] =
                    make_uint4(pkd[4 * v4], pkd[4 * v4 + 1], pkd[4 * v4 + 2], pkd[4 * v4 + 3]);
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
          const int boxes = (D * esz) / 128;
          for (int bx = 0; bx < boxes; ++bx)
            tma_store_3d(&tmO, stg + bx * 16384, bx * (128 / esz), h, (int)(seq0 + m0 + 128 * t));
          bulk_commit_group();
          bulk_wait_group0();                  // shared memory must outlive the stores
        }
      }
    }
  } else {
    regs_lower<kRegsCtl>();             // warps 10, 11: no role
  }
  // Every warpgroup returns to the launch limit before the common tail.
  if (warp < 8) regs_lower<168>();
  else regs_raise<168>();

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL, bool ALIBI, bool BAND>
int launch_impl(const AttnParams& p, cudaStream_t stream) {
  using C = FwdCfg<D>;
  auto kern = fwd_bf16_block_kernel<D, CAUSAL, ALIBI, BAND>;
  if (const int ea = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES)) return ea;
  // The softmax warpgroups' raised register limit draws on what the CTA is
  // launched with (threads x registers per thread); a build that allocated
  // fewer would leave the raise waiting forever, so it is refused here.
  static int regs_ok = -1;
  if (regs_ok < 0) {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, reinterpret_cast<const void*>(kern)) != cudaSuccess)
      return (int)cudaErrorInvalidDeviceFunction;
    regs_ok = a.numRegs >= 168;
  }
  if (!regs_ok) return (int)cudaErrorInvalidConfiguration;
  CUtensorMap tq, tk, tv, to;
  int r = make_tmap_bf16_3d(&tq, p.q, D, p.Hq, p.T, 128);
  if (!r) r = make_tmap_bf16_3d(&tk, p.k, D, p.Hkv, p.T, 128);
  if (!r) r = make_tmap_bf16_3d(&tv, p.v, D, p.Hkv, p.T, 128);
  if (!r) r = p.o_f32 ? make_tmap_f32_3d(&to, p.o, D, p.Hq, p.T, 128) : make_tmap_bf16_3d(&to, p.o, D, p.Hq, p.T, 128);
  if (r) return r;
  dim3 grid((unsigned)(((p.N + 255) / 256) * p.Hq * p.B));
  kern<<<grid, kThreads, C::SMEM_BYTES, stream>>>(tq, tk, tv, to, p);
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

int launch_fwd_bf16_block(const AttnParams& p, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  return p.d == 128 ? launch_masks<128>(p, stream) : launch_masks<64>(p, stream);
}

}  // namespace fa
