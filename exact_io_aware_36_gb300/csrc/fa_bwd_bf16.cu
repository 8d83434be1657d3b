// fa_bwd_bf16.cu -- tensor-core backward of exact attention for sm_103a.
//
// Method ("FlashAttention: Faster Attention Without Dropping a Single
// Interaction", Key design 3): S and P are recomputed tile by tile from Q, K
// and the saved LSE; D_i = dO_i . O_i replaces the row reduction of P o dP;
// dS = P o (dP - D); dV += P^T dO, dK += dS^T Q, dQ += dS K.  The scale
// factor of S enters dK and dQ once more (chain rule) and is applied at the
// end.
//
// Three kernels on the caller's stream:
//   preprocess  D = rowsum(dO o O) in fp32 ([Hq, T]) and dQacc = 0
//               ([Hq, T, d] fp32, head-major so a query tile is contiguous).
//   dkdv        one persistent CTA per SM takes work items, each a (key tile
//               of 128, kv head, sequence): it loops over the query heads of
//               the kv head's group and over query tiles of 64 (causal: only
//               tiles at or after the key tile), keeping dK and dV in TMEM;
//               each step's dQ contribution is added to dQacc with a bulk
//               fp32 reduction from shared memory.
//   dq_convert  dQ = scale * dQacc -> bf16 [T, Hq, d].
//
// dkdv roles (320 threads):
//   warps 0-3  "compute": one TMEM lane = one key row; recompute
//              P^T = 2^(S^T * scale * log2 e + bias - L2) and
//              dS^T = P^T o (dP^T - D); P^T and dS^T go back to TMEM (bf16)
//              as A operands and dS^T also to shared memory (swizzled) as
//              the B operand of dQ^T.
//   warps 4-7  dQ drain: dQ^T rows (one TMEM lane = one head-dim column)
//              to shared memory, then one bulk reduce-add into dQacc.
//   warp 8     MMA issuer; warp 9 TMA producer (K, V once; Q, dO per step
//              into 3 stages, with that step's L2 = LSE * log2 e and D).
// MMAs per step i (M = 128 keys; queries N = 64):
//   S^T(i) = K Q_i^T and dP^T(i) = V dO_i^T          (SS, both K-major)
//   dV += P^T(i) dO_i and dK += dS^T(i) Q_i           (TS, B MN-major)
//   dQ^T(i) = K^T dS^T(i)                             (SS, A and B MN-major)
// TMEM: dV [0,d), dK [d,2d), S^T buffers at 256/320, dP^T buffers at
// 384/448 (64 columns each, double buffered); dQ^T(i) reuses the dP^T
// buffer of step i once dK(i) has read dS^T(i) from it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "fa_host_util.h"
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 320;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kQStages = 3;
constexpr int kItemSlots = 4;     // ring of work-item indices passed to the roles

template <int D>
struct BwdCfg {
  static constexpr int NB = D / 64;
  static constexpr int KV_BOX = 128 * 64 * 2;     // 128 rows x 64 columns
  static constexpr int KV_TILE = NB * KV_BOX;
  static constexpr int Q_BOX = 64 * 64 * 2;       // 64 rows x 64 columns
  static constexpr int Q_TILE = NB * Q_BOX;
  static constexpr int DS_BYTES = 128 * 64 * 2;   // dS^T: 128 keys x 64 queries
  static constexpr int DQ_BYTES = 64 * D * 4;     // fp32 dQ staging, [64][D]
  static constexpr int SIDE_BYTES = 528;          // L2[64], D[64], slope
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KV_TILE;
  static constexpr int Q_OFF = V_OFF + KV_TILE;
  static constexpr int DO_OFF = Q_OFF + kQStages * Q_TILE;
  static constexpr int DS_OFF = DO_OFF + kQStages * Q_TILE;
  static constexpr int DQ_OFF = DS_OFF + 2 * DS_BYTES;
  static constexpr int SIDE_OFF = DQ_OFF + DQ_BYTES;
  static constexpr int BAR_OFF = SIDE_OFF + kQStages * SIDE_BYTES;
  static constexpr int SMEM_BYTES = BAR_OFF + 256 + 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per block");
  static constexpr uint32_t DV_COL = 0, DK_COL = D;
  static constexpr uint32_t SB_COL0 = 256, PB_COL0 = 384;   // + 64 * buffer
};

struct BwdBars {
  uint64_t kv_full;
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t sdp_full[2];
  uint64_t p_ready[2];       // per step parity: arrivals can never run a phase ahead
  uint64_t dq_full, dq_free, dqs_free, dqs_full, dkdv_done;
  uint64_t acc_free;                     // both epilogues have read dV and dK
  uint64_t item_full[kItemSlots], item_empty[kItemSlots];
  int item_q[kItemSlots];                // work item per slot, -1: no more
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(BwdBars) <= 256, "barrier block");

// Per-step query statistics, written by the producer warp:
//   nL2[q] = -LSE_q * log2(e) - slope2 * q   (-inf for queries past the
//            sequence end, so their P is exactly 0; slope2 = 0 without ALiBi)
//   Dv[q]  = D_q                              (0 past the end)
struct alignas(16) Side {
  float nL2[64];
  float Dv[64];
  float slope2;
};
static_assert(sizeof(Side) == 528, "side buffer stride");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// ----------------------------------------------------------------- preprocess
// D = dO . O in fp32 per (token, query head), and the dQ accumulator row
// zeroed (not in the deterministic backward, which has no accumulator);
// also the dK/dV kernel's work counters.
// A thread takes 8 consecutive elements of a row (16-byte loads), D / 8
// threads share a row, and each thread handles kPreRows rows, their loads
// issued before any arithmetic so that enough bytes are in flight to stream
// at HBM speed.
constexpr int kPreRows = 2;

template <int D>
__device__ __forceinline__ void load8_f32(const void* base, bool f32, long long off, float (&x)[8]) {
  if (f32) {
    const float4* q = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    const float4 a = q[0], b = q[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + off);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const AttnParams p) {
  constexpr int G = D / 8;                       // threads per row
  constexpr int RPB = 256 / G;                   // rows per block and pass
  const int c8 = threadIdx.x % G;
  // The dK/dV kernel's work-item counter and its count of finished CTAs
  // start at zero (that kernel also puts them back to zero when it ends).
  if (blockIdx.x == 0 && threadIdx.x < 2) p.work_ctr[threadIdx.x] = 0;
  const long long rows = p.T * p.Hq;
  float o_v[kPreRows][8], g_v[kPreRows][8];
  long long r[kPreRows];
#pragma unroll
  for (int i = 0; i < kPreRows; ++i) {
    r[i] = ((long long)blockIdx.x * kPreRows + i) * RPB + threadIdx.x / G;
    if (r[i] < rows) {
      load8_f32<D>(p.dO, false, r[i] * D + 8 * c8, g_v[i]);
      load8_f32<D>(p.o, p.o_f32 != 0, r[i] * D + 8 * c8, o_v[i]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) g_v[i][e] = o_v[i][e] = 0.f;
    }
  }
#pragma unroll
  for (int i = 0; i < kPreRows; ++i) {
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc = fmaf(o_v[i][e], g_v[i][e], acc);
#pragma unroll
    for (int s = G / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (r[i] >= rows) continue;
    const long long t = r[i] / p.Hq;
    const int h = (int)(r[i] - t * p.Hq);
    if (c8 == 0) p.D[(long long)h * p.T + t] = acc;
    if (!p.deterministic) {          // the deterministic backward's dQ kernel has no accumulator
      float4* z = reinterpret_cast<float4*>(p.dq_acc + ((long long)h * p.T + t) * D + 8 * c8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// ------------------------------------------------------------ final outputs
// One launch: dq = scale * dQacc -> bf16 [T, Hq, d] and, for split dK/dV
// items (kv_split > 1), dK = scale * the sum of the parts and dV = the sum
// of the parts, added in part order (deterministic), -> bf16 [T, Hkv, d].
// A block takes kCvtRows rows of one tensor: the first n_dq blocks dq (rows
// of one head: contiguous in the accumulator), the rest dK then dV.  D / 8
// threads share a row, 8 elements each, and every thread issues the loads
// of its kCvtRows / (256 / (D / 8)) rows before any store.
constexpr int kCvtRows = 64;

template <int D>
__global__ void __launch_bounds__(256) bwd_convert_kernel(const AttnParams p, int nbh, long long n_dq) {
  constexpr int G = D / 8;                       // threads per row
  constexpr int RB = 256 / G;                    // rows per pass
  constexpr int U = kCvtRows / RB;               // rows per thread
  const int c8 = threadIdx.x % G, rr = threadIdx.x / G;
  const long long blk = blockIdx.x;
  if (blk < n_dq) {
    const int h = (int)(blk / nbh);
    const long long t0 = (blk % nbh) * kCvtRows;
    float4 a[U], b[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long t = t0 + u * RB + rr;
      if (t < p.T) {
        const float4* src = reinterpret_cast<const float4*>(p.dq_acc + ((long long)h * p.T + t) * D + c8 * 8);
        a[u] = src[0];
        b[u] = src[1];
      }
    }
    const float s = p.scale;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long t = t0 + u * RB + rr;
      if (t < p.T)
        reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dq) + (t * p.Hq + h) * D + c8 * 8)[0] =
            make_uint4(pack_bf16x2(a[u].x * s, a[u].y * s), pack_bf16x2(a[u].z * s, a[u].w * s),
                       pack_bf16x2(b[u].x * s, b[u].y * s), pack_bf16x2(b[u].z * s, b[u].w * s));
    }
    return;
  }
  // dK (which 0) or dV (which 1): rows of [T * Hkv]
  const long long R = p.T * p.Hkv;
  const long long nbk = (R + kCvtRows - 1) / kCvtRows;
  const long long b2 = blk - n_dq;
  const int which = (int)(b2 / nbk);
  const long long r0 = (b2 % nbk) * kCvtRows;
  const long long slot = R * D;
  constexpr int kMaxParts = 2;
  float4 x[U][kMaxParts], y[U][kMaxParts];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const long long r = r0 + u * RB + rr;
#pragma unroll
    for (int q = 0; q < kMaxParts; ++q)
      if (r < R && q < p.kv_split) {
        const float4* src = reinterpret_cast<const float4*>(p.dkv_part + (2 * q + which) * slot + r * D + c8 * 8);
        x[u][q] = src[0];
        y[u][q] = src[1];
      }
  }
  const float f = which ? 1.f : p.scale;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const long long r = r0 + u * RB + rr;
    if (r >= R) continue;
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
#pragma unroll
    for (int q = 0; q < kMaxParts; ++q)
      if (q < p.kv_split) {
        v[0] += x[u][q].x; v[1] += x[u][q].y; v[2] += x[u][q].z; v[3] += x[u][q].w;
        v[4] += y[u][q].x; v[5] += y[u][q].y; v[6] += y[u][q].z; v[7] += y[u][q].w;
      }
    reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(which ? p.dv : p.dk) + r * D + c8 * 8)[0] =
        make_uint4(pack_bf16x2(v[0] * f, v[1] * f), pack_bf16x2(v[2] * f, v[3] * f),
                   pack_bf16x2(v[4] * f, v[5] * f), pack_bf16x2(v[6] * f, v[7] * f));
  }
}

// ---------------------------------------------------------------------- dkdv
// Work item w (a key tile of 128 rows of one kv head of one sequence) in
// launch order.  Dense batches: key tile slowest, so with a causal mask the
// first key tiles of every sequence and kv head (they meet the most query
// tiles) are handed out first and the SMs are loaded longest-first.  Packed
// batches hold many sequences of different lengths: there the key tiles of
// one (sequence, kv head) are handed out together instead, so they share
// its Q / dO stream through L2.
struct DkdvItem {
  int g, b, n0;          // kv head, sequence, first key row
  long long seq0;        // first token of the sequence
  int L;                 // sequence length
  int qt0, nqt, n_iter;  // first query tile, query tiles per head, steps
  int h0, part;          // first query head of the item; its part of the group
};

template <bool CAUSAL, bool BAND>
__device__ __forceinline__ bool dkdv_item(const AttnParams& p, int w, DkdvItem& it) {
  const int nkt = (p.N + 127) / 128;
  // With kv_split > 1 the parts of one (key tile, kv head, sequence) are
  // adjacent items: they run at the same time on different SMs and share
  // its K / V through L2.  Part r takes query heads g*group + r*group/split ...
  it.part = w % p.kv_split;
  w /= p.kv_split;
  if (p.cu_seqlens) {
    const int gb = w / nkt;
    it.g = gb % p.Hkv;
    it.b = gb / p.Hkv;
    it.n0 = (w % nkt) * 128;
  } else {
    const int gb = w % (p.Hkv * p.B);
    it.g = gb % p.Hkv;
    it.b = gb / p.Hkv;
    it.n0 = (w / (p.Hkv * p.B)) * 128;
  }
  if (!seq_bounds(p, it.b, &it.seq0, &it.L)) return false;
  // Query tiles that see this key tile: all of them without a mask; under
  // the causal mask those from the diagonal on, and with a sliding window w
  // only those up to query n0 + 127 + w.
  const int nqt_all = (it.L + 63) / 64;
  it.qt0 = CAUSAL ? it.n0 / 64 : 0;
  const int qt_end = BAND ? min(nqt_all, (it.n0 + 127 + p.window) / 64 + 1) : nqt_all;
  it.nqt = qt_end - it.qt0;
  const int heads = p.group / p.kv_split;
  it.h0 = it.g * p.group + it.part * heads;
  it.n_iter = heads * it.nqt;
  return true;
}

// Persistent: one CTA per SM takes work items from a counter in the
// workspace until none are left.  The producer
// fetches an item and passes its index to the other roles through a ring of
// four slots; every ring, barrier and buffer index continues across items
// by a per-CTA step count, so the next item's Q/dO loads, its K/V load and
// its first S/dP products overlap the previous item's last products and its
// dK/dV epilogue.  Extra orderings at an item boundary:
//   - K/V are single-buffered: the producer loads the next item's K/V once
//     dkdv_done says every product of the previous item has completed;
//   - the first dV/dK products of an item overwrite the accumulators, so
//     they wait for acc_free: the compute warps have written the previous
//     item's dV and dK out (both epilogues are theirs, so the dQ drain
//     never waits for the end of an item and keeps pace with the products).
// BAND: causal band (sliding window p.window); only with CAUSAL.
// DQ: also accumulate dQ into the workspace (otherwise the deterministic
// backward's dQ kernel computes it; this kernel then writes dK and dV only).
template <int D, bool CAUSAL, bool ALIBI, bool BAND, bool DQ>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                const AttnParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + C::BAR_OFF);
  Side* side = reinterpret_cast<Side*>(smem + C::SIDE_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nwork = ((p.N + 127) / 128) * p.Hkv * p.B * p.kv_split;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&bars->q_full[s], 33);
      mbar_init(&bars->q_empty[s], 1);
    }
    mbar_init(&bars->sdp_full[0], 1);
    mbar_init(&bars->sdp_full[1], 1);
    mbar_init(&bars->p_ready[0], 4);
    mbar_init(&bars->p_ready[1], 4);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 4);
    mbar_init(&bars->dqs_free, 1);
    mbar_init(&bars->dqs_full, 4);
    mbar_init(&bars->dkdv_done, 1);
    mbar_init(&bars->acc_free, 4);                 // the 4 compute warps
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(&bars->item_full[s], 1);
      mbar_init(&bars->item_empty[s], 9);          // MMA warp + 4 compute + 4 drain warps
    }
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

  // Consumers' view of the item ring: the k-th item's index, or -1 when the
  // CTA is done (also on an abort).
  auto next_item = [&](int k) -> int {
    const int sl = k % kItemSlots;
    if (!wait_warp(&bars->item_full[sl], (k / kItemSlots) & 1, wc)) return -1;
    const int w = bars->item_q[sl];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->item_empty[sl]);
    return w;
  };

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
    }
    __syncwarp();
    bool ok = true;
    int G = 0;            // steps of the items before this one
    int issued = 0;       // steps whose Q/dO loads were issued, over all items
    int kv_loads = 0;     // K/V loads issued
    for (int k = 0;; ++k) {
      // Take the next item that has work (a key tile past a short packed
      // sequence has none); a malformed cu_seqlens is recorded and skipped.
      int w = 0;
      DkdvItem it{};
      if (lane == 0) {
        while (true) {
          w = atomicAdd(p.work_ctr, 1);
          if (w < 0) {                     // counter never zeroed: no item is trusted
            record_status(p.status, FA_ERR_WORKSPACE);
            w = nwork;
          }
          if (w >= nwork) break;
          if (!dkdv_item<CAUSAL, BAND>(p, w, it)) { record_status(p.status, FA_ERR_CU_SEQLENS); continue; }
          if (it.n0 < it.L) break;
        }
      }
      w = __shfl_sync(0xffffffffu, w, 0);
      const int sl = k % kItemSlots;
      if (!(ok = wait_warp(&bars->item_empty[sl], ((k / kItemSlots) & 1) ^ 1, wc))) break;
      if (lane == 0) {
        bars->item_q[sl] = w < nwork ? w : -1;
        mbar_arrive(&bars->item_full[sl]);
      }
      __syncwarp();
      if (w >= nwork) break;
      dkdv_item<CAUSAL, BAND>(p, w, it);
      auto load_step = [&](int i) -> bool {           // Q, dO and the side data of step G + i
        const int s = G + i;
        const int st = s % kQStages;
        if (!wait_warp(&bars->q_empty[st], ((s / kQStages) & 1) ^ 1, wc)) return false;
        const int h = it.h0 + i / it.nqt;
        const int q0 = (it.qt0 + i % it.nqt) * 64;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->q_full[st], 2 * C::Q_TILE);
#pragma unroll
          for (int bx = 0; bx < C::NB; ++bx) {
            tma_load_3d(smem + C::Q_OFF + st * C::Q_TILE + bx * C::Q_BOX, &tmQ, bx * 64, h,
                        (int)(it.seq0 + q0), &bars->q_full[st]);
            tma_load_3d(smem + C::DO_OFF + st * C::Q_TILE + bx * C::Q_BOX, &tmdO, bx * 64, h,
                        (int)(it.seq0 + q0), &bars->q_full[st]);
          }
        }
        Side* sd = side + st;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int qq = lane + 32 * r;
          const bool valid = q0 + qq < it.L;
          const long long idx = (long long)h * p.T + it.seq0 + q0 + qq;
          const float sl2 = ALIBI ? __ldg(p.alibi + h) * kLog2e : 0.f;
          sd->nL2[qq] = valid ? fmaf(-sl2, (float)qq, -__ldg(p.lse + idx) * kLog2e) : -INFINITY;
          sd->Dv[qq] = valid ? __ldg(p.D + idx) : 0.f;
        }
        if (lane == 0) sd->slope2 = ALIBI ? __ldg(p.alibi + h) * kLog2e : 0.f;
        __syncwarp();
        mbar_arrive(&bars->q_full[st]);
        issued = s + 1;
        return true;
      };
      // After the first item, the first two steps' Q/dO need only ring slots
      // the previous item's last products free, while K/V must wait until
      // all of them are done: those two go first.  On the first item K/V go
      // first (the side data of a step waits for its loads of LSE and D).
      const int pre = k > 0 ? min(2, it.n_iter) : 0;
      for (int i = 0; ok && i < pre; ++i) ok = load_step(i);
      if (!ok) break;
      if (k > 0 && !(ok = wait_warp(&bars->dkdv_done, (k - 1) & 1, wc))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->kv_full, 2 * C::KV_TILE);
#pragma unroll
        for (int bx = 0; bx < C::NB; ++bx) {
          tma_load_3d(smem + C::K_OFF + bx * C::KV_BOX, &tmK, bx * 64, it.g, (int)(it.seq0 + it.n0), &bars->kv_full);
          tma_load_3d(smem + C::V_OFF + bx * C::KV_BOX, &tmV, bx * 64, it.g, (int)(it.seq0 + it.n0), &bars->kv_full);
        }
      }
      __syncwarp();
      ++kv_loads;
      for (int i = pre; ok && i < it.n_iter; ++i) ok = load_step(i);
      if (!ok) break;
      G += it.n_iter;
    }
    // Loads in flight must land before this CTA's shared memory goes away.
    if (kv_loads > 0) wait_warp_drain(&bars->kv_full, (kv_loads - 1) & 1);
    for (int s = max(0, issued - kQStages); s < issued; ++s)
      wait_warp_drain(&bars->q_full[s % kQStages], (s / kQStages) & 1);
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t ID_S = idesc_bf16_f32(128, 64, 0, 0);   // S^T, dP^T
    constexpr uint32_t ID_KV = idesc_bf16_f32(128, D, 0, 1);   // dV, dK (A from TMEM)
    constexpr uint32_t ID_DQ = idesc_bf16_f32(128, 64, 1, 1);  // dQ^T
    const uint32_t sK = smem_u32(smem + C::K_OFF);
    const uint32_t sV = smem_u32(smem + C::V_OFF);
    const uint32_t sQ = smem_u32(smem + C::Q_OFF);
    const uint32_t sdO = smem_u32(smem + C::DO_OFF);
    const uint32_t sdS = smem_u32(smem + C::DS_OFF);
    // Base descriptors, built once; each MMA's operand is an offset from them.
    const uint64_t kdesc = smem_desc_sw128(sK, 16, 1024), vdesc = smem_desc_sw128(sV, 16, 1024);
    const uint64_t qdesc0 = smem_desc_sw128(sQ, 16, 1024), odesc0 = smem_desc_sw128(sdO, 16, 1024);
    const uint64_t qmn0 = smem_desc_sw128(sQ, C::Q_BOX, 1024), omn0 = smem_desc_sw128(sdO, C::Q_BOX, 1024);
    const uint64_t kmn = smem_desc_sw128(sK, C::KV_BOX, 1024), dsmn0 = smem_desc_sw128(sdS, C::Q_BOX, 1024);

    // Step s (counted over the CTA's items): S^T(s) and dP^T(s) into buffer
    // s % 2, dQ^T(s) over dP^T(s).  dq_full is one barrier, so dq_full(s)
    // may be committed only once the drain has taken dq_full(s - 1), i.e.
    // once dq_free(s - 1) was waited; dP^T(s) overwrites dQ^T(s - 2), so it
    // waits for dq_free(s - 2).  Inside an item both hold because dP(s + 2)
    // waits for dq_free(s); need_dqf covers the first and last steps of an
    // item.  dqf is the next dq_free phase to wait for.
    int dqf = 0;
    bool ok = true;
    auto need_dqf = [&](int upto) -> bool {      // dq_free(0 .. upto) waited
      if constexpr (!DQ) return true;
      if (dqf > upto) return true;
      do {
        if (!wait_warp(&bars->dq_free, dqf & 1, wc)) return false;
      } while (++dqf <= upto);
      tc_fence_after();
      return true;
    };
    auto issue_s = [&](int s) {
      const uint64_t qd = desc_add(qdesc0, (s % kQStages) * C::Q_TILE);
      const uint32_t dcol = C::SB_COL0 + 64 * (uint32_t)(s & 1);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(tmem + dcol, desc_add(kdesc, (kk >> 2) * C::KV_BOX + (kk & 3) * 32),
               desc_add(qd, (kk >> 2) * C::Q_BOX + (kk & 3) * 32), ID_S, kk > 0 ? 1u : 0u);
    };
    auto issue_dp = [&](int s) {
      const uint64_t od = desc_add(odesc0, (s % kQStages) * C::Q_TILE);
      const uint32_t dcol = C::PB_COL0 + 64 * (uint32_t)(s & 1);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(tmem + dcol, desc_add(vdesc, (kk >> 2) * C::KV_BOX + (kk & 3) * 32),
               desc_add(od, (kk >> 2) * C::Q_BOX + (kk & 3) * 32), ID_S, kk > 0 ? 1u : 0u);
    };

    int G = 0;
    int k = 0;
    for (;; ++k) {
      const int w = next_item(k);
      if (w < 0) break;
      DkdvItem it{};
      dkdv_item<CAUSAL, BAND>(p, w, it);
      const int G_end = G + it.n_iter;
      if (!(ok = wait_warp(&bars->kv_full, k & 1, wc))) break;
      // S/dP of the item's first two steps (Q/dO by TMA need no tcgen05
      // fence once the stage's transaction count has completed)
      for (int s = G; ok && s < G + 2 && s < G_end; ++s) {
        if (!(ok = wait_warp(&bars->q_full[s % kQStages], (s / kQStages) & 1, wc))) break;
        if (lane == 0) issue_s(s);
        __syncwarp();
        if (s >= 2 && !(ok = need_dqf(s - 2))) break;
        if (lane == 0) {
          issue_dp(s);
          mma_commit(&bars->sdp_full[s & 1]);
        }
        __syncwarp();
      }
      if (!ok) break;
      // The item's first dV/dK products overwrite the accumulators the
      // previous item's epilogues read.
      if (k > 0) {
        if (!(ok = wait_warp(&bars->acc_free, (k - 1) & 1, wc))) break;
        tc_fence_after();
      }
      for (int s = G; s < G_end; ++s) {
        const int st = s % kQStages;
        const uint32_t buf = (uint32_t)(s & 1);
        if (!(ok = wait_warp(&bars->p_ready[buf], (s >> 1) & 1, wc))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint64_t od = desc_add(omn0, st * C::Q_TILE);
          const uint64_t qd = desc_add(qmn0, st * C::Q_TILE);
          const uint32_t acc0 = s > G ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)   // dV += P^T dO   (K = 64 queries)
            mma_ts(tmem + C::DV_COL, tmem + C::SB_COL0 + 64 * buf + 8 * kk, desc_add(od, kk * 2048), ID_KV,
                   kk > 0 ? 1u : acc0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)   // dK += dS^T Q
            mma_ts(tmem + C::DK_COL, tmem + C::PB_COL0 + 64 * buf + 8 * kk, desc_add(qd, kk * 2048), ID_KV,
                   kk > 0 ? 1u : acc0);
          mma_commit(&bars->q_empty[st]);
        }
        __syncwarp();
        if (DQ) {
          // the item's first and last steps: dq_free(s - 1) may be pending
          if ((s == G || s + 1 == G_end) && s >= 1 && !(ok = need_dqf(s - 1))) break;
          if (lane == 0) {
            const uint64_t dsd = desc_add(dsmn0, buf * C::DS_BYTES);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)   // dQ^T = K^T dS^T   (K = 128 keys)
              mma_ss(tmem + C::PB_COL0 + 64 * buf, desc_add(kmn, kk * 2048), desc_add(dsd, kk * 2048), ID_DQ,
                     kk > 0 ? 1u : 0u);
            mma_commit(&bars->dq_full);
          }
          __syncwarp();
        }
        // S/dP two steps ahead, within the item (the next item's first two
        // need its K/V, loaded once this item's products are done).
        const int nx = s + 2;
        if (nx < G_end) {
          if (!(ok = wait_warp(&bars->q_full[nx % kQStages], (nx / kQStages) & 1, wc))) break;
          if (lane == 0) issue_s(nx);
          __syncwarp();
          // dP(nx) reuses the columns of dQ^T(s) (DQ) or of dS^T(s), which
          // the dK(s) MMA issued above reads first (MMAs run in issue order)
          if (DQ) {
            if (!(ok = wait_warp(&bars->dq_free, s & 1, wc))) break;
            dqf = s + 1;
            tc_fence_after();
          }
          if (lane == 0) {
            issue_dp(nx);
            mma_commit(&bars->sdp_full[buf]);
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(&bars->dkdv_done);
      __syncwarp();
      G = G_end;
    }
    // Tensor-core work must be finished before the TMEM is released; after
    // an abort in the middle of an item, one more commit covers what it
    // issued.
    int commits = k;
    if (!ok) {
      if (lane == 0) mma_commit(&bars->dkdv_done);
      __syncwarp();
      ++commits;
    }
    if (commits > 0) wait_warp_drain(&bars->dkdv_done, (commits - 1) & 1);
  } else if (warp < 4) {
    // ------------------------------------------------------------- compute
    const int kr = 32 * warp + lane;          // key row within the tile
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
    const float c2 = p.scale_log2;
    bool ok = true;
    int G = 0;
    for (int k = 0; ok; ++k) {
      const int w = next_item(k);
      if (w < 0) break;
      DkdvItem itm{};
      dkdv_item<CAUSAL, BAND>(p, w, itm);
      const int n0 = itm.n0, L = itm.L, nqt = itm.nqt;
      const int key = n0 + kr;
      const bool key_ok = key < L;
      for (int i = 0; i < itm.n_iter; ++i) {
        const int s = G + i;
        const int st = s % kQStages;
        const int buf = s & 1;
        const int q0 = (itm.qt0 + i % nqt) * 64;
        if (!(ok = wait_warp(&bars->sdp_full[buf], (s >> 1) & 1, wc))) break;
        tc_fence_after();
        const Side* sd = side + st;
        const bool need_mask = (CAUSAL && q0 < n0 + 127) || (BAND && q0 + 63 > n0 + p.window) || !key_ok;
        // x = S^T * scale * log2(e) + slope2 * (key - q0) + nL2[q]: the bias
        // term is split into a per-thread part (key - q0, exact integer) and a
        // per-query part folded into nL2 by the producer.
        const float kb = ALIBI ? sd->slope2 * (float)(key - q0) : 0.f;
        const uint64_t c2p = f2(c2, c2);
        const uint64_t kbp = f2(kb, kb);
        uint8_t* dsrow = smem + C::DS_OFF + buf * C::DS_BYTES + kr * 128;
        const uint32_t tSb = lane_base + C::SB_COL0 + 64 * buf;
        const uint32_t tPb = lane_base + C::PB_COL0 + 64 * buf;
  #pragma unroll 1
        for (int half = 0; half < 2; ++half) {    // 32 queries at a time
          uint32_t sv[32], dp[32];
          tmem_ld32(tSb + 32 * half, sv);
          tmem_ld32(tPb + 32 * half, dp);
          tmem_wait_ld();
          reg_fence32(sv);
          reg_fence32(dp);
          uint32_t pk[16], dk[16];
          const float4* nl4 = reinterpret_cast<const float4*>(sd->nL2 + 32 * half);
          const float4* dd4 = reinterpret_cast<const float4*>(sd->Dv + 32 * half);
  #pragma unroll
          for (int g4 = 0; g4 < 8; ++g4) {        // 4 queries per group
            const float4 nl = nl4[g4];
            const float4 dd = dd4[g4];
  #pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
              const int ql = 4 * g4 + 2 * pr;     // query within the half
              uint64_t bias = pr ? f2(nl.z, nl.w) : f2(nl.x, nl.y);
              if (ALIBI) bias = fadd2(bias, kbp);
              float x0, x1;
              f2split(ffma2(f2(__uint_as_float(sv[ql]), __uint_as_float(sv[ql + 1])), c2p, bias), x0, x1);
              float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
              if (need_mask) {
                const int q = q0 + 32 * half + ql;
                if (!key_ok || (CAUSAL && key > q) || (BAND && q > key + p.window)) p0 = 0.f;
                if (!key_ok || (CAUSAL && key > q + 1) || (BAND && q + 1 > key + p.window)) p1 = 0.f;
              }
              const uint64_t pp = f2(p0, p1);
              const uint64_t dsd = fmul2(pp, fsub2(f2(__uint_as_float(dp[ql]), __uint_as_float(dp[ql + 1])),
                                                   pr ? f2(dd.z, dd.w) : f2(dd.x, dd.y)));
              float d0, d1;
              f2split(dsd, d0, d1);
              pk[ql / 2] = pack_bf16x2(p0, p1);
              dk[ql / 2] = pack_bf16x2(d0, d1);
            }
          }
          tmem_st16(tSb + 16 * half, pk);          // P^T (bf16) over consumed S^T columns
          tmem_st16(tPb + 16 * half, dk);          // dS^T (bf16) over consumed dP^T columns
          if (DQ) {
  #pragma unroll
            for (int q16 = 0; q16 < 4; ++q16) {    // dS^T row into shared memory (swizzled)
              const int chunk = 4 * half + q16;
              const int phys = chunk ^ (kr & 7);
              *reinterpret_cast<uint4*>(dsrow + phys * 16) =
                  make_uint4(dk[4 * q16], dk[4 * q16 + 1], dk[4 * q16 + 2], dk[4 * q16 + 3]);
            }
          }
        }
        if (DQ) fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_ready[buf]);
      }
      if (!ok) break;
      // dV and dK epilogues (one key row per thread), then the accumulators
      // are free for the next item
      if (!(ok = wait_warp(&bars->dkdv_done, k & 1, wc))) break;
      tc_fence_after();
      const float sc = p.scale;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {        // 0: dV, 1: dK (times the scale)
        const float f = which ? sc : 1.f;
        const long long row = (itm.seq0 + key) * p.Hkv + itm.g;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(which ? p.dk : p.dv) + row * D;
        // split items: this part's fp32 sums go to its own slot, summed in a
        // fixed order by the convert kernel (dK's scale is applied there)
        float* part_dst = p.kv_split > 1
            ? p.dkv_part + ((long long)(itm.part * 2 + (1 - which)) * p.T * p.Hkv + row) * D : nullptr;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(lane_base + (which ? C::DK_COL : C::DV_COL) + c0, r);
          tmem_wait_ld();
          reg_fence32(r);
          if (!key_ok) continue;
          if (part_dst) {
            float4* d4 = reinterpret_cast<float4*>(part_dst + c0);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              d4[v4] = make_float4(__uint_as_float(r[4 * v4]), __uint_as_float(r[4 * v4 + 1]),
                                   __uint_as_float(r[4 * v4 + 2]), __uint_as_float(r[4 * v4 + 3]));
          } else {
            uint32_t pkd[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pkd[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * f, __uint_as_float(r[2 * e + 1]) * f);
            uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) d4[v4] = make_uint4(pkd[4 * v4], pkd[4 * v4 + 1], pkd[4 * v4 + 2], pkd[4 * v4 + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->acc_free);
      G += itm.n_iter;
    }
  } else {
    // ------------------------------------------------------------ dQ drain
    const int q4 = warp & 3;
    const int c = 32 * q4 + lane;             // head-dim column of dQ^T
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q4) << 16);
    float* dqs = reinterpret_cast<float*>(smem + C::DQ_OFF);
    bool ok = true;
    int G = 0;
    for (int k = 0; ok; ++k) {
      const int w = next_item(k);
      if (w < 0) break;
      DkdvItem itm{};
      dkdv_item<CAUSAL, BAND>(p, w, itm);
      for (int i = 0; DQ && i < itm.n_iter; ++i) {
        const int s = G + i;
        const int buf = s & 1;
        const int h = itm.h0 + i / itm.nqt;
        const int q0 = (itm.qt0 + i % itm.nqt) * 64;
        const int nvalid = min(64, itm.L - q0);
        if (!(ok = wait_warp(&bars->dq_full, s & 1, wc))) break;
        tc_fence_after();
        uint32_t r[64];
        tmem_ld32(lane_base + C::PB_COL0 + 64 * buf, r);
        tmem_ld32(lane_base + C::PB_COL0 + 64 * buf + 32, r + 32);
        tmem_wait_ld();
        reg_fence32(r);
        reg_fence32(r + 32);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->dq_free);
        if (!(ok = wait_warp(&bars->dqs_free, (s & 1) ^ 1, wc))) break;
        if (c < D) {
#pragma unroll
          for (int qq = 0; qq < 64; ++qq) dqs[qq * D + c] = __uint_as_float(r[qq]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->dqs_full);
        if (q4 == 0) {
          if (!(ok = wait_warp(&bars->dqs_full, s & 1, wc))) break;
          if (lane == 0) {
            bulk_reduce_add_f32(p.dq_acc + ((long long)h * p.T + itm.seq0 + q0) * D, dqs,
                                (uint32_t)(nvalid * D * 4));
            bulk_commit_group();
            bulk_wait_group_read0();
            mbar_arrive(&bars->dqs_free);
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      G += itm.n_iter;
    }
    // The dQ reductions still in flight must finish before the kernel ends.
    if (DQ && q4 == 0 && lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // The last CTA to finish (all have stopped taking items by then) puts the
  // counters back to zero, so the next launch on this workspace starts
  // from item 0 even without the preprocess.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.work_ctr + 1, 1) == (int)gridDim.x - 1) {
      p.work_ctr[0] = 0;
      p.work_ctr[1] = 0;
    }
  }
}

template <int D, bool CAUSAL, bool ALIBI, bool BAND, bool DQ>
int launch_dkdv(const AttnParams& p, cudaStream_t stream) {
  using C = BwdCfg<D>;
  auto kern = bwd_dkdv_kernel<D, CAUSAL, ALIBI, BAND, DQ>;
  if (const int ea = set_max_dynamic_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES)) return ea;
  CUtensorMap tq, tk, tv, tdo;
  int r = make_tmap_bf16_3d(&tq, p.q, D, p.Hq, p.T, 64);
  if (!r) r = make_tmap_bf16_3d(&tdo, p.dO, D, p.Hq, p.T, 64);
  if (!r) r = make_tmap_bf16_3d(&tk, p.k, D, p.Hkv, p.T, 128);
  if (!r) r = make_tmap_bf16_3d(&tv, p.v, D, p.Hkv, p.T, 128);
  if (r) return r;
  // Persistent: one CTA per SM (at most one per item), items handed out by
  // the workspace counter (zeroed by the preprocess and by the previous
  // launch's last CTA).
  const long long nwork = (long long)((p.N + 127) / 128) * p.Hkv * p.B * p.kv_split;
  int nsm = 0;
  if (const int es = sm_count(&nsm)) return es;
  dim3 grid((unsigned)std::min<long long>(nwork, nsm));
  kern<<<grid, kThreads, C::SMEM_BYTES, stream>>>(tq, tk, tv, tdo, p);
  return (int)cudaGetLastError();
}

template <int D, bool DQ>
int launch_dkdv_masks(const AttnParams& p, cudaStream_t stream) {
  const bool alibi = p.alibi != nullptr;
  if (p.causal && p.window != kNoWindow)
    return alibi ? launch_dkdv<D, true, true, true, DQ>(p, stream) : launch_dkdv<D, true, false, true, DQ>(p, stream);
  if (p.causal)
    return alibi ? launch_dkdv<D, true, true, false, DQ>(p, stream) : launch_dkdv<D, true, false, false, DQ>(p, stream);
  return alibi ? launch_dkdv<D, false, true, false, DQ>(p, stream) : launch_dkdv<D, false, false, false, DQ>(p, stream);
}

template <int D>
int launch_stages(const AttnParams& p, cudaStream_t stream, int stage) {
  const long long rows = p.T * p.Hq;
  if (stage < 0 || stage == 0) {
    const long long per_block = (long long)kPreRows * (256 / (D / 8));
    bwd_preprocess_kernel<D><<<(unsigned)((rows + per_block - 1) / per_block), 256, 0, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
  }
  if (stage < 0 || stage == 1) {
    const int r = p.deterministic ? launch_dkdv_masks<D, false>(p, stream)
                                  : launch_dkdv_masks<D, true>(p, stream);
    if (r) return r;
  }
  if (stage < 0 || stage == 2) {
    // dq (unless deterministic: its own kernel computes it) and the split
    // parts' sum, in one launch
    if (p.kv_split > 2) return (int)cudaErrorInvalidValue;     // the sum reads two parts at most
    const int nbh = (int)((p.T + kCvtRows - 1) / kCvtRows);
    const long long n_dq = p.deterministic ? 0 : (long long)nbh * p.Hq;
    const long long n_kv = p.kv_split > 1 ? 2 * ((p.T * p.Hkv + kCvtRows - 1) / kCvtRows) : 0;
    if (n_dq + n_kv > 0) {
      bwd_convert_kernel<D><<<(unsigned)(n_dq + n_kv), 256, 0, stream>>>(p, nbh, n_dq);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return (int)e;
    }
    if (p.deterministic) return launch_bwd_dq_bf16(p, stream);
  }
  return 0;
}

}  // namespace

int launch_bwd_bf16(const AttnParams& p, void* stream, int stage) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return p.d == 128 ? launch_stages<128>(p, s, stage) : launch_stages<64>(p, s, stage);
}

}  // namespace fa
