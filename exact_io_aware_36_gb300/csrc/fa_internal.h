// fa_internal.h -- parameters shared by the host library and its kernels.
#pragma once
#include <stdint.h>

#include "../../include/fa.h"

namespace fa {

// Limit of every pipeline wait inside a kernel (wall clock, nanoseconds).
// A healthy wait lasts microseconds; the limit only turns a lost arrival
// into an error status instead of a hung GPU.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// log2(e): scores are moved to the base-2 domain so the softmax uses exp2.
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Band width that stands for "no sliding window": larger than any sequence
// (lengths are below 2^30), small enough that key + window cannot overflow.
constexpr int kNoWindow = 1 << 30;

struct AttnParams {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  const void* dO;
  void* dq;
  void* dk;
  void* dv;
  float* D;          // workspace: D_i = dO_i . O_i, [Hq, T]
  float* dq_acc;     // workspace: fp32 dQ accumulator, [Hq, T, d]
  int* work_ctr;     // workspace: dK/dV work-item counter, finished-CTA count
  float* dkv_part;   // workspace (kv_split > 1): fp32 dK / dV partial sums,
                     // [kv_split][2][T, Hkv, d] (part, then 0: dK, 1: dV)
  int kv_split;      // dK/dV work items per (key tile, kv head, sequence):
                     // the group's query heads are split into this many parts
  const int32_t* cu_seqlens;   // [B+1] or nullptr
  const float* alibi;          // [Hq] or nullptr
  unsigned int* status;        // per-device status word
  long long T;
  int B, Hq, Hkv, N, d;
  int group;                   // Hq / Hkv
  int causal;
  int window;                  // causal band: key j visible to query i iff
                               // i - window <= j <= i; kNoWindow when unbanded
  int deterministic;           // backward: dQ by its own kernel, no atomics
  int o_f32;                    // o stored as fp32 (else the input dtype)
  float scale;
  float scale_log2;            // scale * log2(e)
  // FP8 forward: per-block scales ([H, B * nblk]) and the largest V scale
  // of each kv head; q, k are the e4m3 codes, v the transposed V codes
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  const float* v_smax;
  int nblk;
  long long vt_stride;         // bytes per row of the transposed V codes
};

// FP8 quantization (Q' = (Q D) H, K' = (K D) H, V; e4m3 per 128-row block).
struct QuantParams {
  const void* q;               // bf16 [T, Hq, 128]
  const void* k;               // bf16 [T, Hkv, 128]
  const void* v;               // bf16 [T, Hkv, 128]
  const float* signs;          // [128], +-1
  const int32_t* cu_seqlens;
  unsigned int* status;
  uint8_t* q8;
  uint8_t* k8;
  uint8_t* v8t;
  float* q_scale;
  float* k_scale;
  float* v_scale;
  float* v_smax;
  long long T, vt_stride;
  int B, Hq, Hkv, N, nblk;
};

// Decode over a KV cache: the q_len newest tokens of each sequence attend to
// its cache of cache_seqlens[b] tokens.  The keys of one (sequence, kv head)
// are cut into chunks of `chunk`; one block computes the partial (m, l, O) of
// one chunk for the R = group * q_len query rows of that kv head, and a
// combine kernel merges the chunks.
struct DecodeParams {
  const void* q;               // bf16 [B * q_len, Hq, d]
  const void* k;               // bf16 [B, S_max, Hkv, d]
  const void* v;               // bf16 [B, S_max, Hkv, d]
  void* o;                     // [B * q_len, Hq, d], fp32 or bf16
  float* lse;                  // [Hq, B * q_len]
  const int32_t* seqlens;      // [B] or nullptr (every cache holds S_max tokens)
  const float* alibi;          // [Hq] or nullptr
  float* part_o;               // [B, Hkv, nsplit, R, d] fp32: unnormalised partial O
  float* part_ml;              // [B, Hkv, nsplit, R, 3] fp32: partial max (log2 units),
                               // sum of P (exact), sum of P as the PV product used it
  unsigned int* status;
  int B, Hq, Hkv, S_max, q_len, d, group, R;
  int chunk, nsplit;
  int window;                  // kNoWindow when unbanded
  int o_f32;
  float scale, scale_log2;
};

// GB300 has 152 SMs; decode chunks are sized so that a batch of full caches
// gives at least this many (sequence, kv head, chunk) blocks.
constexpr int kDecodeUnitsTarget = 8 * 152;
constexpr int kDecodeMaxRows = 16;

// Keys per decode block: the largest of 128, 256, ..., 4096 that still leaves
// kDecodeUnitsTarget blocks for B caches of S_max tokens.
inline int decode_chunk(int B, int Hkv, int S_max) {
  int c = 128;
  while (c < 4096) {
    const long long n = (long long)B * Hkv * ((S_max + 2 * c - 1) / (2 * c));
    if (n < kDecodeUnitsTarget) break;
    c *= 2;
  }
  return c;
}

// The host-side argument checks of fa_bwd (everything but the workspace), in
// fa_bwd's order.  On FA_OK, *T is the total token count, or 0 when the call
// has nothing to compute.
fa_status bwd_check_args(const void* q, const void* k, const void* v, const void* o,
                         const void* dO, const float* lse, const void* dq, const void* dk,
                         const void* dv, int B, int Hq, int Hkv, int N, int d, float scale,
                         int causal, int window, const int32_t* cu_seqlens,
                         long long total_tokens, fa_dtype dtype, fa_dtype o_dtype,
                         int deterministic, long long* T);

// Launchers (each returns a cudaError_t value as int).
int launch_fwd_fp32(const AttnParams& p, void* stream);
int launch_fwd_bf16(const AttnParams& p, void* stream);             // picks one of:
int launch_fwd_bf16_block(const AttnParams& p, void* stream);       //   one CTA per query block
int launch_fwd_bf16_persistent(const AttnParams& p, void* stream);  //   one CTA per SM
int launch_bwd_bf16(const AttnParams& p, void* stream, int stage);   // stage < 0: all
int launch_bwd_dq_bf16(const AttnParams& p, void* stream);            // deterministic dQ
int launch_decode_bf16(const DecodeParams& p, void* stream);          // split + combine
int launch_fp8_quantize(const QuantParams& p, void* stream);
int launch_fwd_fp8(const AttnParams& p, void* stream);
int launch_selftest_wait(unsigned int* status, unsigned long long limit_ns, void* stream);

#ifdef __CUDACC__
// Start token and length of sequence b; false when cu_seqlens is malformed
// there or the sequence is longer than N.
__device__ __forceinline__ bool seq_bounds(const AttnParams& p, int b, long long* seq0, int* L) {
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
#endif

}  // namespace fa
