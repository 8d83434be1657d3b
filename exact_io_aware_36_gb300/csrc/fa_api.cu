// fa_api.cu -- the C ABI of libfa (declared in include/fa.h): argument
// checks, workspace sizing, the per-device status word and dispatch to the
// kernels.  Every check runs before any launch; nothing here allocates
// device memory.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <functional>
#include <mutex>
#include <queue>
#include <vector>

#include "fa_host_util.h"
#include "fa_internal.h"

namespace {

__device__ unsigned int g_fa_status;   // per-device status word

constexpr int kMaxDevices = 64;

unsigned int* status_ptr() {
  static unsigned int* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned int*>(p);
  }
  return ptrs[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Shared size checks of fa_fwd / fa_bwd.  Fills T.
fa_status check_sizes(int B, int Hq, int Hkv, int N, int d, float scale,
                      const int32_t* cu_seqlens, long long total_tokens, fa_dtype dtype,
                      bool backward, long long* T) {
  if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || total_tokens < 0) return FA_ERR_SHAPE;
  if (Hq % Hkv != 0) return FA_ERR_SHAPE;
  if (dtype != FA_BF16 && dtype != FA_FP32) return FA_ERR_UNSUPPORTED;
  if (backward && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (dtype == FA_BF16 && d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (dtype == FA_FP32 && d > 128) return FA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_UNSUPPORTED;
  if (B > 65535 || Hq > 65535) return FA_ERR_UNSUPPORTED;
  // 1-D grids of (blocks per sequence) x heads x sequences must fit 2^31 - 1
  if ((long long)((N + 127) / 128) * Hq * B >= (1ll << 31)) return FA_ERR_UNSUPPORTED;
  const long long dense = (long long)B * N;
  if (cu_seqlens == nullptr) {
    if (total_tokens != 0 && total_tokens != dense) return FA_ERR_SHAPE;
    *T = dense;
  } else {
    *T = total_tokens;
  }
  // token coordinates are 32-bit in the TMA descriptors and the kernels
  if (*T >= (1ll << 31) || (long long)N >= (1ll << 30)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Window argument -> band width: < 0 means none; a band that reaches back
// over the whole longest sequence (window >= N - 1) masks nothing beyond the
// causal mask, so it is run as unbanded.
int band_width(int window, int N) { return (window < 0 || window >= N - 1) ? fa::kNoWindow : window; }

fa::AttnParams base_params(int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                           int window, const int32_t* cu_seqlens, long long T,
                           const float* alibi) {
  fa::AttnParams p = {};
  p.window = band_width(window, N);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.d = d;
  p.T = T;
  p.group = Hq / Hkv;
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = scale * fa::kLog2e;
  p.cu_seqlens = cu_seqlens;
  p.alibi = alibi;
  return p;
}

}  // namespace

extern "C" {

int fa_version(void) { return 10000; }

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_SHAPE: return "invalid or inconsistent sizes";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration (head dim, dtype or scale)";
    case FA_ERR_ALIGN: return "a bf16 tensor is not 16-byte aligned";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    case FA_ERR_CUDA: return "CUDA runtime or launch error";
    case FA_ERR_DEVICE_TIMEOUT: return "device pipeline wait exceeded its time limit";
    case FA_ERR_CU_SEQLENS: return "cu_seqlens malformed or a sequence longer than N";
  }
  return "unknown status";
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                 int Hkv, int N, int d, float scale, int causal, int window,
                 const int32_t* cu_seqlens, long long total_tokens, const float* alibi_slopes,
                 fa_dtype dtype, fa_dtype o_dtype, void* stream) {
  long long T = 0;
  fa_status st = check_sizes(B, Hq, Hkv, N, d, scale, cu_seqlens, total_tokens, dtype, false, &T);
  if (st != FA_OK) return st;
  if (window >= 0 && !causal) return FA_ERR_UNSUPPORTED;
  if (o_dtype != FA_FP32 && !(o_dtype == FA_BF16 && dtype == FA_BF16)) return FA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  if (dtype == FA_BF16 && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)))
    return FA_ERR_ALIGN;
  if (dtype == FA_FP32 && ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                            reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o)) & 3u))
    return FA_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_ALIGN;
  if (T == 0 || B == 0 || N == 0) return FA_OK;
  fa::AttnParams p = base_params(B, Hq, Hkv, N, d, scale, causal, window, cu_seqlens, T,
                                 alibi_slopes);
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  p.o_f32 = o_dtype == FA_FP32;
  p.status = status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  const int e = dtype == FA_FP32 ? fa::launch_fwd_fp32(p, stream) : fa::launch_fwd_bf16(p, stream);
  return e == 0 ? FA_OK : FA_ERR_CUDA;
}

size_t fa_bwd_workspace_size(int B, int Hq, int N, int d, long long total_tokens) {
  if (B < 0 || Hq <= 0 || N < 0 || d <= 0 || total_tokens < 0) return 0;
  const long long T = total_tokens > 0 ? total_tokens : (long long)B * N;
  return round256((size_t)Hq * T * sizeof(float)) + round256((size_t)Hq * T * d * sizeof(float)) + 256;
}

// Largest number of parts the dK/dV work of a GQA group may be split into:
// 2 when the group splits evenly, else 1 (no split).  (Four parts were
// measured no faster than two on the GQA workload, B=2 Hq=32 Hkv=4 N=8192,
// while their sum costs twice as much.)
static int gqa_split_max(int Hq, int Hkv) {
  const int group = Hkv > 0 ? Hq / Hkv : 0;
  return (group >= 2 && group % 2 == 0) ? 2 : 1;
}

// How many parts to split each dense batch's dK/dV work items into (1 or
// 2).  The kernel's SMs take items largest first as they finish; with few,
// large items (a long causal sequence and few kv heads) the last ones leave
// SMs idle.  For each allowed split this simulates that list schedule over
// the items' step counts (a step is 64 queries of one head against the key
// tile), estimates the time as its longest SM in steps, plus the stage that
// adds the parts up (reads 2 x split fp32 tensors [T, Hkv, d]), and keeps
// the fastest.  Results are cached per shape.  Packed batches, whose
// lengths the host does not see, are not split.
static int dkdv_split(int B, int Hq, int Hkv, int N, int d, int causal, int window) {
  const int smax = gqa_split_max(Hq, Hkv);
  if (smax == 1) return 1;
  int nsm = 0;
  if (fa::sm_count(&nsm) != 0 || nsm <= 0) return 1;
  struct Entry { int B, Hq, Hkv, N, d, causal, window, nsm, split; };
  static Entry cache[16];
  static int ncache = 0;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < ncache; ++i) {
      const Entry& e = cache[i];
      if (e.B == B && e.Hq == Hq && e.Hkv == Hkv && e.N == N && e.d == d && e.causal == causal &&
          e.window == window && e.nsm == nsm)
        return e.split;
    }
  }
  const int group = Hq / Hkv;
  const long long nkt = (N + 127) / 128, nqt_all = (N + 63) / 64;
  std::vector<long long> per_kt((size_t)nkt);
  for (long long kt = 0; kt < nkt; ++kt) {
    const long long qt0 = causal ? 2 * kt : 0;
    long long qt_end = nqt_all;
    if (causal && window != fa::kNoWindow)
      qt_end = std::min(nqt_all, (kt * 128 + 127 + window) / 64 + 1);
    per_kt[(size_t)kt] = std::max(0ll, qt_end - qt0);
  }
  std::sort(per_kt.begin(), per_kt.end(), std::greater<long long>());
  const double step_s = 1.6e-6 * d / 128.0;         // measured per-step time of one SM
  const double bytes_per_s = 6.0e12;                // HBM rate of the adding stage
  int best = 1;
  double best_t = 0.0;
  for (int split = 1; split <= smax; split *= 2) {
    std::priority_queue<long long, std::vector<long long>, std::greater<long long>> load;
    for (int i = 0; i < nsm; ++i) load.push(0);
    const long long per_item = (long long)B * Hkv * split;
    for (long long steps : per_kt)
      for (long long i = 0; i < per_item; ++i) {
        const long long x = load.top();
        load.pop();
        load.push(x + steps * group / split);
      }
    long long makespan = 0;
    while (!load.empty()) { makespan = load.top(); load.pop(); }
    double t = makespan * step_s;
    if (split > 1) t += (double)split * 2 * B * N * Hkv * d * 4 / bytes_per_s;
    if (split == 1 || t < best_t) {
      best = split;
      best_t = t;
    }
  }
  std::lock_guard<std::mutex> lock(mu);
  cache[ncache < 16 ? ncache++ : (B + N) % 16] = Entry{B, Hq, Hkv, N, d, causal, window, nsm, best};
  return best;
}

size_t fa_bwd_workspace_size_gqa(int B, int Hq, int Hkv, int N, int d, long long total_tokens) {
  const size_t base = fa_bwd_workspace_size(B, Hq, N, d, total_tokens);
  if (base == 0 || Hkv <= 0 || Hq % Hkv != 0) return 0;
  const int split = gqa_split_max(Hq, Hkv);
  if (split == 1) return base;
  const long long T = total_tokens > 0 ? total_tokens : (long long)B * N;
  return base + round256((size_t)split * 2 * T * Hkv * d * sizeof(float));
}

}  // extern "C"

namespace fa {

fa_status bwd_check_args(const void* q, const void* k, const void* v, const void* o,
                         const void* dO, const float* lse, const void* dq, const void* dk,
                         const void* dv, int B, int Hq, int Hkv, int N, int d, float scale,
                         int causal, int window, const int32_t* cu_seqlens,
                         long long total_tokens, fa_dtype dtype, fa_dtype o_dtype,
                         int deterministic, long long* T) {
  fa_status st = check_sizes(B, Hq, Hkv, N, d, scale, cu_seqlens, total_tokens, dtype, true, T);
  if (st != FA_OK) return st;
  if (o_dtype != FA_FP32 && o_dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (window >= 0 && !causal) return FA_ERR_UNSUPPORTED;
  if (deterministic != 0 && deterministic != 1) return FA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(lse))
    return FA_ERR_ALIGN;
  if (B == 0 || N == 0) *T = 0;
  return FA_OK;
}

}  // namespace fa

extern "C" {

static fa_status bwd_impl(int stage, const void* q, const void* k, const void* v, const void* o,
                          const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                          int Hq, int Hkv, int N, int d, float scale, int causal, int window,
                          const int32_t* cu_seqlens, long long total_tokens,
                          const float* alibi_slopes, fa_dtype dtype, fa_dtype o_dtype,
                          int deterministic, void* workspace, size_t workspace_bytes,
                          void* stream) {
  if (stage < -1 || stage > 2) return FA_ERR_UNSUPPORTED;
  long long T = 0;
  fa_status st = fa::bwd_check_args(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale,
                                    causal, window, cu_seqlens, total_tokens, dtype, o_dtype,
                                    deterministic, &T);
  if (st != FA_OK) return st;
  if (T == 0) return FA_OK;
  const size_t need = fa_bwd_workspace_size(B, Hq, N, d, T);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_ALIGN;
  fa::AttnParams p = base_params(B, Hq, Hkv, N, d, scale, causal, window, cu_seqlens, T,
                                 alibi_slopes);
  p.deterministic = deterministic;
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = const_cast<void*>(o);
  p.lse = const_cast<float*>(lse);
  p.o_f32 = o_dtype == FA_FP32;
  p.dO = dO;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.D = static_cast<float*>(workspace);
  p.dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                      round256((size_t)Hq * T * sizeof(float)));
  p.work_ctr = reinterpret_cast<int*>(static_cast<char*>(workspace) + round256((size_t)Hq * T * sizeof(float)) +
                                      round256((size_t)Hq * T * d * sizeof(float)));
  // A workspace of fa_bwd_workspace_size_gqa bytes also holds per-part dK /
  // dV sums, which lets the dK/dV kernel split each GQA group's work.
  p.kv_split = 1;
  if (!cu_seqlens && gqa_split_max(Hq, Hkv) > 1 &&
      workspace_bytes >= fa_bwd_workspace_size_gqa(B, Hq, Hkv, N, d, 0)) {
    p.kv_split = dkdv_split(B, Hq, Hkv, N, d, causal, p.window);
    p.dkv_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + need);
  }
  p.status = status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  const int e = fa::launch_bwd_bf16(p, stream, stage);
  return e == 0 ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                 const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                 int d, float scale, int causal, int window, const int32_t* cu_seqlens,
                 long long total_tokens, const float* alibi_slopes, fa_dtype dtype,
                 fa_dtype o_dtype, int deterministic, void* workspace, size_t workspace_bytes,
                 void* stream) {
  return bwd_impl(-1, q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, causal, window,
                  cu_seqlens, total_tokens, alibi_slopes, dtype, o_dtype, deterministic,
                  workspace, workspace_bytes, stream);
}

fa_status fa_bwd_stage(int stage, const void* q, const void* k, const void* v, const void* o,
                       const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                       int Hq, int Hkv, int N, int d, float scale, int causal, int window,
                       const int32_t* cu_seqlens, long long total_tokens,
                       const float* alibi_slopes, fa_dtype dtype, fa_dtype o_dtype,
                       int deterministic, void* workspace, size_t workspace_bytes,
                       void* stream) {
  if (stage < 0 || stage > 2) return FA_ERR_UNSUPPORTED;
  return bwd_impl(stage, q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, causal,
                  window, cu_seqlens, total_tokens, alibi_slopes, dtype, o_dtype, deterministic,
                  workspace, workspace_bytes, stream);
}

// Decode: sizes valid and supported?  Fills the derived sizes.
static fa_status decode_sizes(int B, int Hq, int Hkv, int S_max, int q_len, int d, int* R,
                              int* chunk, int* nsplit) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || S_max < 0 || q_len <= 0 || d <= 0) return FA_ERR_SHAPE;
  if (Hq % Hkv != 0) return FA_ERR_SHAPE;
  if (B > 0 && q_len > S_max) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long rows = (long long)(Hq / Hkv) * q_len;
  if (rows > fa::kDecodeMaxRows) return FA_ERR_UNSUPPORTED;
  if ((long long)B * S_max >= (1ll << 31) || (long long)B * q_len * Hq >= (1ll << 31))
    return FA_ERR_UNSUPPORTED;
  *R = (int)rows;
  *chunk = fa::decode_chunk(B, Hkv, S_max);
  *nsplit = S_max > 0 ? (S_max + *chunk - 1) / *chunk : 0;
  return FA_OK;
}

size_t fa_decode_workspace_size(int B, int Hq, int Hkv, int S_max, int q_len, int d) {
  int R = 0, chunk = 0, nsplit = 0;
  if (decode_sizes(B, Hq, Hkv, S_max, q_len, d, &R, &chunk, &nsplit) != FA_OK) return 0;
  const size_t units = (size_t)B * Hkv * nsplit;
  return round256(units * R * d * sizeof(float)) + round256(units * R * 3 * sizeof(float));
}

fa_status fa_decode(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* cache_seqlens, void* o, float* lse, int B, int Hq, int Hkv,
                    int S_max, int q_len, int d, float scale, int window,
                    const float* alibi_slopes, fa_dtype o_dtype, void* workspace,
                    size_t workspace_bytes, void* stream) {
  int R = 0, chunk = 0, nsplit = 0;
  fa_status st = decode_sizes(B, Hq, Hkv, S_max, q_len, d, &R, &chunk, &nsplit);
  if (st != FA_OK) return st;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_UNSUPPORTED;
  if (o_dtype != FA_FP32 && o_dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (!q || !k_cache || !v_cache || !o || !lse) return FA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
    return FA_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_ALIGN;
  if (B == 0) return FA_OK;
  const size_t need = fa_decode_workspace_size(B, Hq, Hkv, S_max, q_len, d);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_ALIGN;
  fa::DecodeParams p = {};
  p.q = q;
  p.k = k_cache;
  p.v = v_cache;
  p.o = o;
  p.lse = lse;
  p.seqlens = cache_seqlens;
  p.alibi = alibi_slopes;
  const size_t units = (size_t)B * Hkv * nsplit;
  p.part_o = static_cast<float*>(workspace);
  p.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                       round256(units * R * d * sizeof(float)));
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.S_max = S_max;
  p.q_len = q_len;
  p.d = d;
  p.group = Hq / Hkv;
  p.R = R;
  p.chunk = chunk;
  p.nsplit = nsplit;
  p.window = band_width(window, S_max);
  p.o_f32 = o_dtype == FA_FP32;
  p.scale = scale;
  p.scale_log2 = scale * fa::kLog2e;
  p.status = status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  const int e = fa::launch_decode_bf16(p, stream);
  return e == 0 ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fp8_layout_get(int B, int Hq, int Hkv, int N, int d, long long total_tokens,
                            fa_fp8_layout* out) {
  if (!out) return FA_ERR_NULL;
  if (B < 0 || N < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || total_tokens < 0) return FA_ERR_SHAPE;
  if (Hq % Hkv != 0) return FA_ERR_SHAPE;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  const long long T = total_tokens > 0 ? total_tokens : (long long)B * N;
  const long long nblk = ((long long)N + 127) / 128;
  const long long vt = (long long)B * nblk * 128;      // keys per transposed V row
  // token and key coordinates are 32-bit in the TMA descriptors
  if (T >= (1ll << 31) || vt >= (1ll << 31) || (long long)N >= (1ll << 30)) return FA_ERR_UNSUPPORTED;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = round256(off + bytes);
    return at;
  };
  out->q8 = take((size_t)T * Hq * 128);
  out->k8 = take((size_t)T * Hkv * 128);
  out->v8t = take((size_t)Hkv * 128 * vt);
  out->q_scale = take(sizeof(float) * Hq * B * nblk);
  out->k_scale = take(sizeof(float) * Hkv * B * nblk);
  out->v_scale = take(sizeof(float) * Hkv * B * nblk);
  out->v_scale_max = take(sizeof(float) * Hkv);
  out->total = off;
  out->nblk = (int)nblk;
  return FA_OK;
}

fa_status fa_fp8_quantize(const void* q, const void* k, const void* v, const float* signs,
                          int B, int Hq, int Hkv, int N, int d, const int32_t* cu_seqlens,
                          long long total_tokens, void* fp8_buf, size_t fp8_bytes, void* stream) {
  long long T = 0;
  fa_status st = check_sizes(B, Hq, Hkv, N, d, 1.0f, cu_seqlens, total_tokens, FA_BF16, false, &T);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !signs) return FA_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return FA_ERR_ALIGN;
  if (T == 0 || B == 0 || N == 0) return FA_OK;
  fa_fp8_layout lay;
  st = fa_fp8_layout_get(B, Hq, Hkv, N, d, cu_seqlens ? T : 0, &lay);
  if (st != FA_OK) return st;
  if (!fp8_buf || fp8_bytes < lay.total) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(fp8_buf) & 255u) != 0) return FA_ERR_ALIGN;
  char* base = static_cast<char*>(fp8_buf);
  fa::QuantParams p = {};
  p.q = q;
  p.k = k;
  p.v = v;
  p.signs = signs;
  p.cu_seqlens = cu_seqlens;
  p.q8 = reinterpret_cast<uint8_t*>(base + lay.q8);
  p.k8 = reinterpret_cast<uint8_t*>(base + lay.k8);
  p.v8t = reinterpret_cast<uint8_t*>(base + lay.v8t);
  p.q_scale = reinterpret_cast<float*>(base + lay.q_scale);
  p.k_scale = reinterpret_cast<float*>(base + lay.k_scale);
  p.v_scale = reinterpret_cast<float*>(base + lay.v_scale);
  p.v_smax = reinterpret_cast<float*>(base + lay.v_scale_max);
  p.T = T;
  p.vt_stride = (long long)B * lay.nblk * 128;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.nblk = lay.nblk;
  p.status = status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  return fa::launch_fp8_quantize(p, stream) == 0 ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_fwd_fp8(const void* fp8_buf, size_t fp8_bytes, void* o, float* lse, int B, int Hq,
                     int Hkv, int N, int d, float scale, int causal, int window,
                     const int32_t* cu_seqlens, long long total_tokens,
                     const float* alibi_slopes, fa_dtype o_dtype, void* stream) {
  long long T = 0;
  fa_status st = check_sizes(B, Hq, Hkv, N, d, scale, cu_seqlens, total_tokens, FA_BF16, false, &T);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (window >= 0 && !causal) return FA_ERR_UNSUPPORTED;
  if (o_dtype != FA_FP32 && o_dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  if (!fp8_buf || !o || !lse) return FA_ERR_NULL;
  if (!aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(fp8_buf) & 255u) != 0) return FA_ERR_ALIGN;
  if (T == 0 || B == 0 || N == 0) return FA_OK;
  fa_fp8_layout lay;
  st = fa_fp8_layout_get(B, Hq, Hkv, N, d, cu_seqlens ? T : 0, &lay);
  if (st != FA_OK) return st;
  if (fp8_bytes < lay.total) return FA_ERR_WORKSPACE;
  const char* base = static_cast<const char*>(fp8_buf);
  fa::AttnParams p = base_params(B, Hq, Hkv, N, d, scale, causal, window, cu_seqlens, T,
                                 alibi_slopes);
  p.q = base + lay.q8;
  p.k = base + lay.k8;
  p.v = base + lay.v8t;
  p.q_scale = reinterpret_cast<const float*>(base + lay.q_scale);
  p.k_scale = reinterpret_cast<const float*>(base + lay.k_scale);
  p.v_scale = reinterpret_cast<const float*>(base + lay.v_scale);
  p.v_smax = reinterpret_cast<const float*>(base + lay.v_scale_max);
  p.nblk = lay.nblk;
  p.vt_stride = (long long)B * lay.nblk * 128;
  p.o = o;
  p.lse = lse;
  p.o_f32 = o_dtype == FA_FP32;
  p.status = status_ptr();
  if (!p.status) return FA_ERR_CUDA;
  return fa::launch_fwd_fp8(p, stream) == 0 ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_selftest_wait_timeout(unsigned long long limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull) return FA_ERR_UNSUPPORTED;
  unsigned int* status = status_ptr();
  if (!status) return FA_ERR_CUDA;
  return fa::launch_selftest_wait(status, limit_ns, stream) == 0 ? FA_OK : FA_ERR_CUDA;
}

int fa_bwd_dkdv_split(int B, int Hq, int Hkv, int N, int d, int causal, int window,
                      const int32_t* cu_seqlens, size_t workspace_bytes) {
  if (B <= 0 || N <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return 1;
  if (cu_seqlens || gqa_split_max(Hq, Hkv) == 1) return 1;
  if (workspace_bytes < fa_bwd_workspace_size_gqa(B, Hq, Hkv, N, d, 0)) return 1;
  return dkdv_split(B, Hq, Hkv, N, d, causal ? 1 : 0, band_width(window, N));
}

void fa_host_cache_stats(unsigned long long* tmaps_encoded, unsigned long long* tmaps_reused,
                         unsigned long long* smem_attrs_set) {
  fa::host_cache_stats(tmaps_encoded, tmaps_reused, smem_attrs_set);
}

fa_status fa_check_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int* p = status_ptr();
  if (!p) return FA_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (v != 0 && cudaMemset(p, 0, sizeof(v)) != cudaSuccess) return FA_ERR_CUDA;
  return static_cast<fa_status>(v);
}

}  // extern "C"
