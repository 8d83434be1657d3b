// fa_bwd_static.cu -- the backward for callers that cannot allocate device
// memory.
//
// fa_bwd needs a workspace (D and the fp32 dQ accumulator) that its caller
// allocates.  Some callers cannot do that: a plugin or custom-op hook inside
// another framework that hands out no workspace and whose allocator it cannot
// reach, a runtime that fixes its device memory at start-up and forbids any
// allocation on the request path, or code that must not call cudaMalloc
// because it would synchronise the device or break a capture in progress.
// For them, fa_bwd_static_scratch runs the same three backward kernels with
// the workspace placed in a fixed array in the library's own device memory.
//
// The array is a file-scope __device__ variable: once reserved on a GPU it
// stays until the process exits.  When it is reserved depends on how CUDA
// loads modules: eagerly, with the library's module; under lazy loading
// (CUDA_MODULE_LOADING=LAZY, the default since CUDA 12.2) only when this
// file's module is first needed, which is the first call's
// cudaGetSymbolAddress below.  So the first call on each device may itself
// reserve the 64 MiB.  In host code the array's name is only a host-side
// stand-in, so the device address is looked up once per device with
// cudaGetSymbolAddress and passed to the kernels like any caller-owned
// workspace.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "fa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[FA_BWD_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_bwd_scratch on the current device, resolved on the
// first call made with that device current; nullptr if the lookup fails.
void* scratch_ptr() {
  static void* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace

extern "C" fa_status fa_bwd_static_scratch(
    const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
    void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, float scale, int causal,
    int window, const int32_t* cu_seqlens, long long total_tokens, const float* alibi_slopes,
    fa_dtype dtype, fa_dtype o_dtype, int deterministic, void* stream) {
  // fa_bwd's own argument checks come first, so a bad argument gets the same
  // status as from fa_bwd, and an empty problem (no tokens) succeeds without
  // touching the GPU whatever its nominal sizes.  The size check follows; it
  // needs no GPU either: a problem whose D and dQ accumulator do not fit the
  // fixed array is refused before anything runs.
  long long T = 0;
  const fa_status st = fa::bwd_check_args(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, d,
                                          scale, causal, window, cu_seqlens, total_tokens, dtype,
                                          o_dtype, deterministic, &T);
  if (st != FA_OK || T == 0) return st;
  const size_t need = fa_bwd_workspace_size(B, Hq, N, d, T);
  if (need > (size_t)FA_BWD_STATIC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
  void* ws = scratch_ptr();
  if (!ws) return FA_ERR_CUDA;
  // Everything the kernels read from the scratch is written by the same call
  // first: D by the preprocess kernel, and the dQ accumulator is zeroed
  // there too, so the previous call's contents never leak into this one.
  // The workspace is declared at the size fa_bwd_workspace_size gives, so the
  // same schedule runs as for a caller who allocated exactly that much.
  return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, causal, window,
                cu_seqlens, total_tokens, alibi_slopes, dtype, o_dtype, deterministic, ws, need,
                stream);
}
