// sustained tcgen05.mma rate per shape (one CTA per SM, one issuing
// thread, fp32 accumulate in TMEM).  Operands are all zero, or (fill = 1)
// pseudo-random bf16 values in [-2, 2): in shared memory, and for the TS
// form also in the TMEM columns that hold A.  Zero operands switch fewer
// bits, so the pair shows how much the data itself costs.
#include <cstdio>
#include <cuda_runtime.h>
#include "../../exact_io_aware_36_gb300/csrc/fa_internal.h"
#include "../../exact_io_aware_36_gb300/csrc/fa_ptx.cuh"
using namespace fa;

struct __align__(8) PBars { uint64_t done; uint32_t tmem; int abort_flag; };

// MODE 0: SS, A K-major 128 rows, B K-major N rows, K = 64 per round (4 MMAs)
// MODE 1: TS, A from TMEM, B MN-major (N = 128 columns), K = 64 per round
__device__ __forceinline__ uint32_t rnd_bf16x2(uint32_t i) {
  uint32_t h = i * 0x9E3779B1u;
  h ^= h >> 15; h *= 0x85EBCA77u; h ^= h >> 13;
  // two bf16 values with exponents 2^-1 .. 2^0 and random signs and mantissas
  const uint32_t lo = 0x3F00u | (h & 0x807Fu), hi = 0x3F00u | ((h >> 16) & 0x807Fu);
  return lo | (hi << 16);
}

template <int N, int MODE>
__global__ void __launch_bounds__(128, 1) probe(int rounds, int fill, unsigned long long* cycles, unsigned int* status) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;                     // 128 x 64 bf16 = 16 KB
  uint8_t* sB = smem + 16384;             // N x 64 bf16 (K-major) or 64 x N (MN-major)
  PBars* bars = reinterpret_cast<PBars*>(smem + 16384 + 65536);
  for (int i = threadIdx.x; i < (16384 + 65536) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = fill ? make_uint4(rnd_bf16x2(4 * i), rnd_bf16x2(4 * i + 1), rnd_bf16x2(4 * i + 2),
                                                          rnd_bf16x2(4 * i + 3))
                                             : make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) { mbar_init(&bars->done, 1); bars->abort_flag = 0; fence_mbarrier_init(); }
  fence_proxy_async_smem();
  if (threadIdx.x < 32) { tmem_alloc(&bars->tmem, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  const WaitCtx wc{&bars->abort_flag, status};
  if (MODE == 1) {      // A of the TS form: TMEM columns 0..31, one lane quarter per warp
    uint32_t v[16];
    for (int half = 0; half < 2; ++half) {
#pragma unroll
      for (int c = 0; c < 16; ++c) v[c] = fill ? rnd_bf16x2(threadIdx.x * 64 + half * 16 + c) : 0u;
      tmem_st16(tmem + ((uint32_t)(32 * (threadIdx.x >> 5)) << 16) + 16 * half, v);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) {
    const uint32_t a = smem_u32(sA), bb = smem_u32(sB);
    long long t0 = clock64();
    if (threadIdx.x == 0) {
      for (int r = 0; r < rounds; ++r) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          if (MODE == 0) {
            constexpr uint32_t ID = idesc_bf16_f32(128, N, 0, 0);
            mma_ss(tmem + 256 * (r & 1) * (N <= 256 ? 0 : 0), smem_desc_sw128(a + kk * 32, 16, 1024),
                   smem_desc_sw128(bb + kk * 32, 16, 1024), ID, (r > 0 || kk > 0) ? 1u : 0u);
          } else {
            constexpr uint32_t ID = idesc_bf16_f32(128, N, 0, 1);
            mma_ts(tmem + 256, tmem + 8 * kk, smem_desc_sw128(bb + kk * 2048, 8192, 1024), ID,
                   (r > 0 || kk > 0) ? 1u : 0u);
          }
        }
      }
      mma_commit(&bars->done);
    }
    __syncwarp();
    wait_warp(&bars->done, 0, wc);
    long long t1 = clock64();
    if (threadIdx.x == 0) cycles[blockIdx.x] = (unsigned long long)(t1 - t0);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

template <int N, int MODE>
void run(const char* name, int rounds, int fill, int nsm, unsigned long long* d_cyc, unsigned int* d_st) {
  auto k = probe<N, MODE>;
  const int smem = 16384 + 65536 + 64 + 1024;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  k<<<nsm, 128, smem>>>(rounds, fill, d_cyc, d_st);      // warm-up
  cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
  cudaEventRecord(e0);
  k<<<nsm, 128, smem>>>(rounds, fill, d_cyc, d_st);
  cudaEventRecord(e1);
  cudaError_t err = cudaDeviceSynchronize();
  float ms = 0; cudaEventElapsedTime(&ms, e0, e1);
  unsigned int st = 0; cudaMemcpy(&st, d_st, 4, cudaMemcpyDeviceToHost);
  double flops = 2.0 * 128 * N * 64 * (double)rounds * nsm;
  printf("%-28s N=%3d %-6s rounds=%d: %.3f ms  %.1f TFLOP/s  err=%d status=%u\n", name, N,
         fill ? "random" : "zero", rounds, ms,
         flops / (ms * 1e-3) / 1e12, (int)err, st);
}

int main() {
  int nsm = 0; cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
  unsigned long long* d_cyc; unsigned int* d_st;
  cudaMalloc(&d_cyc, 8 * 1024); cudaMalloc(&d_st, 4); cudaMemset(d_st, 0, 4);
  printf("SMs %d\n", nsm);
  for (int fill = 0; fill < 2; ++fill) {
    run<64, 0>("SS K-major", 20000, fill, nsm, d_cyc, d_st);
    run<128, 0>("SS K-major", 10000, fill, nsm, d_cyc, d_st);
    run<256, 0>("SS K-major", 5000, fill, nsm, d_cyc, d_st);
    run<128, 1>("TS, B MN-major", 10000, fill, nsm, d_cyc, d_st);
    run<64, 1>("TS, B MN-major", 20000, fill, nsm, d_cyc, d_st);
  }
  return 0;
}
