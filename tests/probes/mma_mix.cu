// The per-step MMA mixes of the attention kernels, issued back to back by one
// thread per SM on zero operands, d = 128:
//  * dK/dV kernel: five products per 64-query step over 128 keys;
//  * forward: per 128-key step, for two 128-row query tiles t,
//    O_t += P_t V (A = P_t from TMEM over S_t's columns) then S_t = Q_t K^T,
//    in the kernel's order PV0, S0, PV1, S1, and once more with P read from
//    columns no S product writes (no write-after-read between them).
#include <cstdio>
#include <cuda_runtime.h>
#include "../../exact_io_aware_36_gb300/csrc/fa_internal.h"
#include "../../exact_io_aware_36_gb300/csrc/fa_ptx.cuh"
using namespace fa;
struct __align__(8) PBars { uint64_t done; uint32_t tmem; int abort_flag; };

// MASK bit 0: S, 1: dP, 2: dV, 3: dK, 4: dQ^T
template <int MASK>
__global__ void __launch_bounds__(128, 1) mix(int steps, unsigned int* status) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  // K 32 KB, V 32 KB, Q 16 KB, dO 16 KB, dS 16 KB
  const int TOT = 32768 * 2 + 16384 * 3;
  PBars* bars = reinterpret_cast<PBars*>(smem + TOT);
  for (int i = threadIdx.x; i < TOT / 16; i += blockDim.x) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) { mbar_init(&bars->done, 1); bars->abort_flag = 0; fence_mbarrier_init(); }
  fence_proxy_async_smem();
  if (threadIdx.x < 32) { tmem_alloc(&bars->tmem, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  const WaitCtx wc{&bars->abort_flag, status};
  if (threadIdx.x < 32) {
    const uint32_t sK = smem_u32(smem), sV = sK + 32768, sQ = sV + 32768, sdO = sQ + 16384, sdS = sdO + 16384;
    constexpr uint32_t ID_S = idesc_bf16_f32(128, 64, 0, 0);
    constexpr uint32_t ID_KV = idesc_bf16_f32(128, 128, 0, 1);
    constexpr uint32_t ID_DQ = idesc_bf16_f32(128, 64, 1, 1);
    if (threadIdx.x == 0) {
      for (int it = 0; it < steps; ++it) {
        const int buf = it & 1;
        if (MASK & 1)
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t offk = (kk >> 2) * 16384 + (kk & 3) * 32, offq = (kk >> 2) * 8192 + (kk & 3) * 32;
            mma_ss(tmem + 256 + 64 * buf, smem_desc_sw128(sK + offk, 16, 1024), smem_desc_sw128(sQ + offq, 16, 1024), ID_S, kk > 0);
          }
        if (MASK & 2)
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t offk = (kk >> 2) * 16384 + (kk & 3) * 32, offq = (kk >> 2) * 8192 + (kk & 3) * 32;
            mma_ss(tmem + 384 + 64 * buf, smem_desc_sw128(sV + offk, 16, 1024), smem_desc_sw128(sdO + offq, 16, 1024), ID_S, kk > 0);
          }
        if (MASK & 4)
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + 0, tmem + 256 + 64 * buf + 8 * kk, smem_desc_sw128(sdO + kk * 2048, 8192, 1024), ID_KV, 1u);
        if (MASK & 8)
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem + 128, tmem + 384 + 64 * buf + 8 * kk, smem_desc_sw128(sQ + kk * 2048, 8192, 1024), ID_KV, 1u);
        if (MASK & 16)
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + 384 + 64 * buf, smem_desc_sw128(sK + kk * 2048, 16384, 1024), smem_desc_sw128(sdS + kk * 2048, 8192, 1024), ID_DQ, kk > 0);
      }
      mma_commit(&bars->done);
    }
    __syncwarp();
    wait_warp(&bars->done, 0, wc);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

// HAZARD 1: P_t read from S_t's columns (the kernel's layout); 0: P read from
// columns 384.. that no S product writes, both PVs into one accumulator.
template <int HAZARD>
__global__ void __launch_bounds__(128, 1) fwd_mix(int steps, unsigned int* status) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  // Q0, Q1, K, V: 32 KB each (128 x 128 bf16 in two 64-column boxes)
  const int TOT = 32768 * 4;
  PBars* bars = reinterpret_cast<PBars*>(smem + TOT);
  for (int i = threadIdx.x; i < TOT / 16; i += blockDim.x) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) { mbar_init(&bars->done, 1); bars->abort_flag = 0; fence_mbarrier_init(); }
  fence_proxy_async_smem();
  if (threadIdx.x < 32) { tmem_alloc(&bars->tmem, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  const WaitCtx wc{&bars->abort_flag, status};
  if (threadIdx.x < 32) {
    const uint32_t sQ = smem_u32(smem), sK = sQ + 65536, sV = sK + 32768;
    constexpr uint32_t ID_S = idesc_bf16_f32(128, 128, 0, 0);
    constexpr uint32_t ID_O = idesc_bf16_f32(128, 128, 0, 1);
    if (threadIdx.x == 0) {
      for (int it = 0; it < steps; ++it) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint32_t colS = 128 * t, colO = HAZARD ? 256 + 128 * t : 256;
          const uint32_t colP = HAZARD ? colS : 384;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + colO, tmem + colP + 8 * kk, smem_desc_sw128(sV + kk * 2048, 16384, 1024), ID_O, 1u);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(tmem + colS, smem_desc_sw128(sQ + 32768 * t + off, 16, 1024),
                   smem_desc_sw128(sK + off, 16, 1024), ID_S, kk > 0 ? 1u : 0u);
          }
        }
      }
      mma_commit(&bars->done);
    }
    __syncwarp();
    wait_warp(&bars->done, 0, wc);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) { tc_fence_after(); tmem_dealloc(tmem, 512); }
}

template <int HAZARD>
void run_fwd(const char* name, int steps, int nsm, unsigned int* st) {
  auto k = fwd_mix<HAZARD>;
  const int smem = 32768 * 4 + 64 + 1024;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  k<<<nsm, 128, smem>>>(steps, st);
  cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
  cudaEventRecord(e0);
  k<<<nsm, 128, smem>>>(steps, st);
  cudaEventRecord(e1);
  cudaError_t err = cudaDeviceSynchronize();
  float ms; cudaEventElapsedTime(&ms, e0, e1);
  unsigned int s = 0; cudaMemcpy(&s, st, 4, cudaMemcpyDeviceToHost);
  const double flop_per_step = 4 * 2.0 * 128 * 128 * 128;
  printf("%-30s %.3f us/step  %.0f TFLOP/s  err=%d status=%u\n", name, ms * 1e3 / steps,
         flop_per_step * steps * nsm / (ms * 1e-3) / 1e12, (int)err, s);
}

template <int MASK>
void run(const char* name, double flop_per_step, int steps, int nsm, unsigned int* st) {
  auto k = mix<MASK>;
  const int smem = 32768 * 2 + 16384 * 3 + 64 + 1024;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  k<<<nsm, 128, smem>>>(steps, st);
  cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
  cudaEventRecord(e0);
  k<<<nsm, 128, smem>>>(steps, st);
  cudaEventRecord(e1);
  cudaError_t err = cudaDeviceSynchronize();
  float ms; cudaEventElapsedTime(&ms, e0, e1);
  unsigned int s = 0; cudaMemcpy(&s, st, 4, cudaMemcpyDeviceToHost);
  printf("%-30s %.3f us/step  %.0f TFLOP/s  err=%d status=%u\n", name, ms * 1e3 / steps,
         flop_per_step * steps * nsm / (ms * 1e-3) / 1e12, (int)err, s);
}

int main() {
  int nsm; cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
  unsigned int* st; cudaMalloc(&st, 4); cudaMemset(st, 0, 4);
  const double f = 2.0 * 128 * 64 * 128;   // one product of a step
  run<1>("S only (SS N64)", f, 20000, nsm, st);
  run<16>("dQ^T only (SS N64 MN/MN)", f, 20000, nsm, st);
  run<4>("dV only (TS N128)", f, 20000, nsm, st);
  run<3>("S + dP", 2 * f, 10000, nsm, st);
  run<12>("dV + dK", 2 * f, 10000, nsm, st);
  run<15>("S dP dV dK", 4 * f, 10000, nsm, st);
  run<31>("all five", 5 * f, 10000, nsm, st);
  run_fwd<1>("fwd PV0 S0 PV1 S1 (kernel)", 5000, nsm, st);
  run_fwd<0>("fwd, P apart from S", 5000, nsm, st);
  return 0;
}
