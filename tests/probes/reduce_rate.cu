// L2 throughput of cp.reduce.async.bulk .add.f32 from shared memory.
// Each CTA (one per SM) repeatedly adds a 32 KB staging buffer into its own
// region of a global accumulator (disjoint regions; the accumulator is sized
// beyond L2 when `spread` is large), with `inflight` reductions outstanding.
#include <cstdio>
#include <cuda_runtime.h>
#include "../../exact_io_aware_36_gb300/csrc/fa_internal.h"
#include "../../exact_io_aware_36_gb300/csrc/fa_ptx.cuh"
using namespace fa;

template <int INFLIGHT>
__global__ void __launch_bounds__(128, 1) probe(float* acc, long long region_floats, int reps, int chunk_bytes) {
  extern __shared__ __align__(128) uint8_t sm[];
  float* stg = reinterpret_cast<float*>(sm);
  for (int i = threadIdx.x; i < chunk_bytes / 4 * INFLIGHT; i += blockDim.x) stg[i] = 1.0f;
  fence_proxy_async_smem();
  __syncthreads();
  if (threadIdx.x == 0) {
    float* base = acc + (long long)blockIdx.x * region_floats;
    const long long nchunks = region_floats * 4 / chunk_bytes;
    for (int r = 0; r < reps; ++r) {
      const int slot = r % INFLIGHT;
      float* dst = base + (long long)(r % nchunks) * (chunk_bytes / 4);
      bulk_reduce_add_f32(dst, stg + slot * (chunk_bytes / 4), (uint32_t)chunk_bytes);
      bulk_commit_group();
      if (INFLIGHT == 1) bulk_wait_group_read0();
      else asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(INFLIGHT - 1) : "memory");
    }
    bulk_wait_group0();
  }
}

template <int INFLIGHT>
void run(float* acc, long long region, int nsm, int reps, int chunk) {
  auto k = probe<INFLIGHT>;
  const int smem = chunk * INFLIGHT;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  k<<<nsm, 128, smem>>>(acc, region, 4, chunk);
  cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
  cudaEventRecord(e0);
  k<<<nsm, 128, smem>>>(acc, region, reps, chunk);
  cudaEventRecord(e1);
  cudaError_t err = cudaDeviceSynchronize();
  float ms = 0; cudaEventElapsedTime(&ms, e0, e1);
  double bytes = (double)chunk * reps * nsm;
  printf("inflight=%d chunk=%d region/CTA=%lld MB: %.3f ms, %.2f TB/s of fp32 adds, err=%d\n", INFLIGHT, chunk,
         region * 4 >> 20, ms, bytes / (ms * 1e-3) / 1e12, (int)err);
}

int main() {
  int nsm = 0; cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
  const long long region = (8ll << 20) / 4;         // 8 MB per CTA: 1.2 GB in total, beyond L2
  float* acc; cudaMalloc(&acc, region * 4 * nsm); cudaMemset(acc, 0, region * 4 * nsm);
  run<1>(acc, region, nsm, 2000, 32768);
  run<2>(acc, region, nsm, 2000, 32768);
  run<4>(acc, region, nsm, 2000, 32768);
  run<6>(acc, region, nsm, 2000, 32768);
  const long long small = (256ll << 10) / 4;         // 256 KB per CTA: 38 MB in total, inside L2
  run<1>(acc, small, nsm, 2000, 32768);
  run<4>(acc, small, nsm, 2000, 32768);
  cudaFree(acc);
  return 0;
}
