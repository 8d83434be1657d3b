// Throughput of the softmax's per-score instructions on one GB300, and of the
// whole per-pair body of the forward's exp pass in two forms: P packed to
// bf16 with cvt.rn.bf16x2.f32 (round to nearest) or with prmt (the upper
// halves of the two fp32 words).  Each of 4 x #SM blocks of 512 threads runs
// 8 independent chains of ITER dependent steps; the third launch is timed
// with CUDA events.  Rates are instructions (x 32 lanes) per SM per clock at
// the device's reported maximum clock, so they read low if the clock sagged.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

constexpr int ITER = 2048;
constexpr int CH = 8;

__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void split(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}

__global__ void k_ex2(float* out, float seed) {
  float a[CH];
  for (int i = 0; i < CH; ++i) a[i] = seed * (i + 1) * 1e-3f - 0.5f;
  for (int it = 0; it < ITER; ++it)
#pragma unroll
    for (int i = 0; i < CH; ++i) asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(a[i]));
  float s = 0.f;
  for (int i = 0; i < CH; ++i) s += a[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

__global__ void k_cvt(float* out, float seed) {
  uint32_t a[CH];
  for (int i = 0; i < CH; ++i) a[i] = __float_as_uint(seed + i);
  for (int it = 0; it < ITER; ++it)
#pragma unroll
    for (int i = 0; i < CH; ++i)
      asm volatile("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(a[i]) : "f"(__uint_as_float(a[i])), "f"(seed));
  uint32_t s = 0;
  for (int i = 0; i < CH; ++i) s ^= a[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = (float)(s & 0xffff);
}

__global__ void k_prmt(float* out, float seed) {
  uint32_t a[CH];
  const uint32_t b = __float_as_uint(seed);
  for (int i = 0; i < CH; ++i) a[i] = __float_as_uint(seed + i);
  for (int it = 0; it < ITER; ++it)
#pragma unroll
    for (int i = 0; i < CH; ++i) asm volatile("prmt.b32 %0, %0, %1, 0x7632;" : "+r"(a[i]) : "r"(b));
  uint32_t s = 0;
  for (int i = 0; i < CH; ++i) s ^= a[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = (float)(s & 0xffff);
}

__global__ void k_fadd2(float* out, float seed) {
  uint64_t a[CH];
  const uint64_t b = f2(seed, seed);
  for (int i = 0; i < CH; ++i) a[i] = f2(seed + i, seed - i);
  for (int it = 0; it < ITER; ++it)
#pragma unroll
    for (int i = 0; i < CH; ++i) asm volatile("add.rn.f32x2 %0, %0, %1;" : "+l"(a[i]) : "l"(b));
  uint64_t s = 0;
  for (int i = 0; i < CH; ++i) s ^= a[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = (float)(s & 0xffff);
}

__global__ void k_ffma2(float* out, float seed) {
  uint64_t a[CH];
  const uint64_t b = f2(0.999f, 0.999f), c = f2(seed, seed);
  for (int i = 0; i < CH; ++i) a[i] = f2(seed + i, seed - i);
  for (int it = 0; it < ITER; ++it)
#pragma unroll
    for (int i = 0; i < CH; ++i) asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(a[i]) : "l"(b), "l"(c));
  uint64_t s = 0;
  for (int i = 0; i < CH; ++i) s ^= a[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = (float)(s & 0xffff);
}

__global__ void k_ffma(float* out, float seed) {
  float a[CH];
  for (int i = 0; i < CH; ++i) a[i] = seed + i;
  for (int it = 0; it < ITER; ++it)
#pragma unroll
    for (int i = 0; i < CH; ++i) asm volatile("fma.rn.f32 %0, %0, 0f3F7FBE77, %1;" : "+f"(a[i]) : "f"(seed));
  float s = 0.f;
  for (int i = 0; i < CH; ++i) s += a[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// One pair of scores as the exp pass treats it: x*c - m (packed), two exp2,
// the pair summed into acc, the pair packed to bf16, and the packed values
// summed into accr.  PRMT selects the packing.
template <bool PRMT>
__global__ void k_pair(float* out, float seed) {
  uint64_t acc[CH], accr[CH], xy[CH];
  const uint64_t c2 = f2(0.18f, 0.18f), nm = f2(-1.0f, -1.0f);
  for (int i = 0; i < CH; ++i) {
    acc[i] = accr[i] = f2(0.f, 0.f);
    xy[i] = f2(seed * i * 1e-3f, seed * i * 2e-3f);
  }
  for (int it = 0; it < ITER; ++it)
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      uint64_t e;
      asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(e) : "l"(xy[i]), "l"(c2), "l"(nm));
      float e0, e1, p0, p1;
      split(e, e0, e1);
      asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(p0) : "f"(e0));
      asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(p1) : "f"(e1));
      asm volatile("add.rn.f32x2 %0, %0, %1;" : "+l"(acc[i]) : "l"(f2(p0, p1)));
      uint32_t pk;
      if (PRMT)
        asm volatile("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(pk) : "r"(__float_as_uint(p0)), "r"(__float_as_uint(p1)));
      else
        asm volatile("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(pk) : "f"(p1), "f"(p0));
      const uint64_t r = f2(__uint_as_float(pk << 16), __uint_as_float(pk & 0xFFFF0000u));
      asm volatile("add.rn.f32x2 %0, %0, %1;" : "+l"(accr[i]) : "l"(r));
      xy[i] ^= (uint64_t)(pk & 1u);                 // keeps the chain dependent
    }
  uint64_t s = 0;
  for (int i = 0; i < CH; ++i) s ^= acc[i] ^ accr[i];
  out[blockIdx.x * blockDim.x + threadIdx.x] = (float)(s & 0xffff);
}

int main() {
  int sms = 0, clk_khz = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, 0);
  const int blocks = sms * 4, threads = 512;
  float* out = nullptr;
  cudaMalloc(&out, sizeof(float) * blocks * threads);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  struct K { const char* name; void (*fn)(float*, float); int per_step; };
  const K ks[] = {{"ex2.approx.ftz.f32", k_ex2, 1},
                  {"cvt.rn.bf16x2.f32", k_cvt, 1},
                  {"prmt.b32", k_prmt, 1},
                  {"add.rn.f32x2", k_fadd2, 1},
                  {"fma.rn.f32x2", k_ffma2, 1},
                  {"fma.rn.f32", k_ffma, 1},
                  {"exp-pass pair, cvt packing", k_pair<false>, 1},
                  {"exp-pass pair, prmt packing", k_pair<true>, 1}};
  for (const K& k : ks) {
    float ms = 0.f;
    for (int rep = 0; rep < 3; ++rep) {
      cudaEventRecord(e0);
      k.fn<<<blocks, threads>>>(out, 1.0f);
      cudaEventRecord(e1);
      cudaEventSynchronize(e1);
      cudaEventElapsedTime(&ms, e0, e1);
    }
    const double steps = (double)blocks * threads * ITER * CH * k.per_step;
    const double per_sm_clk = steps / (ms * 1e-3) / sms / (clk_khz * 1e3);
    printf("%-30s %.3f ms  per SM per clock at %d MHz: rate=%.2f\n", k.name, ms, clk_khz / 1000, per_sm_clk);
  }
  const cudaError_t err = cudaDeviceSynchronize();
  printf("err=%d status=0\n", (int)err);
  cudaFree(out);
  return 0;
}
