// fa_host_util.cu -- host set-up shared by the launchers: TMA descriptors
// (encoded through the driver entry point, so the library does not link
// libcuda and loads on machines without a driver), kept in a per-shape
// cache; the per-kernel shared-memory limit and the SM count, each set or
// read once per device.
#include "fa_host_util.h"

#include <atomic>
#include <cstring>
#include <mutex>

namespace fa {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Everything a tiled 3-D descriptor is made of.  Two calls with equal keys
// get bit-identical descriptors, so the encoded one is kept and reused.
struct TmapKey {
  const void* base;
  uint64_t dims[3];
  uint64_t strides[2];
  uint32_t box[3];
  int dtype;
  bool operator==(const TmapKey& o) const { return std::memcmp(this, &o, sizeof(*this)) == 0; }
};

// Direct-mapped cache: a slot holds the last descriptor whose key hashed to
// it.  A hit returns a copy; a miss encodes and replaces the slot.
constexpr int kCacheSlots = 256;
struct CacheSlot {
  bool used = false;
  TmapKey key;
  CUtensorMap map;
};
CacheSlot g_cache[kCacheSlots];
std::mutex g_cache_mu;
std::atomic<unsigned long long> g_encoded{0}, g_reused{0}, g_attr_set{0};

size_t hash_key(const TmapKey& k) {
  const unsigned char* p = reinterpret_cast<const unsigned char*>(&k);
  uint64_t h = 1469598103934665603ull;          // FNV-1a over the key's bytes
  for (size_t i = 0; i < sizeof(k); ++i) h = (h ^ p[i]) * 1099511628211ull;
  return (size_t)(h % kCacheSlots);
}

int encode(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, const uint64_t dims[3],
           const uint64_t strides[2], const uint32_t box[3]) {
  TmapKey key;
  std::memset(&key, 0, sizeof(key));                 // padding bytes take part in ==
  key.base = base;
  std::memcpy(key.dims, dims, sizeof(key.dims));
  std::memcpy(key.strides, strides, sizeof(key.strides));
  std::memcpy(key.box, box, sizeof(key.box));
  key.dtype = (int)dtype;
  const size_t slot = hash_key(key);
  {
    std::lock_guard<std::mutex> lock(g_cache_mu);
    if (g_cache[slot].used && g_cache[slot].key == key) {
      *map = g_cache[slot].map;
      g_reused.fetch_add(1, std::memory_order_relaxed);
      return 0;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return (int)cudaErrorInitializationError;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t s[2] = {strides[0], strides[1]};
  cuuint32_t b[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dtype, 3, const_cast<void*>(base), d, s, b, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return (int)cudaErrorInvalidValue;
  g_encoded.fetch_add(1, std::memory_order_relaxed);
  std::lock_guard<std::mutex> lock(g_cache_mu);
  g_cache[slot].used = true;
  g_cache[slot].key = key;
  g_cache[slot].map = *map;
  return 0;
}

constexpr int kMaxDevices = 64;
constexpr int kMaxKernels = 256;

}  // namespace

int make_tmap_bf16_3d(CUtensorMap* map, const void* base, int d, int H, long long T,
                      int box_rows) {
  const uint64_t dims[3] = {(uint64_t)d, (uint64_t)H, (uint64_t)T};
  const uint64_t strides[2] = {(uint64_t)d * 2, (uint64_t)d * 2 * H};
  const uint32_t box[3] = {64, 1, (uint32_t)box_rows};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, dims, strides, box);
}

int make_tmap_bf16_3d_box(CUtensorMap* map, const void* base, int d, int H, long long T,
                          int box_h, int box_t) {
  const uint64_t dims[3] = {(uint64_t)d, (uint64_t)H, (uint64_t)T};
  const uint64_t strides[2] = {(uint64_t)d * 2, (uint64_t)d * 2 * H};
  const uint32_t box[3] = {64, (uint32_t)box_h, (uint32_t)box_t};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, dims, strides, box);
}

int make_tmap_f32_3d(CUtensorMap* map, const void* base, int d, int H, long long T, int box_rows) {
  const uint64_t dims[3] = {(uint64_t)d, (uint64_t)H, (uint64_t)T};
  const uint64_t strides[2] = {(uint64_t)d * 4, (uint64_t)d * 4 * H};
  const uint32_t box[3] = {32, 1, (uint32_t)box_rows};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, dims, strides, box);
}

int make_tmap_u8_3d(CUtensorMap* map, const void* base, long long n0, long long n1, long long n2,
                    long long s1, long long s2, int b0, int b1, int b2) {
  const uint64_t dims[3] = {(uint64_t)n0, (uint64_t)n1, (uint64_t)n2};
  const uint64_t strides[2] = {(uint64_t)s1, (uint64_t)s2};
  const uint32_t box[3] = {(uint32_t)b0, (uint32_t)b1, (uint32_t)b2};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, dims, strides, box);
}

int set_max_dynamic_smem(const void* kernel, int bytes) {
  // (device, kernel) pairs already set; the attribute belongs to the
  // kernel's function in the current device's context.
  static const void* done[kMaxDevices][kMaxKernels] = {};
  static int ndone[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  std::lock_guard<std::mutex> lock(mu);
  const bool known = dev >= 0 && dev < kMaxDevices;
  if (known)
    for (int i = 0; i < ndone[dev]; ++i)
      if (done[dev][i] == kernel) return 0;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return (int)e;
  g_attr_set.fetch_add(1, std::memory_order_relaxed);
  if (known && ndone[dev] < kMaxKernels) done[dev][ndone[dev]++] = kernel;
  return 0;
}

int sm_count(int* nsm) {
  static std::atomic<int> cached[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) {
      *nsm = c;
      return 0;
    }
  }
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return (int)e;
  if (dev >= 0 && dev < kMaxDevices) cached[dev].store(n, std::memory_order_relaxed);
  *nsm = n;
  return 0;
}

void host_cache_stats(unsigned long long* encoded, unsigned long long* reused,
                      unsigned long long* attr_set) {
  if (encoded) *encoded = g_encoded.load();
  if (reused) *reused = g_reused.load();
  if (attr_set) *attr_set = g_attr_set.load();
}

}  // namespace fa
