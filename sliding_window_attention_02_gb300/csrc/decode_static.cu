// Fused decode step whose split-K scratch lives in a static device array.
//
// rswa_decode_step_fused keeps its split-K partials and arrival counters in
// the caller's cache buffer, sized by rswa_cache_footprint.  This entry point
// runs the same kernel but takes that scratch from g_static_scratch below, a
// fixed array in the library's own device memory, so the call allocates
// nothing and touches no memory beyond the cache and the caller's q/k/v/o.
#include <mutex>

#include "rswa_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

// Split-K partials followed by the arrival counters.  Every GPU that loads
// the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device, looked up once
// per device (host code must not use the symbol itself as an address).
cudaError_t scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

namespace rswa {

// Bytes of static scratch a cache view needs: partials, then counters.
size_t static_scratch_need(const CacheView& cv, size_t* part_bytes,
                           size_t* cnt_bytes) {
  *part_bytes = align256(sizeof(float) * (size_t)cv.B * cv.H *
                         decode_part_slots(cv) * (cv.d + 2));
  *cnt_bytes = align256(sizeof(int32_t) * (size_t)cv.B * cv.H);
  return *part_bytes + *cnt_bytes;
}

size_t static_scratch_capacity() { return kStaticScratchBytes; }

// Runs the fused decode kernel with its scratch redirected to the static
// array.  The counters are cleared first, on the same stream.
cudaError_t launch_decode_fused_static(const CacheView& cv, int dev,
                                       const void* q, const void* k,
                                       const void* v, void* o, float* lse,
                                       bool prefetch_prefix, cudaStream_t s) {
  size_t part_bytes = 0, cnt_bytes = 0;
  if (static_scratch_need(cv, &part_bytes, &cnt_bytes) > kStaticScratchBytes)
    return cudaErrorInvalidValue;
  void* base = nullptr;
  cudaError_t e = scratch_address(dev, &base);
  if (e != cudaSuccess) return e;
  char* b = static_cast<char*>(base);
  CacheView sv = cv;
  sv.part = reinterpret_cast<float*>(b);
  sv.part_slots = decode_part_slots(cv);
  sv.cnt_bh = reinterpret_cast<int32_t*>(b + part_bytes);
  e = cudaMemsetAsync(sv.cnt_bh, 0, cnt_bytes, s);
  if (e != cudaSuccess) return e;
  return launch_decode(sv, q, k, v, o, lse, true, prefetch_prefix, s);
}

}  // namespace rswa
