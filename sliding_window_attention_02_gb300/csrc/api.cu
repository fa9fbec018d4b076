// Host side of the C ABI: validation, cache layout, handle registry and
// kernel dispatch.  No exception crosses the ABI; every entry point returns
// an rswa_status.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <new>
#include <unordered_set>
#include <vector>

#include "rswa_internal.h"

using namespace rswa;

struct rswa_cache {
  CacheView cv;
  int device;
  void* buf;
  size_t buf_bytes;
  // False from creation and after every prefill or t restore until the next
  // decode launch: the launch right after one of those must not read prefix
  // rows or m_b before its dependency wait, later decode launches may.
  std::atomic<bool> prefix_stable{false};
};

namespace {

std::mutex g_mu;
std::unordered_set<rswa_cache*> g_live;
std::atomic<int> g_fail_next{0};
std::atomic<uint64_t> g_wait_limit_ns{0};      // 0: the default bound

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool live(rswa_cache* c) {
  std::lock_guard<std::mutex> lk(g_mu);
  return c != nullptr && g_live.count(c) != 0;
}

// Test hook: simulated CUDA failure before anything is launched.
bool injected_failure() {
  int v = g_fail_next.load();
  while (v > 0) {
    if (g_fail_next.compare_exchange_weak(v, v - 1)) return true;
  }
  return false;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? RSWA_OK : RSWA_ECUDA; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Makes the cache's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
      return;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev)
      cudaSetDevice(prev);
  }
};

// Runs a decode launch with the handle's permission to read prefix rows and
// m_b before the dependency wait.  Only a launch that succeeded counts as the
// decode launch that follows a prefill: when no kernel was launched, the next
// decode call must still wait before it reads them.
template <typename F>
int run_decode(rswa_cache* cache, F launch) {
  const bool prefetch = cache->prefix_stable.load();
  const cudaError_t e = launch(prefetch);
  if (e == cudaSuccess) cache->prefix_stable.store(true);
  return status_of(e);
}

struct Layout {
  size_t m_off, t_off, err_off, k_off, v_off, part_off, cnt_bh_off;
  size_t total;
  int chunk, max_chunks, part_slots;
};

int valid_shape(int64_t m, int64_t n, int heads, int kv_heads, int head_dim,
                int batch, int dtype) {
  if (dtype != RSWA_F32 && dtype != RSWA_BF16) return RSWA_EDTYPE;
  if (head_dim != 64 && head_dim != 128) return RSWA_EDTYPE;
  if (m < 0 || n < 1 || heads < 1 || kv_heads < 1 || batch < 1) return RSWA_EINVAL;
  if (heads % kv_heads != 0) return RSWA_EINVAL;
  if (m > (int64_t(1) << 30) || n > (int64_t(1) << 30)) return RSWA_EINVAL;
  if (heads > 4096 || batch > (1 << 20)) return RSWA_EINVAL;
  return RSWA_OK;
}

#ifndef RSWA_DECODE_CTAS_PER_SM
#define RSWA_DECODE_CTAS_PER_SM 32
#endif

// Keys per decode CTA, a power of two, for a device of `sms` SMs.  Many
// heads (more than the SMs): sized so that the largest possible decode grid
// holds about RSWA_DECODE_CTAS_PER_SM CTAs per SM.  Few heads: about 40
// chunks per head, 128..256 keys each (measured best on GB300 for one
// sequence with a 1K-10K key cache; shorter caches take the cluster path).
// Never below kMinChunk, which bounds the split-K scratch.
#ifndef RSWA_TC_WAVES
#define RSWA_TC_WAVES 2
#endif

constexpr int kMinChunk = 64;

int choose_chunk(int64_t m, int64_t n, int heads, int kv_heads, int head_dim,
                 int dtype, int batch, int sms) {
#ifdef RSWA_DECODE_CHUNK
  static_assert(RSWA_DECODE_CHUNK >= kMinChunk, "decode chunk");
  return RSWA_DECODE_CHUNK;
#endif
  if (gqa_tc_shape(heads, kv_heads, head_dim, dtype)) {
    // Tensor-core grouped decode: one CTA per chunk of a KV head, two
    // resident per SM; chunks are whole 128-key tiles, sized for about
    // RSWA_TC_WAVES waves of CTAs.
    const int64_t keys = (int64_t)batch * kv_heads * (m + n);
    const int64_t target = (int64_t)sms * 2 * RSWA_TC_WAVES;
    const int64_t want = (keys + target - 1) / target;
    int c = 128;
    while (c < want && c < 2048) c <<= 1;
    return c;
  }
  if ((int64_t)batch * heads <= sms) {
    const int64_t want = (m + n + 39) / 40;
    int c = 128;
    while (c < want && c < 256) c <<= 1;
    return c;
  }
  // one CTA per chunk of one K/V stream; a grouped kernel streams each KV
  // head once per group of query heads.  The largest power of two (128 to
  // 2048) within 1.5 x the wanted keys per CTA: on GB300 the batched step
  // (287 wanted) runs 59.5 us with 256-key chunks against 61.9 with 512, the
  // long-output sweep (180) is best at 256 (67.7 with 128), and a
  // 128-key-per-head cache keeps one 128-key chunk per head (40.5 us with
  // 64-key chunks against 30.0).
  const int streams = heads / gqa_heads_per_cta(heads, kv_heads);
  const int64_t keys = (int64_t)batch * streams * (m + n);
  const int64_t target = (int64_t)sms * RSWA_DECODE_CTAS_PER_SM;
  const int64_t want = (keys + target - 1) / target;
  int c = 128;
  while (2 * (int64_t)c <= want * 3 / 2 && c < 2048) c <<= 1;
  return c;
}

// Layout of a cache buffer.  The decode chunk depends on the device's SM
// count (`sms`, 0 when no device is known: footprint queries); the split-K
// scratch is sized for the smallest chunk, so the footprint is the same for
// every device.
Layout make_layout(int64_t m, int64_t n, int heads, int kv_heads, int head_dim,
                   int batch, int dtype, int sms) {
  Layout L{};
  const size_t elt = dtype == RSWA_F32 ? 4 : 2;
  L.chunk = sms > 0 ? choose_chunk(m, n, heads, kv_heads, head_dim, dtype, batch, sms)
                    : kMinChunk;
  L.max_chunks = (int)((m + L.chunk - 1) / L.chunk + (n + L.chunk - 1) / L.chunk);
  const int64_t chunks_bound = (m + kMinChunk - 1) / kMinChunk +
                               (n + kMinChunk - 1) / kMinChunk;
  L.part_slots = (int)std::min<int64_t>(chunks_bound, INT32_MAX);
  size_t off = 0;
  L.m_off = off;      off = align_up(off + sizeof(int32_t) * batch);
  L.t_off = off;      off = align_up(off + sizeof(int64_t) * batch * heads);
  L.err_off = off;    off = align_up(off + sizeof(int32_t));
  L.cnt_bh_off = off; off = align_up(off + sizeof(int32_t) * batch * heads);
  const size_t state_end = off;
  (void)state_end;
  L.k_off = off;
  off = align_up(off + elt * (size_t)batch * kv_heads * (size_t)(m + n) * head_dim);
  L.v_off = off;
  off = align_up(off + elt * (size_t)batch * kv_heads * (size_t)(m + n) * head_dim);
  L.part_off = off;
  off = align_up(off + sizeof(float) * (size_t)batch * heads * chunks_bound *
                           (head_dim + 2));
  L.total = off;
  return L;
}

}  // namespace

uint64_t rswa::phase_wait_limit_ns() {
  const uint64_t ns = g_wait_limit_ns.load();
  return ns ? ns : 1000000000ull;
}

extern "C" {

const char* rswa_strerror(int status) {
  switch (status) {
    case RSWA_OK: return "ok";
    case RSWA_EINVAL: return "invalid argument";
    case RSWA_ECAPACITY: return "capacity exceeded (prefix longer than the cache's prefix capacity, or buffer too small)";
    case RSWA_EDTYPE: return "unsupported dtype or head_dim";
    case RSWA_EHANDLE: return "invalid or destroyed cache handle";
    case RSWA_ECUDA: return "CUDA error";
    case RSWA_EDEVICE: return "device-side error flagged by a kernel";
    default: return "unknown status";
  }
}

void rswa_debug_fail_next_cuda(int count) { g_fail_next.store(count < 0 ? 0 : count); }

void rswa_debug_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns); }

int rswa_cache_footprint_gqa(int64_t m, int64_t n, int heads, int kv_heads,
                             int head_dim, int batch, int dtype,
                             size_t* out_bytes) {
  if (!out_bytes) return RSWA_EINVAL;
  const int st = valid_shape(m, n, heads, kv_heads, head_dim, batch, dtype);
  if (st != RSWA_OK) return st;
  *out_bytes = make_layout(m, n, heads, kv_heads, head_dim, batch, dtype, 0).total;
  return RSWA_OK;
}

int rswa_cache_footprint(int64_t m, int64_t n, int heads, int head_dim,
                         int batch, int dtype, size_t* out_bytes) {
  return rswa_cache_footprint_gqa(m, n, heads, heads, head_dim, batch, dtype,
                                  out_bytes);
}

int rswa_cache_create(int64_t m, int64_t n, int heads, int head_dim, int batch,
                      int dtype, void* device_buf, size_t buf_bytes,
                      rswa_cache** out) {
  return rswa_cache_create_gqa(m, n, heads, heads, head_dim, batch, dtype,
                               device_buf, buf_bytes, out);
}

int rswa_cache_create_gqa(int64_t m, int64_t n, int heads, int kv_heads,
                          int head_dim, int batch, int dtype, void* device_buf,
                          size_t buf_bytes, rswa_cache** out) {
  if (!out) return RSWA_EINVAL;
  *out = nullptr;
  const int st = valid_shape(m, n, heads, kv_heads, head_dim, batch, dtype);
  if (st != RSWA_OK) return st;
  if (!device_buf || (reinterpret_cast<uintptr_t>(device_buf) % kAlign) != 0)
    return RSWA_EINVAL;
  if (buf_bytes < make_layout(m, n, heads, kv_heads, head_dim, batch, dtype, 0).total)
    return RSWA_ECAPACITY;
  if (injected_failure()) return RSWA_ECUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms < 1)
    return RSWA_ECUDA;
  const Layout L = make_layout(m, n, heads, kv_heads, head_dim, batch, dtype, sms);

  rswa_cache* c = new (std::nothrow) rswa_cache();
  if (!c) return RSWA_ECUDA;
  char* base = static_cast<char*>(device_buf);
  CacheView& cv = c->cv;
  cv.K = base + L.k_off;
  cv.V = base + L.v_off;
  cv.m_dev = reinterpret_cast<int32_t*>(base + L.m_off);
  cv.t_dev = reinterpret_cast<int64_t*>(base + L.t_off);
  cv.err = reinterpret_cast<int32_t*>(base + L.err_off);
  cv.part = reinterpret_cast<float*>(base + L.part_off);
  cv.cnt_bh = reinterpret_cast<int32_t*>(base + L.cnt_bh_off);
  cv.B = batch;
  cv.H = heads;
  cv.Hkv = kv_heads;
  cv.d = head_dim;
  cv.dtype = dtype;
  cv.m_cap = m;
  cv.n = n;
  cv.slab_rows = m + n;
  cv.chunk = L.chunk;
  cv.max_chunks = L.max_chunks;
  cv.sms = sms;
  cv.part_slots = L.part_slots;
  c->device = dev;
  c->buf = device_buf;
  c->buf_bytes = buf_bytes;
  // Zero the state words (m_b, t_b, error flag, counters) and the K/V
  // slabs: rows no prefill or append has written yet then hold zeros, and
  // a tensor-core tile that reaches past the rows it attends (masked, p = 0)
  // multiplies finite values only.
  cudaError_t e = cudaMemsetAsync(device_buf, 0, L.part_off, 0);
  if (e == cudaSuccess) e = cudaStreamSynchronize(0);
  if (e != cudaSuccess) {
    delete c;
    return RSWA_ECUDA;
  }
  {
    std::lock_guard<std::mutex> lk(g_mu);
    g_live.insert(c);
  }
  *out = c;
  return RSWA_OK;
}

int rswa_cache_destroy(rswa_cache* cache) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!cache || g_live.erase(cache) == 0) return RSWA_EHANDLE;
  }
  delete cache;
  return RSWA_OK;
}

int rswa_prefill_varlen(rswa_cache* cache, const void* Q, const void* K,
                        const void* V, void* O, const int64_t* m_per_seq,
                        const int64_t* t_per_seq, void* stream) {
  if (!live(cache)) return RSWA_EHANDLE;
  const CacheView& cv = cache->cv;
  if (!m_per_seq || !t_per_seq) return RSWA_EINVAL;
  int64_t total_rows = 0;
  for (int b = 0; b < cv.B; ++b) {
    if (m_per_seq[b] < 0 || t_per_seq[b] < 0 || t_per_seq[b] > (int64_t(1) << 40))
      return RSWA_EINVAL;
    if (m_per_seq[b] > cv.m_cap) return RSWA_ECAPACITY;
    total_rows += m_per_seq[b] + t_per_seq[b];
  }
  // With no rows at all (every m_b = 0 and T_b = 0) the tensors may be NULL.
  if (total_rows > 0 && (!K || !V)) return RSWA_EINVAL;
  if (O && !Q) return RSWA_EINVAL;
  if (!aligned16(K) || !aligned16(V) || (Q && !aligned16(Q)) ||
      (O && !aligned16(O)))
    return RSWA_EINVAL;
  if (injected_failure()) return RSWA_ECUDA;
  DeviceGuard g(cache->device);
  if (!g.ok) return RSWA_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  int64_t row = 0;
  // The next decode launch follows kernels that write the prefix and m_b.
  cache->prefix_stable.store(false);
  for (int b0 = 0; b0 < cv.B; b0 += kMaxSeqPerLaunch) {
    SeqTable st{};
    st.seq0 = b0;
    st.nseq = std::min(kMaxSeqPerLaunch, cv.B - b0);
    int64_t max_rows = 0, rows = 0;
    int32_t tiles = 0;
    st.tile_off[0] = 0;
    for (int i = 0; i < st.nseq; ++i) {
      const int64_t mb = m_per_seq[b0 + i], tb = t_per_seq[b0 + i];
      st.m[i] = (int32_t)mb;
      st.T[i] = tb;
      st.row_off[i] = row + rows;
      rows += mb + tb;
      max_rows = std::max(max_rows, mb + std::min(cv.n, tb));
      tiles += (int32_t)((mb + tb + 127) / 128);
      st.tile_off[i + 1] = tiles;
    }
    cudaError_t e = launch_prefill_cache(cv, st, K, V, max_rows, s);
    if (e != cudaSuccess) return RSWA_ECUDA;
    if (O && rows > 0) {
      if (prefill_tc_supported(cv))
        e = launch_prefill_tc(cv, st, Q, K, V, O, rows, s);
      else
        e = launch_prefill_rowwise(cv, st, Q, K, V, O, rows, s);
      if (e != cudaSuccess) return RSWA_ECUDA;
    }
    row += rows;
  }
  return RSWA_OK;
}

int rswa_prefill(rswa_cache* cache, const void* Q, const void* K,
                 const void* V, void* O, const int64_t* m_per_seq, int64_t T,
                 void* stream) {
  if (!live(cache)) return RSWA_EHANDLE;
  if (T < 0) return RSWA_EINVAL;
  std::vector<int64_t> t_per_seq((size_t)cache->cv.B, T);
  return rswa_prefill_varlen(cache, Q, K, V, O, m_per_seq, t_per_seq.data(),
                             stream);
}

int rswa_append_kv(rswa_cache* cache, const void* k, const void* v,
                   void* stream) {
  if (!live(cache)) return RSWA_EHANDLE;
  if (!k || !v || !aligned16(k) || !aligned16(v)) return RSWA_EINVAL;
  if (injected_failure()) return RSWA_ECUDA;
  DeviceGuard g(cache->device);
  if (!g.ok) return RSWA_ECUDA;
  return status_of(launch_append(cache->cv, k, v, static_cast<cudaStream_t>(stream)));
}

int rswa_decode_step(rswa_cache* cache, const void* q, void* o, float* lse,
                     void* stream) {
  if (!live(cache)) return RSWA_EHANDLE;
  if (!q || !o || !aligned16(q)) return RSWA_EINVAL;
  if (injected_failure()) return RSWA_ECUDA;
  DeviceGuard g(cache->device);
  if (!g.ok) return RSWA_ECUDA;
  return run_decode(cache, [&](bool pf) {
    return launch_decode(cache->cv, q, nullptr, nullptr, o, lse, false, pf,
                         static_cast<cudaStream_t>(stream));
  });
}

int rswa_decode_step_fused(rswa_cache* cache, const void* q, const void* k,
                           const void* v, void* o, float* lse, void* stream) {
  if (!live(cache)) return RSWA_EHANDLE;
  if (!q || !k || !v || !o || !aligned16(q) || !aligned16(k) || !aligned16(v))
    return RSWA_EINVAL;
  if (injected_failure()) return RSWA_ECUDA;
  DeviceGuard g(cache->device);
  if (!g.ok) return RSWA_ECUDA;
  return run_decode(cache, [&](bool pf) {
    return launch_decode(cache->cv, q, k, v, o, lse, true, pf,
                         static_cast<cudaStream_t>(stream));
  });
}

int rswa_decode_block(rswa_cache* cache, const void* q, const void* k,
                      const void* v, int64_t block, void* o, float* lse,
                      void* stream) {
  if (!live(cache)) return RSWA_EHANDLE;
  // grid limits of the block kernels: B sequences on grid.y, block * H
  // queries on grid.x
  if (block < 1 || block > (int64_t(1) << 24) || cache->cv.B > 65535 ||
      block * cache->cv.H >= (int64_t(1) << 31))
    return RSWA_EINVAL;
  if (!q || !k || !v || !o || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
      !aligned16(o))
    return RSWA_EINVAL;
  if (injected_failure()) return RSWA_ECUDA;
  DeviceGuard g(cache->device);
  if (!g.ok) return RSWA_ECUDA;
  if (block == 1)  // [B][1][H][d] is the fused single step's [B][H][d]
    return run_decode(cache, [&](bool pf) {
      return launch_decode(cache->cv, q, k, v, o, lse, true, pf,
                           static_cast<cudaStream_t>(stream));
    });
  return run_decode(cache, [&](bool pf) {
    return launch_decode_block(cache->cv, q, k, v, block, o, lse, pf,
                               static_cast<cudaStream_t>(stream));
  });
}

int rswa_decode_step_fused_static(rswa_cache* cache, const void* q,
                                  const void* k, const void* v, void* o,
                                  float* lse, void* stream) {
  if (!live(cache)) return RSWA_EHANDLE;
  if (!q || !k || !v || !o || !aligned16(q) || !aligned16(k) || !aligned16(v))
    return RSWA_EINVAL;
  size_t part_bytes = 0, cnt_bytes = 0;
  if (static_scratch_need(cache->cv, &part_bytes, &cnt_bytes) >
      static_scratch_capacity())
    return RSWA_ECAPACITY;
  if (injected_failure()) return RSWA_ECUDA;
  DeviceGuard g(cache->device);
  if (!g.ok) return RSWA_ECUDA;
  return run_decode(cache, [&](bool pf) {
    return launch_decode_fused_static(cache->cv, cache->device, q, k, v, o, lse,
                                      pf, static_cast<cudaStream_t>(stream));
  });
}

static int read_state(rswa_cache* cache, int b, int64_t* m_b, int64_t* t_b) {
  if (!live(cache)) return RSWA_EHANDLE;
  if (b < 0 || b >= cache->cv.B) return RSWA_EINVAL;
  if (injected_failure()) return RSWA_ECUDA;
  DeviceGuard g(cache->device);
  if (!g.ok) return RSWA_ECUDA;
  int32_t m32 = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return RSWA_ECUDA;
  if (cudaMemcpy(&m32, cache->cv.m_dev + b, sizeof(m32), cudaMemcpyDeviceToHost) !=
          cudaSuccess ||
      cudaMemcpy(t_b, cache->cv.t_dev + (size_t)b * cache->cv.H, sizeof(*t_b),
                 cudaMemcpyDeviceToHost) !=
          cudaSuccess)
    return RSWA_ECUDA;
  *m_b = m32;
  return RSWA_OK;
}

int rswa_cache_len(rswa_cache* cache, int b, int64_t* out) {
  if (!out) return RSWA_EINVAL;
  int64_t m_b, t_b;
  const int st = read_state(cache, b, &m_b, &t_b);
  if (st != RSWA_OK) return st;
  *out = m_b + std::min(cache->cv.n, t_b);
  return RSWA_OK;
}

int rswa_cache_get_t(rswa_cache* cache, int b, int64_t* out) {
  if (!out) return RSWA_EINVAL;
  int64_t m_b, t_b;
  const int st = read_state(cache, b, &m_b, &t_b);
  if (st != RSWA_OK) return st;
  *out = t_b;
  return RSWA_OK;
}

int rswa_cache_bytes(rswa_cache* cache, int b, size_t* out) {
  if (!out) return RSWA_EINVAL;
  int64_t len = 0;
  const int st = rswa_cache_len(cache, b, &len);
  if (st != RSWA_OK) return st;
  const size_t elt = cache->cv.dtype == RSWA_F32 ? 4 : 2;
  *out = (size_t)len * cache->cv.Hkv * cache->cv.d * 2 * elt;
  return RSWA_OK;
}

int rswa_cache_set_t(rswa_cache* cache, const int64_t* t_per_seq, void* stream) {
  if (!live(cache)) return RSWA_EHANDLE;
  if (!t_per_seq) return RSWA_EINVAL;
  for (int b = 0; b < cache->cv.B; ++b)
    if (t_per_seq[b] < 0) return RSWA_EINVAL;
  if (injected_failure()) return RSWA_ECUDA;
  DeviceGuard g(cache->device);
  if (!g.ok) return RSWA_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cache->prefix_stable.store(false);
  if (launch_set_t(cache->cv, t_per_seq, s) != cudaSuccess) return RSWA_ECUDA;
  // The copy source is pageable host memory: finish before returning so the
  // caller may release it.
  return status_of(cudaStreamSynchronize(s));
}

int rswa_cache_kv_offsets(rswa_cache* cache, size_t* k_offset,
                          size_t* v_offset) {
  if (!live(cache)) return RSWA_EHANDLE;
  if (!k_offset || !v_offset) return RSWA_EINVAL;
  const char* base = static_cast<const char*>(cache->buf);
  *k_offset = (size_t)(static_cast<const char*>(cache->cv.K) - base);
  *v_offset = (size_t)(static_cast<const char*>(cache->cv.V) - base);
  return RSWA_OK;
}

int rswa_sync_status(rswa_cache* cache) {
  if (!live(cache)) return RSWA_EHANDLE;
  if (injected_failure()) return RSWA_ECUDA;
  DeviceGuard g(cache->device);
  if (!g.ok) return RSWA_ECUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return RSWA_ECUDA;
  int32_t flag = 0;
  if (cudaMemcpy(&flag, cache->cv.err, sizeof(flag), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return RSWA_ECUDA;
  if (flag != 0) {
    const int32_t zero = 0;
    if (cudaMemcpy(cache->cv.err, &zero, sizeof(zero), cudaMemcpyHostToDevice) !=
        cudaSuccess)
      return RSWA_ECUDA;
    return RSWA_EDEVICE;
  }
  return RSWA_OK;
}

}  // extern "C"
