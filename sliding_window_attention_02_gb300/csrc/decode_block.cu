// R-SWA decode of a block of k consecutive output tokens per sequence.
//
// Output t_b + i (i = 0..k-1) attends to the prefix, to the outputs of its
// window already in the cache, j in [max(0, t_b + i - n + 1), t_b), and to
// the block tokens of its window, i' in [max(0, i - n + 1), i].  The
// attention kernel reads the ring before any slot is overwritten.  On the
// CUDA cores (blocks under 64 tokens) it also appends: the ring of KV head
// (b, kv) is read only by the CTAs of its query heads, so the last of them
// to finish (an arrival counter) stores the block's last keys and values of
// that KV head in the ring and advances t_b of those query heads
// (append_block_group).  After the tensor-core kernel (block_tc.cu) a
// separate append kernel runs, waiting on its completion: there one CTA per
// kept token moves the up to 2 n rows faster than the last CTA of a head
// would (26.8 against 28.7 us for 256 tokens on the single-page cache).
// This is the shape of a speculative-verification forward or of chunked
// prefill of output text into an existing cache.
#include <algorithm>

#include "attend.cuh"

namespace rswa {

// The last of the `ctas` CTAs that read the ring of KV head (b, kv) in this
// launch (counted on the (b, h) counter of the group's first query head)
// stores the block's last kw = min(k, n) keys and values of that KV head in
// ring slots (t_b + i) mod n, i = k - kw .. k - 1 (earlier tokens of a longer
// block would be evicted by later ones), then advances t_b of the group's
// query heads by k and rearms the counter.  Every CTA of the group read t_b
// before its arrival.  Called by every thread of the CTA after a barrier
// that follows the CTA's last read of the ring; each CTA arrives once, also
// after a wait that gave up, so the ring always receives the block.
template <typename T, int D>
__device__ __forceinline__ void append_block_group(const CacheView& cv, const T* kblk,
                                                   const T* vblk, int64_t k, int b, int kv,
                                                   int64_t t_b, int ctas, int tid,
                                                   int nthreads) {
  __shared__ int s_last_grp;
  const int per_kv = cv.H / cv.Hkv;
  int32_t* cnt = cv.cnt_bh + (size_t)b * cv.H + (size_t)kv * per_kv;
  if (tid == 0) s_last_grp = arrive_acq_rel(cnt) == ctas - 1;
  __syncthreads();
  if (!s_last_grp) return;
  const int64_t kw = min(k, cv.n);
  constexpr int NV = D * (int)sizeof(T) / 16;           // 16-byte pieces of a row
  const size_t slab = ((size_t)b * cv.Hkv + kv) * cv.slab_rows + cv.m_cap;
  for (int64_t x = tid; x < 2 * kw * NV; x += nthreads) {
    const int isv = x >= kw * NV;
    const int64_t y = x - isv * kw * NV;
    const int64_t i = k - kw + y / NV;
    const int vi = (int)(y % NV);
    const T* in = (isv ? vblk : kblk) + (((size_t)b * k + i) * cv.Hkv + kv) * D;
    T* out = static_cast<T*>(isv ? cv.V : cv.K) + (slab + (size_t)((t_b + i) % cv.n)) * D;
    reinterpret_cast<uint4*>(out)[vi] = reinterpret_cast<const uint4*>(in)[vi];
  }
  if (tid == 0) {
    for (int g = 0; g < per_kv; ++g) cv.t_dev[(size_t)b * cv.H + (size_t)kv * per_kv + g] = t_b + k;
    *cnt = 0;
  }
}

// One CTA of NW warps per (b, i, h): the warps split every key segment of
// query i (prefix, cached outputs of its window, block tokens 0..i) between
// them, NW * KEYS_WARP rows per round, and merge in shared memory.  8 warps
// in general; 16 (one CTA per SM) when the grid fits one wave of the
// device's SMs, so that each query takes half as many dependent row batches.
// PREFETCH: the preceding kernel of the stream writes no prefix row and no
// m_b of this cache (the host's per-handle flag), so each warp reads m_b and
// loads its first batch of prefix rows before the dependency wait.
constexpr int kBlockWarps = 8;
constexpr int kBlockWarpsWide = 16;

template <typename T, int D, int NW, bool PREFETCH>
__global__ void __launch_bounds__(NW * 32)
decode_block_kernel(CacheView cv, const T* __restrict__ q,
                    const T* __restrict__ kblk, const T* __restrict__ vblk,
                    int64_t k, T* __restrict__ o, float* __restrict__ lse) {
  using C = AttendCfg<T, D>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.y;
  const int64_t qi = blockIdx.x;                         // i * H + h
  const int64_t i = qi / cv.H;
  const int h = (int)(qi % cv.H);
  const size_t bh = (size_t)b * cv.H + h;
  const int kvh = h / (cv.H / cv.Hkv);
  const size_t bkv = (size_t)b * cv.Hkv + kvh;
  const int64_t first = (int64_t)warp * C::KEYS_WARP;
  const int64_t step = (int64_t)NW * C::KEYS_WARP;
  const T* Kb = static_cast<const T*>(cv.K) + bkv * cv.slab_rows * D;
  const T* Vb = static_cast<const T*>(cv.V) + bkv * cv.slab_rows * D;
  int64_t m_b = 0;
  AttendBatch<T, D> pre;
  bool have_pre = false;
  if (PREFETCH) {
    m_b = cv.m_dev[b];
    if (first < m_b) {
      attend_load<T, D>(Kb, Vb, D, first, 0, m_b, -1, nullptr, nullptr, lane, INT64_MAX,
                        0, pre);
      have_pre = true;
    }
  }
  griddep_wait();
  griddep_launch_dependents();
  if (!PREFETCH) m_b = cv.m_dev[b];
  const int64_t t_b = cv.t_dev[bh];
  const int64_t n = cv.n;
  const int64_t row_stride = (int64_t)cv.Hkv * D;        // k, v: [B][k][Hkv][D]
  const size_t qrow = ((size_t)b * k + i) * cv.H + h;    // q, o: [B][k][H][D]

  float qf[C::EPL];
  load_q_frag<T, D>(q + qrow * D, lane, qf);
  SoftmaxState<C::EPL> st;
  st.init();
  // prefix (the first batch already loaded with PREFETCH)
  if (have_pre) attend_consume<T, D>(qf, pre, st);
  attend_range<T, D>(qf, Kb, Vb, D, 0, m_b, have_pre ? first + step : first, step, -1,
                     nullptr, nullptr,
                     lane, st);
  // cached outputs of the window: j in [j_lo, t_b), slot j mod n
  const int64_t j_lo = max((int64_t)0, t_b + i - n + 1);
  if (j_lo < t_b) {
    const T* Kr = Kb + cv.m_cap * D;
    const T* Vr = Vb + cv.m_cap * D;
    const int64_t a = j_lo % n, cnt = t_b - j_lo;
    const int64_t first_end = min(n, a + cnt);
    attend_range<T, D>(qf, Kr, Vr, D, a, first_end, first, step, -1, nullptr,
                       nullptr, lane, st);
    if (a + cnt > n)
      attend_range<T, D>(qf, Kr, Vr, D, 0, a + cnt - n, first, step, -1, nullptr,
                         nullptr, lane, st);
  }
  // block tokens of the window, max(0, i - n + 1) .. i (rows of the input,
  // stride H_kv * D)
  const T* Kk = kblk + ((size_t)b * k * cv.Hkv + kvh) * D;
  const T* Vk = vblk + ((size_t)b * k * cv.Hkv + kvh) * D;
  attend_range<T, D>(qf, Kk, Vk, row_stride, max((int64_t)0, i - n + 1), i + 1,
                     first, step, -1, nullptr, nullptr, lane, st);
  merge_groups<T, D>(st);
  __shared__ float s_m[NW], s_l[NW];
  __shared__ float s_acc[NW][D];
  if (lane < C::LPK) {
#pragma unroll
    for (int e = 0; e < C::EPL; ++e) s_acc[warp][lane * C::EPL + e] = st.acc[e];
    if (lane == 0) {
      s_m[warp] = st.m;
      s_l[warp] = st.l;
    }
  }
  __syncthreads();
  const int tid = threadIdx.x;
  if (tid < D) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, s_m[w]);
    const float ref = (M == -INFINITY) ? 0.f : M;
    float L = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float sc = fast_exp2(s_m[w] - ref);
      L += s_l[w] * sc;
      A += s_acc[w][tid] * sc;
    }
    o[qrow * D + tid] = (T)(A / L);          // self is always visible: L > 0
    if (tid == 0 && lse) lse[qrow] = (ref + log2f(L)) * kLn2;
  }
  // Every load of this CTA (ring slots included) has been consumed above.
  __syncthreads();
  append_block_group<T, D>(cv, kblk, vblk, k, b, kvh, t_b,
                           (int)k * (cv.H / cv.Hkv), tid, blockDim.x);
}

// One CTA per kept block token and sequence: the last kw = min(k, n) tokens
// i = k - kw + blockIdx.x go to ring slot (t_b + i) mod n for every KV head
// (earlier tokens of a longer block would be evicted by later ones).  Each
// CTA reads t_b before it counts itself done on the sequence's counter; the
// last of the kw CTAs sets t_b += k for every query head and rearms the
// counter.  The writes wait for the attention kernel (programmatic dependent
// launch), which reads slots that block tokens overwrite.
template <typename T, int D>
__global__ void __launch_bounds__(128)
append_block_kernel(CacheView cv, const T* __restrict__ kblk,
                    const T* __restrict__ vblk, int k) {
  griddep_wait();
  const int kw = (int)min((int64_t)k, cv.n);
  const int i = k - kw + blockIdx.x, b = blockIdx.y;
  const int Hkv = cv.Hkv;                        // k, v carry the KV heads
  const int64_t t_b = cv.t_dev[(size_t)b * cv.H];
  constexpr int NV = D * (int)sizeof(T) / 16;
  const int per_kv = Hkv * NV;
  const size_t slot = (size_t)((t_b + i) % cv.n);
  const size_t in_row = ((size_t)b * k + i) * Hkv;
  for (int x = threadIdx.x; x < 2 * per_kv; x += blockDim.x) {
    const int kv = x >= per_kv;
    const int r = x - kv * per_kv;
    const int h = r / NV, vi = r % NV;
    const T* in = (kv ? vblk : kblk) + (in_row + h) * D;
    T* out = static_cast<T*>(kv ? cv.V : cv.K) +
             (((size_t)b * Hkv + h) * cv.slab_rows + cv.m_cap + slot) * D;
    reinterpret_cast<uint4*>(out)[vi] = reinterpret_cast<const uint4*>(in)[vi];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    int32_t* cnt = cv.cnt_bh + (size_t)b * cv.H;
    if (atomicAdd(cnt, 1) == kw - 1) {
      __threadfence();
      for (int h = 0; h < cv.H; ++h) cv.t_dev[(size_t)b * cv.H + h] = t_b + k;
      *cnt = 0;
    }
  }
}

// Programmatic stream serialization: a kernel may begin launching while the
// previous kernel of the stream drains; each one waits (griddepcontrol) before
// it touches memory that the previous one writes.
template <typename K, typename... Args>
static cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename T, int D, bool PF>
static cudaError_t launch_block_cc(const CacheView& cv, const void* q, const void* k,
                                   const void* v, int64_t block, void* o, float* lse,
                                   cudaStream_t s) {
  const int64_t nq = block * cv.H;
  const dim3 grid((unsigned)nq, (unsigned)cv.B);
  return nq * cv.B <= cv.sms
             ? launch_pdl(decode_block_kernel<T, D, kBlockWarpsWide, PF>, grid,
                          dim3(kBlockWarpsWide * 32), s, cv, (const T*)q, (const T*)k,
                          (const T*)v, block, (T*)o, lse)
             : launch_pdl(decode_block_kernel<T, D, kBlockWarps, PF>, grid,
                          dim3(kBlockWarps * 32), s, cv, (const T*)q, (const T*)k,
                          (const T*)v, block, (T*)o, lse);
}

template <typename T, int D>
static cudaError_t launch_block_t(const CacheView& cv, const void* q,
                                  const void* k, const void* v, int64_t block,
                                  void* o, float* lse, bool prefetch, cudaStream_t s) {
  cudaError_t e;
  if (block_tc_supported(cv, block)) {
    e = launch_block_tc(cv, q, k, v, block, o, lse, s);
    if (e != cudaSuccess) return e;
    const int64_t kw = std::min<int64_t>(block, cv.n);
    return launch_pdl(append_block_kernel<T, D>, dim3((unsigned)kw, (unsigned)cv.B),
                      dim3(128), s, cv, (const T*)k, (const T*)v, (int)block);
  } else {
    e = prefetch ? launch_block_cc<T, D, true>(cv, q, k, v, block, o, lse, s)
                 : launch_block_cc<T, D, false>(cv, q, k, v, block, o, lse, s);
  }
  return e;
}

cudaError_t launch_decode_block(const CacheView& cv, const void* q, const void* k,
                                const void* v, int64_t block, void* o, float* lse,
                                bool prefetch, cudaStream_t s) {
  if (cv.dtype == RSWA_F32) {
    if (cv.d == 64)
      return launch_block_t<float, 64>(cv, q, k, v, block, o, lse, prefetch, s);
    return launch_block_t<float, 128>(cv, q, k, v, block, o, lse, prefetch, s);
  }
  if (cv.d == 64)
    return launch_block_t<__nv_bfloat16, 64>(cv, q, k, v, block, o, lse, prefetch, s);
  return launch_block_t<__nv_bfloat16, 128>(cv, q, k, v, block, o, lse, prefetch, s);
}

}  // namespace rswa
