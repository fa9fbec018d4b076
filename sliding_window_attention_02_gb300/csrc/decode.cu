// R-SWA decode step: split-K over the cache with a log-sum-exp combine.
//
// Grid (max_chunks, H, B).  The keys of sequence b are the prefix rows
// 0..m_b-1 of its slab and the filled ring slots; CTA c of (b, h) takes
// prefix chunk c (c < ceil(m_b / chunk)) or ring chunk c - ceil(m_b / chunk).
// The number of CTAs per (b, h) depends on m_b only - never on t_b - so a
// fused step may advance t_b while late CTAs of the same launch still start.
//
// Every CTA publishes (m, l, acc[d]) for its chunk; the last CTA of (b, h) to
// arrive (atomic counter, no waiting) merges the partials and writes o and
// lse.  Per-step cost is m_b + min(n, t_b) keys: flat in t_b once t_b >= n
// ("Unlimited OCR", GeekNews, kernel analysis).
#include "attend.cuh"

namespace rswa {

template <typename T, int D, bool FUSED>
__global__ void __launch_bounds__(kDecodeThreads)
decode_kernel(CacheView cv, const T* __restrict__ q, const T* __restrict__ knew,
              const T* __restrict__ vnew, T* __restrict__ o,
              float* __restrict__ lse) {
  using C = AttendCfg<T, D>;
  constexpr int NW = kDecodeThreads / 32;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // Launched as a programmatic dependent: wait until the previous kernel in
  // the stream has completed and its writes are visible.
  griddep_wait();

  const int64_t m_b = cv.m_dev[b];
  const int chunk = cv.chunk;
  const int cp = (int)((m_b + chunk - 1) / chunk);
  const int cr = (int)((cv.n + chunk - 1) / chunk);
  const int nch = cp + cr;
  if (c >= nch) return;
  const size_t bh = (size_t)b * cv.H + h;
  const int64_t t_b = cv.t_dev[bh];

  const T* Kb = static_cast<const T*>(cv.K) + bh * cv.slab_rows * D;
  const T* Vb = static_cast<const T*>(cv.V) + bh * cv.slab_rows * D;
  const T* kn = FUSED ? knew + bh * D : nullptr;
  const T* vn = FUSED ? vnew + bh * D : nullptr;

  int64_t j0, j1, sub = -1;
  if (c < cp) {
    j0 = (int64_t)c * chunk;
    j1 = min(j0 + chunk, m_b);
  } else {
    const int64_t s0 = (int64_t)(c - cp) * chunk;
    const int64_t filled = FUSED ? min(cv.n, t_b + 1) : min(cv.n, t_b);
    const int64_t s1 = max(s0, min(s0 + chunk, filled));
    j0 = cv.m_cap + s0;
    j1 = cv.m_cap + s1;
    if (FUSED) {
      const int64_t w = t_b % cv.n;  // slot of the new output
      if (w >= s0 && w < s0 + chunk) {
        sub = cv.m_cap + w;
        // This CTA owns slot w: store the new k, v there.  No CTA of this
        // launch reads slot w from the slab (it reads (knew, vnew) instead).
        T* Kw = static_cast<T*>(cv.K) + (bh * cv.slab_rows + sub) * D;
        T* Vw = static_cast<T*>(cv.V) + (bh * cv.slab_rows + sub) * D;
        constexpr int NV = D * sizeof(T) / 16;
        for (int i = threadIdx.x; i < 2 * NV; i += blockDim.x) {
          if (i < NV)
            reinterpret_cast<uint4*>(Kw)[i] = reinterpret_cast<const uint4*>(kn)[i];
          else
            reinterpret_cast<uint4*>(Vw)[i - NV] =
                reinterpret_cast<const uint4*>(vn)[i - NV];
        }
      }
    }
  }

  float qf[C::EPL];
  load_q_frag<T, D>(q + bh * D, lane, qf);
  SoftmaxState<C::EPL> st;
  st.init();
  attend_range<T, D>(qf, Kb, Vb, D, j0, j1, (int64_t)warp * C::KEYS_WARP,
                     (int64_t)NW * C::KEYS_WARP, sub, kn, vn, lane, st);
  // The next step's kernel may start launching; it waits for this one.
  griddep_launch_dependents();
  merge_groups<T, D>(st);

  // Merge the warps through shared memory.
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
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < NW; ++w) M = fmaxf(M, s_m[w]);
  const float ref = (M == -INFINITY) ? 0.f : M;
  float Ls = 0.f, A = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const float sc = fast_exp2(s_m[w] - ref);
    Ls += s_l[w] * sc;
    if (tid < D) A += s_acc[w][tid] * sc;
  }

  // Publish this chunk's partial (m, l, acc[D]).
  float* P = cv.part + (bh * cv.max_chunks) * (D + 2);
  if (tid < D) P[c * (D + 2) + 2 + tid] = A;
  if (tid == 0) {
    P[c * (D + 2)] = M;
    P[c * (D + 2) + 1] = Ls;
  }
  __threadfence();
  __syncthreads();
  __shared__ int s_last;
  if (tid == 0) s_last = (atomicAdd(&cv.cnt_bh[bh], 1) == nch - 1);
  __syncthreads();
  if (s_last) {
    __threadfence();
    float Mx = -INFINITY;
    for (int k = 0; k < nch; ++k) Mx = fmaxf(Mx, __ldcg(P + k * (D + 2)));
    const float r2 = (Mx == -INFINITY) ? 0.f : Mx;
    float Lt = 0.f, At = 0.f;
    for (int k = 0; k < nch; ++k) {
      const float sc = fast_exp2(__ldcg(P + k * (D + 2)) - r2);
      Lt += __ldcg(P + k * (D + 2) + 1) * sc;
      if (tid < D) At += __ldcg(P + k * (D + 2) + 2 + tid) * sc;
    }
    if (tid < D) o[bh * D + tid] = (T)(Lt > 0.f ? At / Lt : 0.f);
    if (tid == 0) {
      if (lse) lse[bh] = Lt > 0.f ? (r2 + log2f(Lt)) * kLn2 : -INFINITY;
      cv.cnt_bh[bh] = 0;
      // The last CTA of (b, h) advances this head's t_b; every other CTA of
      // (b, h) read it before its own arrival.
      if (FUSED) cv.t_dev[bh] = t_b + 1;
    }
  }
}

// Small-batch decode: one CTA of NW warps per (b, h) streams the prefix and
// the ring as one logical key range, merges its warps in shared memory and
// writes o directly - no partials, no second pass.  Used when the whole cache
// of a head is a few CTA-iterations long and there are few heads in flight,
// where the split-K combine would only add latency.
template <typename T, int D, bool FUSED, int NW>
__global__ void __launch_bounds__(NW * 32)
decode_small_kernel(CacheView cv, const T* __restrict__ q,
                    const T* __restrict__ knew, const T* __restrict__ vnew,
                    T* __restrict__ o, float* __restrict__ lse) {
  using C = AttendCfg<T, D>;
  const int h = blockIdx.x, b = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t bh = (size_t)b * cv.H + h;
  griddep_wait();
  griddep_launch_dependents();
  const int64_t m_b = cv.m_dev[b];
  const int64_t t_b = cv.t_dev[bh];
  const T* Kb = static_cast<const T*>(cv.K) + bh * cv.slab_rows * D;
  const T* Vb = static_cast<const T*>(cv.V) + bh * cv.slab_rows * D;
  const T* kn = FUSED ? knew + bh * D : nullptr;
  const T* vn = FUSED ? vnew + bh * D : nullptr;
  const int64_t filled = FUSED ? min(cv.n, t_b + 1) : min(cv.n, t_b);
  int64_t sub = -1;
  if (FUSED) {
    sub = cv.m_cap + t_b % cv.n;
    T* Kw = static_cast<T*>(cv.K) + (bh * cv.slab_rows + sub) * D;
    T* Vw = static_cast<T*>(cv.V) + (bh * cv.slab_rows + sub) * D;
    constexpr int NV = D * sizeof(T) / 16;
    for (int i = threadIdx.x; i < 2 * NV; i += blockDim.x) {
      if (i < NV)
        reinterpret_cast<uint4*>(Kw)[i] = reinterpret_cast<const uint4*>(kn)[i];
      else
        reinterpret_cast<uint4*>(Vw)[i - NV] = reinterpret_cast<const uint4*>(vn)[i - NV];
    }
  }
  float qf[C::EPL];
  load_q_frag<T, D>(q + bh * D, lane, qf);
  SoftmaxState<C::EPL> st;
  st.init();
  // logical keys 0..m_b-1 -> prefix rows, m_b.. -> ring rows m_cap..
  attend_range<T, D>(qf, Kb, Vb, D, 0, m_b + filled, (int64_t)warp * C::KEYS_WARP,
                     (int64_t)NW * C::KEYS_WARP, sub, kn, vn, lane, st, m_b,
                     cv.m_cap - m_b);
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
    float Ls = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float sc = fast_exp2(s_m[w] - ref);
      Ls += s_l[w] * sc;
      A += s_acc[w][tid] * sc;
    }
    o[bh * D + tid] = (T)(Ls > 0.f ? A / Ls : 0.f);
    if (tid == 0 && lse) lse[bh] = Ls > 0.f ? (ref + log2f(Ls)) * kLn2 : -INFINITY;
  }
  // This CTA is the only reader of its head's t_b (read before the
  // __syncthreads above): advance it.
  if (FUSED && tid == 0) cv.t_dev[bh] = t_b + 1;
}

constexpr int kSmallWarps = 16;

// Launch with programmatic stream serialization so that a decode kernel may
// begin launching while the previous kernel of the stream drains.
template <typename K, typename... Args>
static cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename T, int D>
static cudaError_t launch_decode_t(const CacheView& cv, const void* q,
                                   const void* k, const void* v, void* o,
                                   float* lse, bool fused, cudaStream_t s) {
  const T* qq = (const T*)q;
  const T* kk = (const T*)k;
  const T* vv = (const T*)v;
  T* oo = (T*)o;
  cudaError_t e;
  if (decode_use_small(cv)) {
    dim3 grid(cv.H, cv.B);
    if (fused)
      e = launch_pdl(decode_small_kernel<T, D, true, kSmallWarps>, grid,
                     dim3(kSmallWarps * 32), s, cv, qq, kk, vv, oo, lse);
    else
      e = launch_pdl(decode_small_kernel<T, D, false, kSmallWarps>, grid,
                     dim3(kSmallWarps * 32), s, cv, qq, (const T*)nullptr,
                     (const T*)nullptr, oo, lse);
  } else {
    dim3 grid(cv.max_chunks, cv.H, cv.B);
    if (fused)
      e = launch_pdl(decode_kernel<T, D, true>, grid, dim3(kDecodeThreads), s, cv,
                     qq, kk, vv, oo, lse);
    else
      e = launch_pdl(decode_kernel<T, D, false>, grid, dim3(kDecodeThreads), s, cv,
                     qq, (const T*)nullptr, (const T*)nullptr, oo, lse);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// One CTA per head when every head's cache is at most 4 CTA-iterations of
// keys and all heads fit in one wave of CTAs.
bool decode_use_small(const CacheView& cv) {
  const int64_t keys_per_iter = (int64_t)kSmallWarps * 32 *
                                (cv.dtype == RSWA_F32 ? 4 : 8) / cv.d *
                                RSWA_DECODE_UNROLL;
  return (int64_t)cv.B * cv.H <= 152 && cv.m_cap + cv.n <= 4 * keys_per_iter;
}

cudaError_t launch_decode(const CacheView& cv, const void* q, const void* k,
                          const void* v, void* o, float* lse, bool fused,
                          cudaStream_t s) {
  if (cv.dtype == RSWA_F32) {
    if (cv.d == 64) return launch_decode_t<float, 64>(cv, q, k, v, o, lse, fused, s);
    return launch_decode_t<float, 128>(cv, q, k, v, o, lse, fused, s);
  }
  if (cv.d == 64)
    return launch_decode_t<__nv_bfloat16, 64>(cv, q, k, v, o, lse, fused, s);
  return launch_decode_t<__nv_bfloat16, 128>(cv, q, k, v, o, lse, fused, s);
}

}  // namespace rswa
