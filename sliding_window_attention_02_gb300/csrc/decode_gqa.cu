// R-SWA decode step for grouped heads (H query heads over H_kv KV heads):
// split-K like decode_kernel, but one CTA serves G query heads of one KV
// head, so each K/V row of the cache is streamed once per G heads instead of
// once per head.  Grid (max_chunks, H / G, B).
#include "attend.cuh"

#ifndef RSWA_GQA_UNROLL
#define RSWA_GQA_UNROLL 4
#endif

namespace rswa {

template <typename T, int D, bool FUSED, int G>
__global__ void __launch_bounds__(kDecodeThreads, 4)
decode_gqa_kernel(CacheView cv, const T* __restrict__ q,
                  const T* __restrict__ knew, const T* __restrict__ vnew,
                  T* __restrict__ o, float* __restrict__ lse) {
  using C = AttendCfg<T, D, RSWA_GQA_UNROLL>;
  constexpr int NW = kDecodeThreads / 32;
  constexpr int EPL = C::EPL;
  const int c = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  griddep_wait();

  const int64_t m_b = cv.m_dev[b];
  const int chunk = cv.chunk;
  const int cp = (int)((m_b + chunk - 1) / chunk);
  const int cr = (int)((cv.n + chunk - 1) / chunk);
  const int nch = cp + cr;
  if (c >= nch) return;
  const int h0 = hg * G;                          // first query head served
  const int per_kv = cv.H / cv.Hkv;               // query heads per KV head
  const size_t bh0 = (size_t)b * cv.H + h0;
  const size_t bkv = (size_t)b * cv.Hkv + h0 / per_kv;
  const int64_t t_b = cv.t_dev[bh0];              // equal for the G heads

  const T* Kb = static_cast<const T*>(cv.K) + bkv * cv.slab_rows * D;
  const T* Vb = static_cast<const T*>(cv.V) + bkv * cv.slab_rows * D;
  const T* kn = FUSED ? knew + bkv * D : nullptr;
  const T* vn = FUSED ? vnew + bkv * D : nullptr;

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
      if (w >= s0 && w < s0 + chunk) sub = cv.m_cap + w;
      if (sub >= 0 && h0 % per_kv == 0) {
        // The first head group of the KV head stores the new k, v in slot w;
        // no CTA of this launch reads slot w from the slab.
        T* Kw = static_cast<T*>(cv.K) + (bkv * cv.slab_rows + sub) * D;
        T* Vw = static_cast<T*>(cv.V) + (bkv * cv.slab_rows + sub) * D;
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

  float qf[G * EPL];
#pragma unroll
  for (int g = 0; g < G; ++g) load_q_frag<T, D>(q + (bh0 + g) * D, lane, qf + g * EPL);
  SoftmaxState<EPL> st[G];
#pragma unroll
  for (int g = 0; g < G; ++g) st[g].init();
  attend_range_grouped<T, D, RSWA_GQA_UNROLL, G>(
      qf, Kb, Vb, D, j0, j1, (int64_t)warp * C::KEYS_WARP,
      (int64_t)NW * C::KEYS_WARP, sub, kn, vn, lane, st);
  griddep_launch_dependents();
#pragma unroll
  for (int g = 0; g < G; ++g) merge_groups<T, D>(st[g]);

  __shared__ float s_m[NW][G], s_l[NW][G];
  __shared__ float s_acc[NW][G][D];
  if (lane < C::LPK) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) s_acc[warp][g][lane * EPL + e] = st[g].acc[e];
      if (lane == 0) {
        s_m[warp][g] = st[g].m;
        s_l[warp][g] = st[g].l;
      }
    }
  }
  __syncthreads();
  const int tid = threadIdx.x;
  // Publish this chunk's partial (m, l, acc[D]) of each of the G heads.
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, s_m[w][g]);
    const float ref = (M == -INFINITY) ? 0.f : M;
    float Ls = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float sc = fast_exp2(s_m[w][g] - ref);
      Ls += s_l[w][g] * sc;
      if (tid < D) A += s_acc[w][g][tid] * sc;
    }
    float* P = cv.part + ((bh0 + g) * cv.max_chunks + c) * (D + 2);
    if (tid < D) P[2 + tid] = A;
    if (tid == 0) {
      P[0] = M;
      P[1] = Ls;
    }
  }
  __threadfence();
  __syncthreads();
  __shared__ int s_last;
  if (tid == 0) s_last = (atomicAdd(&cv.cnt_bh[bh0], 1) == nch - 1);
  __syncthreads();
  if (s_last) {
    __threadfence();
    for (int g = 0; g < G; ++g) {
      const float* P = cv.part + (bh0 + g) * cv.max_chunks * (D + 2);
      float Mx = -INFINITY;
      for (int k = 0; k < nch; ++k) Mx = fmaxf(Mx, __ldcg(P + k * (D + 2)));
      const float r2 = (Mx == -INFINITY) ? 0.f : Mx;
      float Lt = 0.f, At = 0.f;
      for (int k = 0; k < nch; ++k) {
        const float sc = fast_exp2(__ldcg(P + k * (D + 2)) - r2);
        Lt += __ldcg(P + k * (D + 2) + 1) * sc;
        if (tid < D) At += __ldcg(P + k * (D + 2) + 2 + tid) * sc;
      }
      if (tid < D) o[(bh0 + g) * D + tid] = (T)(Lt > 0.f ? At / Lt : 0.f);
      if (tid == 0) {
        if (lse) lse[bh0 + g] = Lt > 0.f ? (r2 + log2f(Lt)) * kLn2 : -INFINITY;
        // Every CTA of this head group read t_b before its own arrival.
        if (FUSED) cv.t_dev[bh0 + g] = t_b + 1;
      }
    }
    if (tid == 0) cv.cnt_bh[bh0] = 0;
  }
}

int decode_gqa_heads_per_cta(const CacheView& cv) {
  return gqa_heads_per_cta(cv.H, cv.Hkv);
}

template <typename T, int D, int G>
static cudaError_t launch_g(const CacheView& cv, const void* q, const void* k,
                            const void* v, void* o, float* lse, bool fused,
                            cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cv.max_chunks, cv.H / G, cv.B);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (fused)
    return cudaLaunchKernelEx(&cfg, decode_gqa_kernel<T, D, true, G>, cv,
                              (const T*)q, (const T*)k, (const T*)v, (T*)o, lse);
  return cudaLaunchKernelEx(&cfg, decode_gqa_kernel<T, D, false, G>, cv,
                            (const T*)q, (const T*)nullptr, (const T*)nullptr,
                            (T*)o, lse);
}

template <typename T, int D>
static cudaError_t launch_gt(const CacheView& cv, const void* q, const void* k,
                             const void* v, void* o, float* lse, bool fused,
                             cudaStream_t s) {
  if (decode_gqa_heads_per_cta(cv) == 4)
    return launch_g<T, D, 4>(cv, q, k, v, o, lse, fused, s);
  return launch_g<T, D, 2>(cv, q, k, v, o, lse, fused, s);
}

cudaError_t launch_decode_gqa(const CacheView& cv, const void* q, const void* k,
                              const void* v, void* o, float* lse, bool fused,
                              cudaStream_t s) {
  cudaError_t e;
  if (cv.dtype == RSWA_F32)
    e = cv.d == 64 ? launch_gt<float, 64>(cv, q, k, v, o, lse, fused, s)
                   : launch_gt<float, 128>(cv, q, k, v, o, lse, fused, s);
  else
    e = cv.d == 64 ? launch_gt<__nv_bfloat16, 64>(cv, q, k, v, o, lse, fused, s)
                   : launch_gt<__nv_bfloat16, 128>(cv, q, k, v, o, lse, fused, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace rswa
