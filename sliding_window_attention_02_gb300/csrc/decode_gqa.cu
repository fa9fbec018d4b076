// R-SWA decode step for grouped heads (H query heads over H_kv KV heads) on
// the CUDA cores: split-K like decode_kernel, but one CTA serves G query
// heads of one KV head, so each K/V row of the cache is streamed once per G
// heads instead of once per head.  Grid (max_chunks, H / G, B).  Grouped
// caches of the tensor-core shape (bf16, d 128, <= 16 heads per KV head) use
// decode_gqa_tc.cu instead; this kernel serves the other element types and
// head sizes.
#include "attend.cuh"

#ifndef RSWA_GQA_UNROLL
#define RSWA_GQA_UNROLL 4
#endif
// Resident CTAs per SM the register budget of the register-loop kernel is
// cut for.
#ifndef RSWA_GQA_MINB
#define RSWA_GQA_MINB 4
#endif
// 1: the reduce-scatter loop (attend_range_grouped_rs) wherever its shape
// fits; 0: the plain grouped loop everywhere.
#ifndef RSWA_GQA_RS
#define RSWA_GQA_RS 1
#endif

namespace rswa {

// The key range of one split-K chunk of one head group.
struct GqaChunk {
  int64_t j0, j1;   // slab rows [j0, j1)
  int64_t sub;      // slab row read from (knew, vnew), or -1
  int64_t t_b;
  size_t bh0, bkv;  // first query head (b*H + h0) and KV head (b*Hkv + kv)
  int nch;          // chunks of this sequence
};

// Chunk c of head group hg of sequence b: a prefix chunk (c < ceil(m_b /
// chunk)) or a ring chunk.  The first head group of a KV head also stores
// the new k, v of a fused step in their ring slot.  False when c is past
// this sequence's chunks.
template <typename T, int D, bool FUSED, int G>
__device__ __forceinline__ bool gqa_chunk(const CacheView& cv, int c, int hg,
                                          int b, const T* knew, const T* vnew,
                                          GqaChunk& ck) {
  const int64_t m_b = cv.m_dev[b];
  const int chunk = cv.chunk;
  const int cp = (int)((m_b + chunk - 1) / chunk);
  const int cr = (int)((cv.n + chunk - 1) / chunk);
  ck.nch = cp + cr;
  if (c >= ck.nch) return false;
  const int h0 = hg * G;
  const int per_kv = cv.H / cv.Hkv;               // query heads per KV head
  ck.bh0 = (size_t)b * cv.H + h0;
  ck.bkv = (size_t)b * cv.Hkv + h0 / per_kv;
  ck.t_b = cv.t_dev[ck.bh0];                      // equal for the G heads
  ck.sub = -1;
  if (c < cp) {
    ck.j0 = (int64_t)c * chunk;
    ck.j1 = min(ck.j0 + chunk, m_b);
  } else {
    const int64_t s0 = (int64_t)(c - cp) * chunk;
    const int64_t filled = FUSED ? min(cv.n, ck.t_b + 1) : min(cv.n, ck.t_b);
    const int64_t s1 = max(s0, min(s0 + chunk, filled));
    ck.j0 = cv.m_cap + s0;
    ck.j1 = cv.m_cap + s1;
    if (FUSED) {
      const int64_t w = ck.t_b % cv.n;  // slot of the new output
      if (w >= s0 && w < s0 + chunk) ck.sub = cv.m_cap + w;
      if (ck.sub >= 0 && h0 % per_kv == 0) {
        // The first head group of the KV head stores the new k, v in slot
        // w; every CTA that reads slot w takes (knew, vnew) instead.
        T* Kw = static_cast<T*>(cv.K) + (ck.bkv * cv.slab_rows + ck.sub) * D;
        T* Vw = static_cast<T*>(cv.V) + (ck.bkv * cv.slab_rows + ck.sub) * D;
        const T* kn = knew + ck.bkv * D;
        const T* vn = vnew + ck.bkv * D;
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
  return true;
}

// Merge the warps' states of the G heads, publish this chunk's partial
// (m, l, acc[D]) per head, and let the last CTA of the head group (atomic
// counter, no waiting) combine all chunks into o, lse and t_b + 1.
template <typename T, int D, bool FUSED, int G, int EPL>
__device__ __forceinline__ void gqa_combine(const CacheView& cv,
                                            const GqaChunk& ck, int c,
                                            SoftmaxState<EPL>* st,
                                            T* __restrict__ o,
                                            float* __restrict__ lse) {
  constexpr int NW = kDecodeThreads / 32;
  constexpr int LPK = D / EPL;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int g = 0; g < G; ++g) merge_groups<T, D>(st[g]);
  __shared__ float s_m[NW][G], s_l[NW][G];
  __shared__ float s_acc[NW][G][D];
  if (lane < LPK) {
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
    float* P = cv.part + ((ck.bh0 + g) * cv.max_chunks + c) * (D + 2);
    if (tid < D) P[2 + tid] = A;
    if (tid == 0) {
      P[0] = M;
      P[1] = Ls;
    }
  }
  __syncthreads();
  __shared__ int s_last;
  if (tid == 0) s_last = arrive_acq_rel(&cv.cnt_bh[ck.bh0]) == ck.nch - 1;
  __syncthreads();
  if (!s_last) return;
  float M[G], L[G], A[G];
  merge_partials<G, 1>(
      cv.part + ck.bh0 * cv.max_chunks * (D + 2), (size_t)cv.max_chunks * (D + 2),
      ck.nch, D, tid, G, M, L, A);
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (tid < D) o[(ck.bh0 + g) * D + tid] = (T)(L[g] > 0.f ? A[g] / L[g] : 0.f);
    if (tid == 0) {
      if (lse) lse[ck.bh0 + g] = L[g] > 0.f ? (M[g] + log2f(L[g])) * kLn2 : -INFINITY;
      // Every CTA of this head group read t_b before its own arrival.
      if (FUSED) cv.t_dev[ck.bh0 + g] = ck.t_b + 1;
    }
  }
  if (tid == 0) cv.cnt_bh[ck.bh0] = 0;
}

template <typename T, int D, bool FUSED, int G>
__global__ void __launch_bounds__(kDecodeThreads, RSWA_GQA_MINB)
decode_gqa_kernel(CacheView cv, const T* __restrict__ q,
                  const T* __restrict__ knew, const T* __restrict__ vnew,
                  T* __restrict__ o, float* __restrict__ lse) {
  using C = AttendCfg<T, D, RSWA_GQA_UNROLL>;
  constexpr int NW = kDecodeThreads / 32;
  constexpr int EPL = C::EPL;
  const int c = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  griddep_wait();
  GqaChunk ck;
  if (!gqa_chunk<T, D, FUSED, G>(cv, c, blockIdx.y, blockIdx.z, knew, vnew, ck))
    return;
  const T* Kb = static_cast<const T*>(cv.K) + ck.bkv * cv.slab_rows * D;
  const T* Vb = static_cast<const T*>(cv.V) + ck.bkv * cv.slab_rows * D;
  const T* kn = FUSED ? knew + ck.bkv * D : nullptr;
  const T* vn = FUSED ? vnew + ck.bkv * D : nullptr;
  float qf[G * EPL];
#pragma unroll
  for (int g = 0; g < G; ++g) load_q_frag<T, D>(q + (ck.bh0 + g) * D, lane, qf + g * EPL);
  SoftmaxState<EPL> st[G];
#pragma unroll
  for (int g = 0; g < G; ++g) st[g].init();
  using RS = GroupedRsCfg<T, D, G>;
  if constexpr (RS::kUsable && RSWA_GQA_RS) {
    attend_range_grouped_rs<T, D, G>(
        qf, Kb, Vb, D, ck.j0, ck.j1, (int64_t)warp * RS::KEYS_WARP,
        (int64_t)NW * RS::KEYS_WARP, ck.sub, kn, vn, lane, st);
  } else {
    attend_range_grouped<T, D, RSWA_GQA_UNROLL, G>(
        qf, Kb, Vb, D, ck.j0, ck.j1, (int64_t)warp * C::KEYS_WARP,
        (int64_t)NW * C::KEYS_WARP, ck.sub, kn, vn, lane, st);
  }
  griddep_launch_dependents();
  gqa_combine<T, D, FUSED, G, EPL>(cv, ck, c, st, o, lse);
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
  const T* qq = (const T*)q;
  const T* kk = fused ? (const T*)k : nullptr;
  const T* vv = fused ? (const T*)v : nullptr;
  auto kern = fused ? decode_gqa_kernel<T, D, true, G>
                    : decode_gqa_kernel<T, D, false, G>;
  return cudaLaunchKernelEx(&cfg, kern, cv, qq, kk, vv, (T*)o, lse);
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
