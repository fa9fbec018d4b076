// R-SWA decode step for few heads with long caches: every CTA streams a
// contiguous share of one head's keys through shared memory.
//
// The keys of (b, h) are taken in the order [prefix rows 0..m_b-1 | ring
// slots 0..n-1] (the softmax does not depend on the order of its keys); ring
// slot s holds a key iff s < filled = min(n, t_b), or min(n, t_b + 1) in a
// fused step, whose new key sits in slot t_b mod n ("Unlimited-OCR deep
// dive": N(t) = P U D_n(t); the ring evicts the oldest output, GeekNews,
// model architecture).  The S CTAs of a head split this list evenly,
// share = ceil((m_b + n) / S) rows each, so the split depends on m_b only and
// a fused step may advance t_b while late CTAs of the launch still start.
//
// Roles (kWarps + 1 warps):
//   consumers  warps 0..kWarps-1: each stage's rows are split between them, a
//              row being LPK lanes wide (16-byte slices); every warp folds
//              its rows into per-lane online-softmax states
//   producer   warp kWarps: one thread copies the CTA's rows, stage by stage,
//              into a ring of NS shared-memory stages with bulk asynchronous
//              copies (one or two contiguous pieces per tensor and stage:
//              prefix rows and ring rows are contiguous in the slab)
// Prefix rows are read-only between prefills, so with PREFETCH the stages
// made only of prefix rows are requested before the dependency wait, while
// the previous kernel of the stream drains; ring rows, t_b and q are read
// after it.  Every CTA publishes (m, l, acc[d]); the last of the head's CTAs
// to arrive (atomic counter) merges the partials and writes o, lse and
// t_b + 1.  Every wait is bounded (wait_ns, phase_wait_limit_ns(), for the
// pipeline's phases; kWaitLimitNs for the drain); on a timeout the CTA
// drains its copies, publishes what it has, and sets the cache's device
// error flag.
#include <algorithm>

#include "attend.cuh"
#include "tc_ptx.cuh"

namespace rswa {
namespace {

// Consumer warps and stages: a stage holds kWarps * 4 KB of K and as much
// of V; 8 warps x 6 stages (192 KB, one CTA per SM) measured best on GB300
// for one sequence over a 16- or 40-page prefix.  Smaller CTAs that fit two
// per SM (so that the next layer's CTAs are resident and prefetch while this
// launch streams) were slower: 4 x 6 took 15.4-15.6 us per 40-page layer
// against 13.4-13.5, 4 x 3 16.0, 8 x 3 15.0; so was an L2 prefetch of each
// CTA's remaining prefix rows before the dependency wait (17.6 us), whose
// traffic delays the previous launch's combine.
#ifndef RSWA_STREAM_WARPS
#define RSWA_STREAM_WARPS 8
#endif
#ifndef RSWA_STREAM_STAGES
#define RSWA_STREAM_STAGES 6
#endif
constexpr int kWarps = RSWA_STREAM_WARPS;        // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kU = 4;                            // rows per lane group and stage
constexpr int NS = RSWA_STREAM_STAGES;           // stages
// Stages a CTA may request before its dependency wait: a third of its
// stages, at least RSWA_STREAM_EARLY_STAGES and at most 4.  Measured on
// GB300, one sequence through 12 layers (us per layer): 40 pages (11 stages
// per CTA) 12.66 with 2 early stages, 12.48 with 3, 12.42 with 4; 16 pages
// (5 stages) 8.13 with 1, 8.03 with 2, 8.25 with 3 — more early traffic
// slows the previous launch's combine unless the CTA has much left to read.
#ifndef RSWA_STREAM_EARLY_STAGES
#define RSWA_STREAM_EARLY_STAGES 2
#endif
constexpr int kEarlyStages = RSWA_STREAM_EARLY_STAGES;
constexpr int kEarlyStagesMax = 4;
constexpr uint32_t kTensorStage = kWarps * kU * 512;   // K (or V) bytes of a stage
constexpr uint32_t kStageBytes = 2 * kTensorStage;
constexpr uint32_t OFF_BAR = NS * kStageBytes;
constexpr uint32_t OFF_FLAG = OFF_BAR + 16 * NS;
constexpr uint32_t kSmemBytes = OFF_FLAG + 16;
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// cp.async.bulk of `bytes` contiguous bytes into this CTA's shared memory
// with the L2 eviction policy `pol`: the streamed rows are read once per
// launch, so they go with evict-first priority (stream_policy).
__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void* src, uint32_t bytes,
                                               uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// Brings the 128-byte line holding p into L2; no other effect.  L2 is the
// point of coherence for global memory, so a prefetch issued before the
// programmatic dependency wait is safe even for data the preceding kernel
// writes: the loads after the wait still see that kernel's stores.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint4 ld_shared16(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr));
  return r;
}

template <typename T, int D, bool FUSED, bool PREFETCH>
__global__ void __launch_bounds__(kThreads, (NS * kStageBytes <= 100 * 1024) ? 2 : 1)
decode_stream_kernel(CacheView cv, int S, const T* __restrict__ q,
                     const T* __restrict__ knew, const T* __restrict__ vnew,
                     T* __restrict__ o, float* __restrict__ lse, uint64_t wait_ns) {
  using C = AttendCfg<T, D, kU>;
  constexpr int EPL = C::EPL, LPK = C::LPK, KPW = C::KPW;
  constexpr uint32_t ROW_B = D * sizeof(T);            // bytes of a K or V row
  constexpr int SR = kWarps * kU * KPW;                 // rows per stage
  static_assert(SR * ROW_B == kTensorStage, "stage layout");
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sb = ptx::smem_u32(smem);
  auto full = [&](int s) { return sb + OFF_BAR + 8u * (uint32_t)s; };
  auto empty = [&](int s) { return sb + OFF_BAR + 8u * (uint32_t)(NS + s); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_FLAG);
  volatile int* never = reinterpret_cast<volatile int*>(smem + OFF_FLAG + 4);

  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const bool producer = warp == kWarps;
  const int grp = cv.H / cv.Hkv;                        // query heads per KV head
  const size_t bkv = (size_t)b * cv.Hkv + h / grp;
  const size_t bh = (size_t)b * cv.H + h;
  const T* Kb = static_cast<const T*>(cv.K) + bkv * cv.slab_rows * D;
  const T* Vb = static_cast<const T*>(cv.V) + bkv * cv.slab_rows * D;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(full(s), 1);
      ptx::mbar_init(empty(s), kWarps);
    }
    *abort_flag = 0;
    *never = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();

  // This CTA's logical rows [span0, span1) of the head's m_b + n.
  int64_t m_b = 0, share = 1, span0 = 0, span1 = 0;
  int nst = 0;                                          // stages
  auto plan = [&]() {
    const int64_t total = m_b + cv.n;
    share = (total + S - 1) / S;
    span0 = (int64_t)c * share;
    span1 = min(total, span0 + share);
    nst = span1 > span0 ? (int)((span1 - span0 + SR - 1) / SR) : 0;
  };
  // Copies stage k (ring slots from the first unfilled one on are not
  // copied); returns false once the bounded wait for a free slot gave up.
  // t_b is read after the dependency wait, and only stages that hold ring
  // slots use it, so the producer's first stages do not wait for the load.
  const uint64_t pol = stream_policy();               // rows read once per launch
  int64_t t_b = 0;
  auto ring_filled = [&]() { return FUSED ? min(cv.n, t_b + 1) : min(cv.n, t_b); };
  auto issue = [&](int k) {
    const int s = k % NS;
    if (k >= NS && !ptx::mbar_wait(empty(s), ((k / NS) - 1) & 1, abort_flag,
                                   wait_ns))
      return false;
    const int64_t l0 = span0 + (int64_t)k * SR, l1 = min(l0 + SR, span1);
    const int64_t p1 = min(l1, m_b);                    // prefix rows [l0, p1)
    const uint32_t np = p1 > l0 ? (uint32_t)(p1 - l0) : 0u;
    int64_t r0 = 0;                                     // ring slots [r0, r1)
    uint32_t nr = 0;
    if (l1 > m_b) {
      r0 = max(l0, m_b) - m_b;
      nr = (uint32_t)(max(r0, min(l1 - m_b, ring_filled())) - r0);
    }
    ptx::mbar_arrive_expect_tx(full(s), 2u * (np + nr) * ROW_B);
    const uint32_t kd = sb + (uint32_t)s * kStageBytes, vd = kd + kTensorStage;
    if (np) {
      bulk_load_hint(kd, Kb + l0 * D, np * ROW_B, full(s), pol);
      bulk_load_hint(vd, Vb + l0 * D, np * ROW_B, full(s), pol);
    }
    if (nr) {
      const uint32_t off = (uint32_t)(max(l0, m_b) - l0) * ROW_B;
      bulk_load_hint(kd + off, Kb + (cv.m_cap + r0) * D, nr * ROW_B, full(s), pol);
      bulk_load_hint(vd + off, Vb + (cv.m_cap + r0) * D, nr * ROW_B, full(s), pol);
    }
    return true;
  };

  // The first accesses after the wait read a few lines each (q, t_b, the
  // new key and value): have them in L2 by the time the wait returns.
  if (producer) {
    constexpr int QL = (D * (int)sizeof(T) + 127) / 128;  // lines per row
    const char* pf = nullptr;
    if (lane < QL) pf = reinterpret_cast<const char*>(q + bh * D) + lane * 128;
    else if (lane == QL) pf = reinterpret_cast<const char*>(cv.t_dev + bh);
    else if (FUSED && lane < 2 * QL + 1)
      pf = reinterpret_cast<const char*>(knew + bkv * D) + (lane - QL - 1) * 128;
    else if (FUSED && lane < 3 * QL + 1)
      pf = reinterpret_cast<const char*>(vnew + bkv * D) + (lane - 2 * QL - 1) * 128;
    if (pf) prefetch_l2(pf);
  }
  int issued = 0;                                       // stages issued
  if (PREFETCH) {
    m_b = cv.m_dev[b];
    plan();
    if (producer && lane == 0) {
      // Stages made only of prefix rows: their addresses and contents are
      // fixed until the next prefill.
      const int early = min(NS, max(kEarlyStages, min(kEarlyStagesMax, (nst + 1) / 3)));
      while (issued < min(nst, early) &&
             min(span0 + (int64_t)(issued + 1) * SR, span1) <= m_b) {
        issue(issued);
        ++issued;
      }
    }
  }
  griddep_wait();
  griddep_launch_dependents();
  float qf[EPL];
  if (!producer) load_q_frag<T, D>(q + bh * D, lane, qf);   // first request
  if (!PREFETCH) {
    m_b = cv.m_dev[b];
    plan();
  }
  if (nst == 0) return;                                 // no rows: nothing issued
  t_b = cv.t_dev[bh];
  const T* kn = FUSED ? knew + bkv * D : nullptr;
  const T* vn = FUSED ? vnew + bkv * D : nullptr;

  SoftmaxState<EPL> st;
  st.init();
  if (producer) {
    if (lane == 0) {
      while (issued < nst && issue(issued)) ++issued;
      // Drain: every copy issued has landed before the CTA may exit.
      for (int k = max(0, issued - NS); k < issued; ++k)
        ptx::mbar_wait(full(k % NS), (k / NS) & 1, never, kWaitLimitNs);
    }
  } else {
    const int64_t filled = ring_filled();
    const int64_t w = FUSED ? t_b % cv.n : -1;          // slot of the new key
    const bool has_w = FUSED && span0 <= m_b + w && m_b + w < span1;
    if (has_w && h % grp == 0 && warp == 0) {
      // This CTA holds slot w: store the new key and value there.  The
      // copies of this launch that may read the slot race with the store, so
      // the consumers take row w from (knew, vnew) instead.
      constexpr int NV = D * (int)sizeof(T) / 16;
      T* Kw = static_cast<T*>(cv.K) + (bkv * cv.slab_rows + (size_t)(cv.m_cap + w)) * D;
      T* Vw = static_cast<T*>(cv.V) + (bkv * cv.slab_rows + (size_t)(cv.m_cap + w)) * D;
      for (int i = lane; i < 2 * NV; i += 32) {
        if (i < NV)
          reinterpret_cast<uint4*>(Kw)[i] = reinterpret_cast<const uint4*>(kn)[i];
        else
          reinterpret_cast<uint4*>(Vw)[i - NV] = reinterpret_cast<const uint4*>(vn)[i - NV];
      }
    }
    const int gl = lane / LPK;
    const uint32_t col_b = (uint32_t)((lane % LPK) * EPL * sizeof(T));
    for (int k = 0; k < nst; ++k) {
      const int s = k % NS;
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(full(s), (k / NS) & 1, abort_flag,
                                                  wait_ns)))
        break;
      const int64_t l0 = span0 + (int64_t)k * SR, l1 = min(l0 + SR, span1);
      const uint32_t kd = sb + (uint32_t)s * kStageBytes, vd = kd + kTensorStage;
      AttendBatch<T, D, kU> bt;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int r = warp * (kU * KPW) + u * KPW + gl;  // row in the stage
        const int64_t l = l0 + r;
        const bool ring = l >= m_b;
        bt.ok[u] = l < l1 && (!ring || l - m_b < filled);
        if (FUSED && ring && l - m_b == w) {
          bt.k[u] = ld_stream16(reinterpret_cast<const uint8_t*>(kn) + col_b);
          bt.v[u] = ld_stream16(reinterpret_cast<const uint8_t*>(vn) + col_b);
        } else {
          bt.k[u] = ld_shared16(kd + (uint32_t)r * ROW_B + col_b);
          bt.v[u] = ld_shared16(vd + (uint32_t)r * ROW_B + col_b);
        }
        // A row that is not a key may hold any bits: value 0 (its score
        // is set to -inf by attend_consume).
        if (!bt.ok[u]) bt.v[u] = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(empty(s));
      attend_consume<T, D, kU>(qf, bt, st);
    }
    merge_groups<T, D>(st);
  }

  // Merge the consumer warps through shared memory, publish, and let the
  // last CTA of the head combine.
  __shared__ float s_m[kWarps], s_l[kWarps];
  __shared__ float s_acc[kWarps][D];
  __shared__ int s_last;
  if (!producer && lane < LPK) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) s_acc[warp][lane * EPL + e] = st.acc[e];
    if (lane == 0) {
      s_m[warp] = st.m;
      s_l[warp] = st.l;
    }
  }
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) M = fmaxf(M, s_m[i]);
  const float ref = (M == -INFINITY) ? 0.f : M;
  float Ls = 0.f, A = 0.f;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) {
    const float sc = fast_exp2(s_m[i] - ref);
    Ls += s_l[i] * sc;
    if (tid < D) A += s_acc[i][tid] * sc;
  }
  const int nch = (int)((m_b + cv.n + share - 1) / share);
  if (nch == 1) {
    if (tid < D) o[bh * D + tid] = (T)(Ls > 0.f ? A / Ls : 0.f);
    if (tid == 0) {
      if (lse) lse[bh] = Ls > 0.f ? (ref + log2f(Ls)) * kLn2 : -INFINITY;
      if (FUSED) cv.t_dev[bh] = t_b + 1;
      if (*abort_flag) flag_error(cv.err, kErrWaitTimeout);
    }
    return;
  }
  float* P = cv.part + bh * (size_t)S * (D + 2);
  if (tid < D) P[c * (D + 2) + 2 + tid] = A;
  if (tid == 0) {
    P[c * (D + 2)] = M;
    P[c * (D + 2) + 1] = Ls;
  }
  __syncthreads();
  if (tid == 0) s_last = arrive_acq_rel(&cv.cnt_bh[bh]) == nch - 1;
  __syncthreads();
  if (s_last) {
    float r2, Lt, At;
    merge_partials<1, 16>(P, 0, nch, D, tid, 1, &r2, &Lt, &At);
    if (tid < D) o[bh * D + tid] = (T)(Lt > 0.f ? At / Lt : 0.f);
    if (tid == 0) {
      if (lse) lse[bh] = Lt > 0.f ? (r2 + log2f(Lt)) * kLn2 : -INFINITY;
      cv.cnt_bh[bh] = 0;
      // Every CTA of (b, h) read t_b before its own arrival.
      if (FUSED) cv.t_dev[bh] = t_b + 1;
    }
  }
  if (tid == 0 && *abort_flag) flag_error(cv.err, kErrWaitTimeout);
}

template <typename T, int D, bool FUSED, bool PREFETCH>
cudaError_t launch_t(const CacheView& cv, int S, const void* q, const void* k,
                     const void* v, void* o, float* lse, cudaStream_t s) {
  auto kern = decode_stream_kernel<T, D, FUSED, PREFETCH>;
  // Per device (the attribute belongs to the current device's context).
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)S, (unsigned)cv.H, (unsigned)cv.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, cv, S, (const T*)q,
                            (const T*)(FUSED ? k : nullptr),
                            (const T*)(FUSED ? v : nullptr), (T*)o, lse,
                            phase_wait_limit_ns());
}

template <typename T, int D>
cudaError_t launch_td(const CacheView& cv, int S, const void* q, const void* k,
                      const void* v, void* o, float* lse, bool fused, bool pf,
                      cudaStream_t s) {
  if (fused)
    return pf ? launch_t<T, D, true, true>(cv, S, q, k, v, o, lse, s)
              : launch_t<T, D, true, false>(cv, S, q, k, v, o, lse, s);
  return pf ? launch_t<T, D, false, true>(cv, S, q, k, v, o, lse, s)
            : launch_t<T, D, false, false>(cv, S, q, k, v, o, lse, s);
}

// Rows of one stage for the cache's element type and head size.
int stage_rows(const CacheView& cv) {
  const int row_b = cv.d * (cv.dtype == RSWA_F32 ? 4 : 2);
  return (int)(kTensorStage / (uint32_t)row_b);
}

}  // namespace

// CTAs per head: one CTA per SM over all (b, h), at most one per stage of
// the head's m_cap + n rows, and no more than the partial slots the cache
// reserves per head.
#ifndef RSWA_STREAM_MAX_SPLITS
#define RSWA_STREAM_MAX_SPLITS 1024
#endif

int decode_stream_splits(const CacheView& cv) {
  const int64_t heads = (int64_t)cv.B * cv.H;
  int64_t S = std::min<int64_t>(cv.sms / heads, RSWA_STREAM_MAX_SPLITS);
  const int64_t sr = stage_rows(cv);
  S = std::min<int64_t>(S, (cv.m_cap + cv.n + sr - 1) / sr);
  S = std::min<int64_t>(S, cv.part_slots);
  return (int)std::max<int64_t>(S, 1);
}

// Few heads (at least two CTAs per head fit one wave), a ring no longer
// than the prefix capacity, and at least kMinBytesPerSm of keys and values
// per SM.  The split of [prefix | ring] may not depend on t_b, so a long
// ring that is still filling (the full-cache baseline, n >= T) would leave
// most CTAs idle; and a step of less than ~96 KB per SM is a latency chain
// that the split-K kernel's 8-warp CTAs run faster (one sequence over a
// 4-page prefix: 5.5 against 5.9 us per layer).  Those take the split-K
// kernel.
constexpr int64_t kMinBytesPerSm = 96 * 1024;

bool decode_use_stream(const CacheView& cv) {
  const int64_t row_b = (int64_t)cv.d * (cv.dtype == RSWA_F32 ? 4 : 2);
  const int64_t bytes = (int64_t)cv.B * cv.H * (cv.m_cap + cv.n) * 2 * row_b;
  return 2 * (int64_t)cv.B * cv.H <= cv.sms && cv.n <= cv.m_cap &&
         bytes >= kMinBytesPerSm * cv.sms && decode_stream_splits(cv) >= 2;
}

cudaError_t launch_decode_stream(const CacheView& cv, const void* q,
                                 const void* k, const void* v, void* o,
                                 float* lse, bool fused, bool prefetch_prefix,
                                 cudaStream_t s) {
  const int S = decode_stream_splits(cv);
  cudaError_t e;
  if (cv.dtype == RSWA_F32)
    e = cv.d == 64 ? launch_td<float, 64>(cv, S, q, k, v, o, lse, fused,
                                          prefetch_prefix, s)
                   : launch_td<float, 128>(cv, S, q, k, v, o, lse, fused,
                                           prefetch_prefix, s);
  else
    e = cv.d == 64 ? launch_td<__nv_bfloat16, 64>(cv, S, q, k, v, o, lse, fused,
                                                  prefetch_prefix, s)
                   : launch_td<__nv_bfloat16, 128>(cv, S, q, k, v, o, lse, fused,
                                                   prefetch_prefix, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace rswa
