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
#include <algorithm>

#include "attend.cuh"
#include "tc_ptx.cuh"

namespace rswa {

// Stores v at a with the L2 eviction priority of `pol` (a createpolicy
// descriptor).
__device__ __forceinline__ void st_hint(float* a, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(a), "f"(v), "l"(pol)
               : "memory");
}
// Evict-last priority for a split-K partial: kept in L2 while the streamed
// keys pass through, until the merge reads and discards it.
__device__ __forceinline__ uint64_t partial_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Drops, without write-back, the L2 lines that lie wholly inside [lo, hi):
// merged split-K partials, which nothing reads again before a later launch
// rewrites them, would otherwise go back to DRAM when the streamed keys
// evict them.  The lines at the two ends may hold another head's partials
// and are kept.  Thread t of nt takes lines t, t + nt, ...; the caller has
// made every read of the range complete (a barrier after the merge).
__device__ __forceinline__ void discard_l2_inside(const void* lo, const void* hi, int t,
                                                  int nt) {
  const uintptr_t a = (reinterpret_cast<uintptr_t>(lo) + 127) & ~uintptr_t(127);
  const uintptr_t e = reinterpret_cast<uintptr_t>(hi) & ~uintptr_t(127);
  for (uintptr_t p = a + (uintptr_t)t * 128; p < e; p += (uintptr_t)nt * 128)
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// At least 5 resident CTAs per SM: measured best on GB300 for the batched
// and long-output workloads (it also steers the compiler to issue a warp's
// loads ahead of their use).
// PREFETCH: the preceding kernel of the stream writes no prefix row and no
// m_b of this cache (the host's per-handle flag), so a prefix-chunk CTA
// reads m_b and loads its warps' first row batch before the dependency
// wait, while the previous kernel drains.
// NW warps per CTA: 4 (five CTAs per SM) in general; 8 when the grid is
// small enough to stay in one wave, so that each CTA takes half as many
// dependent row batches.
template <typename T, int D, bool FUSED, bool PREFETCH, int NW>
__global__ void __launch_bounds__(NW * 32, NW == 4 ? 5 : 2)
decode_kernel(CacheView cv, const T* __restrict__ q, const T* __restrict__ knew,
              const T* __restrict__ vnew, T* __restrict__ o,
              float* __restrict__ lse) {
  using C = AttendCfg<T, D>;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = cv.H / cv.Hkv;                  // query heads per KV head
  const size_t bkv = (size_t)b * cv.Hkv + h / grp;
  const T* Kb = static_cast<const T*>(cv.K) + bkv * cv.slab_rows * D;
  const T* Vb = static_cast<const T*>(cv.V) + bkv * cv.slab_rows * D;
  // Each key and value row is read once per launch.
  const uint64_t pol = stream_policy();
  AttendBatch<T, D> pre;
  bool have_pre = false;
  int64_t m_b = 0;
  if (PREFETCH) {
    m_b = cv.m_dev[b];
    const int64_t j0 = (int64_t)c * cv.chunk;
    const int64_t j1 = min(j0 + cv.chunk, m_b);
    const int64_t base = j0 + (int64_t)warp * C::KEYS_WARP;
    if (j0 < m_b && base < j1) {                  // a prefix chunk with rows here
      attend_load<T, D, RSWA_DECODE_UNROLL, true>(Kb, Vb, D, base, j0, j1, -1, nullptr,
                                                  nullptr, lane, INT64_MAX, 0, pre, pol);
      have_pre = true;
    }
  }
  // Launched as a programmatic dependent: wait until the previous kernel in
  // the stream has completed and its writes are visible.  The next step's
  // CTAs may then take SM slots as this grid's CTAs finish; they wait for
  // this grid.
  griddep_wait();
  griddep_launch_dependents();

  if (!PREFETCH) m_b = cv.m_dev[b];
  const int chunk = cv.chunk;
  const int cp = (int)((m_b + chunk - 1) / chunk);
  const int cr = (int)((cv.n + chunk - 1) / chunk);
  const int nch = cp + cr;
  if (c >= nch) return;
  const size_t bh = (size_t)b * cv.H + h;
  const int64_t t_b = cv.t_dev[bh];
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
      if (sub >= 0 && h % grp == 0) {
        // This CTA owns slot w for its KV head: store the new k, v there.
        // No CTA of this launch reads slot w from the slab (it reads
        // (knew, vnew) instead).
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

  float qf[C::EPL];
  load_q_frag<T, D>(q + bh * D, lane, qf);
  SoftmaxState<C::EPL> st;
  st.init();
  int64_t first = (int64_t)warp * C::KEYS_WARP;
  if (have_pre) {
    attend_consume<T, D>(qf, pre, st);
    first += (int64_t)NW * C::KEYS_WARP;
  }
  attend_range<T, D, RSWA_DECODE_UNROLL, true>(qf, Kb, Vb, D, j0, j1, first,
                                               (int64_t)NW * C::KEYS_WARP, sub, kn, vn, lane,
                                               st, INT64_MAX, 0, pol);
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
  if (nch == 1) {
    // The only chunk of (b, h) (a short cache, e.g. m_b = 0): no partials.
    if (tid < D) o[bh * D + tid] = (T)(Ls > 0.f ? A / Ls : 0.f);
    if (tid == 0) {
      if (lse) lse[bh] = Ls > 0.f ? (ref + log2f(Ls)) * kLn2 : -INFINITY;
      if (FUSED) cv.t_dev[bh] = t_b + 1;
    }
    return;
  }

  // Publish this chunk's partial (m, l, acc[D]).
  float* P = cv.part + (bh * cv.max_chunks) * (D + 2);
  const uint64_t ppol = partial_policy();
  if (tid < D) st_hint(P + c * (D + 2) + 2 + tid, A, ppol);
  if (tid == 0) {
    st_hint(P + c * (D + 2), M, ppol);
    st_hint(P + c * (D + 2) + 1, Ls, ppol);
  }
  __syncthreads();
  __shared__ int s_last;
  if (tid == 0) s_last = arrive_acq_rel(&cv.cnt_bh[bh]) == nch - 1;
  __syncthreads();
  if (s_last) {
    float r2, Lt, At;
    // Up to 16 chunks per round trip: a batch-1 head with a 40-page prefix
    // has 42 chunks, and this merge is the last step of the decode.
    merge_partials<1, 16>(P, 0, nch, D, tid, 1, &r2, &Lt, &At);
    if (tid < D) o[bh * D + tid] = (T)(Lt > 0.f ? At / Lt : 0.f);
    if (tid == 0) {
      if (lse) lse[bh] = Lt > 0.f ? (r2 + log2f(Lt)) * kLn2 : -INFINITY;
      cv.cnt_bh[bh] = 0;
      // The last CTA of (b, h) advances this head's t_b; every other CTA of
      // (b, h) read it before its own arrival.
      if (FUSED) cv.t_dev[bh] = t_b + 1;
    }
    __syncthreads();
    discard_l2_inside(P, P + (size_t)nch * (D + 2), tid, blockDim.x);
  }
}

// 1: few heads with long caches stream through shared memory
// (decode_stream.cu); 0: they take the split-K kernel.
#ifndef RSWA_STREAM_DECODE
#define RSWA_STREAM_DECODE 1
#endif

constexpr uint32_t kMaxClusterSize = 8;
// Loads in flight per lane in the cluster path: 4 measured best on GB300 for
// the latency-bound single-page step (the split-K path keeps 8).
#ifndef RSWA_CLUSTER_UNROLL
#define RSWA_CLUSTER_UNROLL 4
#endif
constexpr int kClusterUnroll = RSWA_CLUSTER_UNROLL;

// Bound on the cluster path's wait for the partials of its cluster.
constexpr uint64_t kClusterWaitNs = 1000000000ull;

// Small-batch decode: a thread-block cluster of CL CTAs (NW warps each) per
// (b, h).  Each CTA takes an even share of the slab's prefix rows
// 0 .. m_cap-1 and of its ring rows m_cap .. m_cap+n-1, one load per lane
// and row: these addresses depend on neither m_b nor t_b, so all loads are
// issued at once.  With PREFETCH (the preceding kernel of the stream writes
// no prefix row and no m_b of this cache) the prefix rows and m_b are even
// loaded before the dependency wait, while the previous step drains; q, t_b,
// the new k/v and the ring rows follow the wait.  Prefix rows at or past m_b
// and ring slots not yet filled are masked (score -inf, value 0: such a row
// may hold any bits), and the ring slot this step appends to is read from
// (knew, vnew).  Each CTA merges its warps in shared memory and sends its
// partial to CTA rank 0 with asynchronous remote stores that complete an
// mbarrier there; rank 0 waits on that barrier alone (bounded) and combines
// the CL partials from its own shared memory while the other CTAs have
// already exited - no global partials, no atomics, no remote loads and no
// cluster barrier on the critical path.  Used when few heads are in flight
// and every head's cache fits one row batch per CTA.
template <typename T, int D, bool FUSED, int NW, bool PREFETCH>
__global__ void __launch_bounds__(NW * 32)
decode_cluster_kernel(CacheView cv, const T* __restrict__ q,
                      const T* __restrict__ knew, const T* __restrict__ vnew,
                      T* __restrict__ o, float* __restrict__ lse) {
  using C = AttendCfg<T, D, kClusterUnroll>;
  constexpr int EPL = C::EPL, LPK = C::LPK, KPW = C::KPW, U = C::U;
  const uint32_t rank = cluster_rank(), CL = cluster_size();
  const int h = blockIdx.x / CL, b = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp_lane = lane / LPK;
  const int col = (lane % LPK) * EPL;
  const size_t bh = (size_t)b * cv.H + h;
  const int grp = cv.H / cv.Hkv;                  // query heads per KV head
  const size_t bkv = (size_t)b * cv.Hkv + h / grp;
  __shared__ float s_m[NW], s_l[NW];
  __shared__ float s_acc[NW][D];
  __shared__ float c_ml[kMaxClusterSize][2];   // rank 0's copy is the one used
  __shared__ float c_acc[kMaxClusterSize][D];
  __shared__ uint64_t c_bar;                   // rank 0: all partials landed
  // This CTA's prefix rows [a0, a1) and ring slots [r0, r1): local row
  // i < np is prefix row a0 + i, then ring row m_cap + r0 + (i - np).
  const int64_t pp = (cv.m_cap + CL - 1) / CL, pr = (cv.n + CL - 1) / CL;
  // One row batch of NW warps must hold both shares (the host sizes the
  // cluster so); the test is uniform over the cluster.
  if (pp + pr > (int64_t)NW * C::KEYS_WARP) {
    if (threadIdx.x == 0) flag_error(cv.err, kErrLaunchShape);
    return;
  }
  const int64_t a0 = min(cv.m_cap, (int64_t)rank * pp);
  const int64_t a1 = min(cv.m_cap, a0 + pp);
  const int64_t r0 = min(cv.n, (int64_t)rank * pr);
  const int64_t r1 = min(cv.n, r0 + pr);
  const int np = (int)(a1 - a0), nr = (int)(r1 - r0);
  int64_t row[U];
  int kind[U];                                  // 0 none, 1 prefix, 2 ring
  uint4 kr[U], vr[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int i = warp * C::KEYS_WARP + u * KPW + grp_lane;
    kind[u] = i < np ? 1 : (i < np + nr ? 2 : 0);
    row[u] = kind[u] == 1 ? a0 + i : cv.m_cap + r0 + (i - np);
    kr[u] = vr[u] = make_uint4(0, 0, 0, 0);
  }
  const T* Kb = static_cast<const T*>(cv.K) + bkv * cv.slab_rows * D;
  const T* Vb = static_cast<const T*>(cv.V) + bkv * cv.slab_rows * D;
  if (rank == 0 && threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&c_bar), 1);
    ptx::fence_mbar_init();
    ptx::mbar_arrive_expect_tx(ptx::smem_u32(&c_bar), CL * (D + 2) * 4);
  }
  // Publishes rank 0's barrier and marks this CTA as started; the matching
  // wait precedes the first store into rank 0's shared memory.
  cluster_arrive_release();
  int64_t m_b = 0;
  if (PREFETCH) {
    m_b = cv.m_dev[b];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (kind[u] == 1) {
        kr[u] = ld_stream16(Kb + row[u] * D + col);
        vr[u] = ld_stream16(Vb + row[u] * D + col);
      }
  }
  griddep_wait();
  griddep_launch_dependents();
  if (!PREFETCH) {
    m_b = cv.m_dev[b];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (kind[u] == 1) {
        kr[u] = ld_stream16(Kb + row[u] * D + col);
        vr[u] = ld_stream16(Vb + row[u] * D + col);
      }
  }
  const int64_t t_b = cv.t_dev[bh];
  float qf[EPL];
  load_q_frag<T, D>(q + bh * D, lane, qf);
  uint4 kn = make_uint4(0, 0, 0, 0), vn = kn;
  if (FUSED) {
    kn = ld_stream16(knew + bkv * D + col);
    vn = ld_stream16(vnew + bkv * D + col);
  }
#pragma unroll
  for (int u = 0; u < U; ++u)
    if (kind[u] == 2) {
      kr[u] = ld_stream16(Kb + row[u] * D + col);
      vr[u] = ld_stream16(Vb + row[u] * D + col);
    }
  const int64_t filled = FUSED ? min(cv.n, t_b + 1) : min(cv.n, t_b);
  const int64_t sub = FUSED ? cv.m_cap + t_b % cv.n : -1;
  if constexpr (FUSED) {
    if (rank == 0 && h % grp == 0) {
      // Lanes that hold slot sub replace what they loaded with (knew,
      // vnew), so the value this write races with is never used.
      T* Kw = static_cast<T*>(cv.K) + (bkv * cv.slab_rows + (size_t)sub) * D;
      T* Vw = static_cast<T*>(cv.V) + (bkv * cv.slab_rows + (size_t)sub) * D;
      constexpr int NV = D * sizeof(T) / 16;
      for (int i = threadIdx.x; i < 2 * NV; i += blockDim.x) {
        if (i < NV)
          reinterpret_cast<uint4*>(Kw)[i] = reinterpret_cast<const uint4*>(knew + bkv * D)[i];
        else
          reinterpret_cast<uint4*>(Vw)[i - NV] =
              reinterpret_cast<const uint4*>(vnew + bkv * D)[i - NV];
      }
    }
  }
  bool ok[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    ok[u] = kind[u] == 1 ? row[u] < m_b
                         : (kind[u] == 2 && row[u] - cv.m_cap < filled);
    if (kind[u] == 2 && row[u] == sub) {
      kr[u] = kn;
      vr[u] = vn;
    }
    if (!ok[u]) vr[u] = make_uint4(0, 0, 0, 0);
  }
  float s[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    float kf[EPL];
    Elt<T>::widen(kr[u], kf);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc = fmaf(qf[e], kf[e], acc);
    s[u] = acc;
  }
#pragma unroll
  for (int off = LPK / 2; off > 0; off >>= 1) {
#pragma unroll
    for (int u = 0; u < U; ++u) s[u] += __shfl_xor_sync(0xffffffffu, s[u], off);
  }
  SoftmaxState<EPL> st;
  float mx = -INFINITY;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (!ok[u]) s[u] = -INFINITY;
    mx = fmaxf(mx, s[u]);
  }
  const float ref = (mx == -INFINITY) ? 0.f : mx;
  st.m = mx;
  st.l = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) st.acc[e] = 0.f;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const float p = fast_exp2(s[u] - ref);
    st.l += p;
    float vf[EPL];
    Elt<T>::widen(vr[u], vf);
#pragma unroll
    for (int e = 0; e < EPL; ++e) st.acc[e] = fmaf(p, vf[e], st.acc[e]);
  }
  merge_groups<T, D>(st);
  if (lane < LPK) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) s_acc[warp][lane * EPL + e] = st.acc[e];
    if (lane == 0) {
      s_m[warp] = st.m;
      s_l[warp] = st.l;
    }
  }
  __syncthreads();
  const int tid = threadIdx.x;
  float A = 0.f, M = -INFINITY, Ls = 0.f;
  if (tid < D) {
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, s_m[w]);
    const float r0f = (M == -INFINITY) ? 0.f : M;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float sc = fast_exp2(s_m[w] - r0f);
      Ls += s_l[w] * sc;
      A += s_acc[w][tid] * sc;
    }
  }
  cluster_wait();                    // rank 0's barrier is initialised
  if (tid < D) {
    const uint32_t bar = map_dsmem(&c_bar, 0);
    st_async_f32(map_dsmem(&c_acc[rank][tid], 0), bar, A);
    if (tid == 0) {
      st_async_f32(map_dsmem(&c_ml[rank][0], 0), bar, M);
      st_async_f32(map_dsmem(&c_ml[rank][1], 0), bar, Ls);
    }
  }
  // Second phase of the cluster barrier: every thread arrives once it has
  // issued its stores into rank 0.  Only rank 0's give-up path below waits
  // on this phase; the partials themselves land on c_bar.
  __syncwarp();
  cluster_arrive_relaxed();
  if (rank != 0 || tid >= D) return;
  // Bounded wait for the CL partials; gives up at once when an earlier
  // launch on this cache already flagged an error.
  const uint32_t bar = ptx::smem_u32(&c_bar);
  if (!ptx::mbar_try_wait(bar, 0)) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 1; !ptx::mbar_try_wait(bar, 0); ++it) {
      if ((it & 63u) == 0 &&
          (*(volatile int32_t*)cv.err != 0 ||
           ptx::globaltimer_ns() - t0 > kClusterWaitNs)) {
        flag_error(cv.err, kErrWaitTimeout);
        // Giving up: this CTA must not exit while a peer may still store
        // into its shared memory.  Wait until every thread of the cluster
        // has issued its stores (arrived at the second phase) or exited -
        // peers run straight-line code, so they all get there - then give
        // the stores already issued a bounded time to land.
        cluster_wait_divergent();
        const uint64_t t1 = ptx::globaltimer_ns();
        for (uint32_t it2 = 1; !ptx::mbar_try_wait(bar, 0); ++it2)
          if ((it2 & 63u) == 0 && ptx::globaltimer_ns() - t1 > kClusterWaitNs) break;
        return;
      }
    }
  }
  float Mr[kMaxClusterSize], Lr[kMaxClusterSize], Ar[kMaxClusterSize];
  float Mt = -INFINITY;
#pragma unroll
  for (uint32_t r = 0; r < kMaxClusterSize; ++r) {
    const bool in = r < CL;
    Mr[r] = in ? c_ml[r][0] : -INFINITY;
    Lr[r] = in ? c_ml[r][1] : 0.f;
    Ar[r] = in ? c_acc[r][tid] : 0.f;
    Mt = fmaxf(Mt, Mr[r]);
  }
  const float rt = (Mt == -INFINITY) ? 0.f : Mt;
  float Lt = 0.f, At = 0.f;
#pragma unroll
  for (uint32_t r = 0; r < kMaxClusterSize; ++r) {
    const float sc = fast_exp2(Mr[r] - rt);
    Lt += Lr[r] * sc;
    At += Ar[r] * sc;
  }
  o[bh * D + tid] = (T)(Lt > 0.f ? At / Lt : 0.f);
  if (tid == 0) {
    if (lse) lse[bh] = Lt > 0.f ? (rt + log2f(Lt)) * kLn2 : -INFINITY;
    // Every CTA of the cluster read t_b before sending its partial.
    if (FUSED) cv.t_dev[bh] = t_b + 1;
  }
}

#ifndef RSWA_CLUSTER_WARPS
#define RSWA_CLUSTER_WARPS 8
#endif
constexpr int kClusterWarps = RSWA_CLUSTER_WARPS;
constexpr int kMaxCluster = (int)kMaxClusterSize;

// Launch with programmatic stream serialization so that a decode kernel may
// begin launching while the previous kernel of the stream drains; with a
// cluster dimension when cluster > 0.
template <typename K, typename... Args>
static cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, int cluster,
                              cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cluster > 0) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Keys one CTA of the cluster path covers per iteration of its warps.
static int64_t cluster_keys_per_iter(const CacheView& cv) {
  const int epl = cv.dtype == RSWA_F32 ? 4 : 8;
  const int kpw = 32 / (cv.d / epl);
  return (int64_t)kClusterWarps * kpw * kClusterUnroll;
}

// Cluster size: the fewest CTAs (at most 8) whose share of the prefix rows
// plus share of the ring rows fits one row batch of a CTA; kMaxCluster + 1
// when none does.
static int cluster_size_for(const CacheView& cv) {
#ifdef RSWA_CLUSTER_SIZE
  return RSWA_CLUSTER_SIZE;
#endif
  const int64_t per = cluster_keys_per_iter(cv);
  for (int c = 1; c <= kMaxCluster; ++c)
    if ((cv.m_cap + c - 1) / c + (cv.n + c - 1) / c <= per) return c;
  return kMaxCluster + 1;
}

template <typename T, int D, bool FUSED>
static cudaError_t launch_cluster(const CacheView& cv, const T* q, const T* k,
                                  const T* v, T* o, float* lse, bool prefetch,
                                  cudaStream_t s) {
  const int cl = cluster_size_for(cv);
  const dim3 grid(cv.H * cl, cv.B), block(kClusterWarps * 32);
  if (prefetch)
    return launch_pdl(decode_cluster_kernel<T, D, FUSED, kClusterWarps, true>,
                      grid, block, cl, s, cv, q, k, v, o, lse);
  return launch_pdl(decode_cluster_kernel<T, D, FUSED, kClusterWarps, false>,
                    grid, block, cl, s, cv, q, k, v, o, lse);
}

// bf16 split-K CTAs get 8 warps (two resident per SM) when the whole grid
// fits one wave of them (2 x the SM count); otherwise 4 warps (five per SM).
// Measured on the one-sequence, 12-layer workload on GB300 (152 SMs): a
// 4-page prefix (100 CTAs) 6.18 -> 5.5 us per layer with 8 warps; 16 and 40
// pages (340 and 420 CTAs) lose a wave and slow down with them.
constexpr int64_t kWideCtasPerSm = 2;

template <typename T, int D, int NW>
static cudaError_t launch_split(const CacheView& cv, const T* qq, const T* kk,
                                const T* vv, T* oo, float* lse, bool fused,
                                bool prefetch, cudaStream_t s) {
  const dim3 grid(cv.max_chunks, cv.H, cv.B), block(NW * 32);
  const T* nk = nullptr;
  // The preloaded batch costs registers: bf16 caches only (float32 ones
  // would spill).
  if constexpr (sizeof(T) == 2) {
    if (fused && prefetch)
      return launch_pdl(decode_kernel<T, D, true, true, NW>, grid, block, 0, s, cv,
                        qq, kk, vv, oo, lse);
    if (prefetch)
      return launch_pdl(decode_kernel<T, D, false, true, NW>, grid, block, 0, s, cv,
                        qq, nk, nk, oo, lse);
  }
  if (fused)
    return launch_pdl(decode_kernel<T, D, true, false, NW>, grid, block, 0, s, cv, qq,
                      kk, vv, oo, lse);
  return launch_pdl(decode_kernel<T, D, false, false, NW>, grid, block, 0, s, cv, qq,
                    nk, nk, oo, lse);
}

template <typename T, int D>
static cudaError_t launch_decode_t(const CacheView& cv, const void* q,
                                   const void* k, const void* v, void* o,
                                   float* lse, bool fused, bool prefetch,
                                   cudaStream_t s) {
  const T* qq = (const T*)q;
  const T* kk = (const T*)k;
  const T* vv = (const T*)v;
  T* oo = (T*)o;
  cudaError_t e;
  if (decode_use_small(cv)) {
    if (fused)
      e = launch_cluster<T, D, true>(cv, qq, kk, vv, oo, lse, prefetch, s);
    else
      e = launch_cluster<T, D, false>(cv, qq, nullptr, nullptr, oo, lse,
                                      prefetch, s);
  } else if (RSWA_STREAM_DECODE && decode_use_stream(cv)) {
    return launch_decode_stream(cv, q, k, v, o, lse, fused, prefetch, s);
  } else if constexpr (sizeof(T) == 2) {
    if ((int64_t)cv.B * cv.H * cv.max_chunks <= kWideCtasPerSm * cv.sms)
      e = launch_split<T, D, 8>(cv, qq, kk, vv, oo, lse, fused, prefetch, s);
    else
      e = launch_split<T, D, 4>(cv, qq, kk, vv, oo, lse, fused, prefetch, s);
  } else {
    e = launch_split<T, D, 4>(cv, qq, kk, vv, oo, lse, fused, prefetch, s);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// 1: grouped caches of the tensor-core shape decode on the tensor cores;
// 0: on the CUDA cores (decode_gqa.cu).
#ifndef RSWA_GQA_TC
#define RSWA_GQA_TC 1
#endif
// 1: the stream-K form of the tensor-core grouped decode where it applies;
// 0: one CTA per chunk of a KV head (decode_gqa_tc.cu).
#ifndef RSWA_GQA_SK
#define RSWA_GQA_SK 1
#endif

// The cluster path when every head's cache fits one row batch per CTA of a
// cluster of at most 8 (longer caches are the split-K path's job) and all
// clusters fit in one wave of the device's SMs (two CTAs per SM).
bool decode_use_small(const CacheView& cv) {
  const int cl = cluster_size_for(cv);
  return cl <= kMaxCluster && (int64_t)cv.B * cv.H * cl <= 2 * (int64_t)cv.sms;
}

cudaError_t launch_decode(const CacheView& cv, const void* q, const void* k,
                          const void* v, void* o, float* lse, bool fused,
                          bool prefetch_prefix, cudaStream_t s) {
  const bool pf = prefetch_prefix;
  if (cv.H != cv.Hkv && !decode_use_small(cv)) {
    if (RSWA_GQA_TC && RSWA_GQA_SK && gqa_sk_supported(cv))
      return launch_decode_gqa_sk(cv, q, k, v, o, lse, fused, pf, s);
    if (RSWA_GQA_TC && gqa_tc_supported(cv))
      return launch_decode_gqa_tc(cv, q, k, v, o, lse, fused, pf, s);
    if (decode_gqa_heads_per_cta(cv) > 1)
      return launch_decode_gqa(cv, q, k, v, o, lse, fused, s);
  }
  if (cv.dtype == RSWA_F32) {
    if (cv.d == 64)
      return launch_decode_t<float, 64>(cv, q, k, v, o, lse, fused, pf, s);
    return launch_decode_t<float, 128>(cv, q, k, v, o, lse, fused, pf, s);
  }
  if (cv.d == 64)
    return launch_decode_t<__nv_bfloat16, 64>(cv, q, k, v, o, lse, fused, pf, s);
  return launch_decode_t<__nv_bfloat16, 128>(cv, q, k, v, o, lse, fused, pf, s);
}

// Partial slots per (b, h) of the decode path launch_decode takes for cv.
int decode_part_slots(const CacheView& cv) {
  if (cv.H != cv.Hkv && !decode_use_small(cv) && RSWA_GQA_TC && RSWA_GQA_SK &&
      gqa_sk_supported(cv)) {
    // a KV head's partials: at most one per tile of its list
    const int th = (int)((cv.m_cap + 127) / 128 + (cv.n + 127) / 128);
    return std::max(cv.max_chunks, th + 1);
  }
  if (!decode_use_small(cv) && RSWA_STREAM_DECODE && decode_use_stream(cv) &&
      !(cv.H != cv.Hkv && ((RSWA_GQA_TC && gqa_tc_supported(cv)) ||
                           decode_gqa_heads_per_cta(cv) > 1)))
    return std::max(cv.max_chunks, decode_stream_splits(cv));
  return cv.max_chunks;
}

}  // namespace rswa
