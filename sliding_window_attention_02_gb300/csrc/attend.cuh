// Warp-level streaming attention over a contiguous range of key rows.
//
// Lane mapping: a key row of D elements is LPK = D / EPL lanes wide (EPL
// elements = 16 bytes per lane), so one warp load covers KPW = 32 / LPK
// consecutive rows.  Each lane keeps its own running softmax state for the
// rows its lane group sees; groups are merged at the end with shuffles.
// Every lane issues U independent 16-byte loads of K and of V before it uses
// any of them, which keeps 2 * U * 16 bytes per lane in flight.
#pragma once

#include "rswa_device.cuh"

namespace rswa {

#ifndef RSWA_DECODE_UNROLL
#define RSWA_DECODE_UNROLL 8
#endif

template <typename T, int D, int UNROLL = RSWA_DECODE_UNROLL>
struct AttendCfg {
  static constexpr int EPL = Elt<T>::kPerVec;
  static constexpr int LPK = D / EPL;
  static constexpr int KPW = 32 / LPK;
  static constexpr int U = UNROLL;
  static constexpr int KEYS_WARP = U * KPW;
  static_assert(D % EPL == 0 && 32 % LPK == 0, "unsupported head_dim");
};

// Load this lane's q fragment, pre-scaled by (1/sqrt(D)) * log2(e).
template <typename T, int D>
__device__ __forceinline__ void load_q_frag(const T* q_row, int lane,
                                            float* qf) {
  using C = AttendCfg<T, D>;
  const uint4 raw = *reinterpret_cast<const uint4*>(
      q_row + (lane % C::LPK) * C::EPL);
  Elt<T>::widen(raw, qf);
  const float sc = rsqrtf((float)D) * kLog2e;
#pragma unroll
  for (int e = 0; e < C::EPL; ++e) qf[e] *= sc;
}

// Evict-first L2 policy for keys and values a launch reads once (a cache
// streamed from HBM): the streamed rows are the first victims, so they do not
// displace the split-K partials, q and the per-sequence state.
__device__ __forceinline__ uint64_t stream_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 16-byte load through the read-only path, no L1 allocation, with the L2
// eviction policy `pol`.
__device__ __forceinline__ uint4 ld_stream16_hint(const void* p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}

// One batch of a warp's rows for attend_range: this lane's 16-byte slices
// of the U rows of K and V its lane group takes, and which of them are keys.
template <typename T, int D, int UNROLL = RSWA_DECODE_UNROLL>
struct AttendBatch {
  uint4 k[UNROLL], v[UNROLL];
  bool ok[UNROLL];
};

// Load the batch starting at logical row `base` (see attend_range for the
// row mapping); rows at or past j_end are flagged and read row j_begin.
// EVF: the rows are loaded with the L2 policy `pol` (stream_policy).
template <typename T, int D, int UNROLL = RSWA_DECODE_UNROLL, bool EVF = false>
__device__ __forceinline__ void attend_load(
    const T* __restrict__ Kb, const T* __restrict__ Vb, int64_t stride,
    int64_t base, int64_t j_begin, int64_t j_end, int64_t sub_row,
    const T* knew, const T* vnew, int lane, int64_t seg_end, int64_t gap,
    AttendBatch<T, D, UNROLL>& bt, uint64_t pol = 0) {
  using C = AttendCfg<T, D, UNROLL>;
  constexpr int EPL = C::EPL, LPK = C::LPK, KPW = C::KPW, U = C::U;
  const int grp = lane / LPK;
  const int col = (lane % LPK) * EPL;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t row = base + u * KPW + grp;
    bt.ok[u] = row < j_end;
    const int64_t lr = bt.ok[u] ? row : j_begin;
    const int64_t r = lr < seg_end ? lr : lr + gap;
    const T* kp = Kb + r * stride + col;
    const T* vp = Vb + r * stride + col;
    if (r == sub_row) {
      kp = knew + col;
      vp = vnew + col;
    }
    if constexpr (EVF) {
      bt.k[u] = ld_stream16_hint(kp, pol);
      bt.v[u] = ld_stream16_hint(vp, pol);
    } else {
      bt.k[u] = ld_stream16(kp);
      bt.v[u] = ld_stream16(vp);
    }
  }
}

// Fold a loaded batch into this lane's online-softmax state.
template <typename T, int D, int UNROLL = RSWA_DECODE_UNROLL>
__device__ __forceinline__ void attend_consume(
    const float* qf, const AttendBatch<T, D, UNROLL>& bt,
    SoftmaxState<AttendCfg<T, D>::EPL>& st) {
  using C = AttendCfg<T, D, UNROLL>;
  constexpr int EPL = C::EPL, LPK = C::LPK, U = C::U;
  float s[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    float kf[EPL];
    Elt<T>::widen(bt.k[u], kf);
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
  float mx = st.m;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (!bt.ok[u]) s[u] = -INFINITY;
    mx = fmaxf(mx, s[u]);
  }
  const float ref = (mx == -INFINITY) ? 0.f : mx;
  const float alpha = fast_exp2(st.m - ref);
  st.l *= alpha;
#pragma unroll
  for (int e = 0; e < EPL; ++e) st.acc[e] *= alpha;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const float p = fast_exp2(s[u] - ref);
    st.l += p;
    float vf[EPL];
    Elt<T>::widen(bt.v[u], vf);
#pragma unroll
    for (int e = 0; e < EPL; ++e) st.acc[e] = fmaf(p, vf[e], st.acc[e]);
  }
  st.m = mx;
}

// Attend logical rows [j_begin, j_end) of a key/value table whose physical
// row p starts at Kb + p * stride (elements); logical row r maps to
// p = r for r < seg_end and p = r + gap beyond it (two segments of one
// table, e.g. the prefix rows and the ring slots of a cache slab).  This warp
// takes the rows j_begin + first + it * step + (0 .. KEYS_WARP-1).  A row
// whose physical index equals sub_row is read from (knew, vnew) instead.
template <typename T, int D, int UNROLL = RSWA_DECODE_UNROLL, bool EVF = false>
__device__ __forceinline__ void attend_range(
    const float* qf, const T* __restrict__ Kb, const T* __restrict__ Vb,
    int64_t stride, int64_t j_begin, int64_t j_end, int64_t first,
    int64_t step, int64_t sub_row, const T* knew, const T* vnew, int lane,
    SoftmaxState<AttendCfg<T, D>::EPL>& st, int64_t seg_end = INT64_MAX,
    int64_t gap = 0, uint64_t pol = 0) {
  for (int64_t base = j_begin + first; base < j_end; base += step) {
    AttendBatch<T, D, UNROLL> bt;
    attend_load<T, D, UNROLL, EVF>(Kb, Vb, stride, base, j_begin, j_end, sub_row, knew,
                                   vnew, lane, seg_end, gap, bt, pol);
    attend_consume<T, D, UNROLL>(qf, bt, st);
  }
}

// Merge the lane groups of a warp; afterwards lanes 0..LPK-1 hold the warp's
// state for columns lane*EPL .. lane*EPL+EPL-1 (all groups agree).
template <typename T, int D>
__device__ __forceinline__ void merge_groups(SoftmaxState<AttendCfg<T, D>::EPL>& st) {
  using C = AttendCfg<T, D>;
#pragma unroll
  for (int off = C::LPK; off < 32; off <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, st.m, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, st.l, off);
    float a2[C::EPL];
#pragma unroll
    for (int e = 0; e < C::EPL; ++e)
      a2[e] = __shfl_xor_sync(0xffffffffu, st.acc[e], off);
    st.merge(m2, l2, a2);
  }
}

}  // namespace rswa

namespace rswa {

// attend_range for G query heads that share one KV head: every K and V row
// is loaded once and feeds G dot products and G softmax states.  qf holds
// the G heads' fragments back to back (G * EPL floats).
template <typename T, int D, int UNROLL, int G>
__device__ __forceinline__ void attend_range_grouped(
    const float* qf, const T* __restrict__ Kb, const T* __restrict__ Vb,
    int64_t stride, int64_t j_begin, int64_t j_end, int64_t first,
    int64_t step, int64_t sub_row, const T* knew, const T* vnew, int lane,
    SoftmaxState<AttendCfg<T, D>::EPL>* st) {
  using C = AttendCfg<T, D, UNROLL>;
  constexpr int EPL = C::EPL, LPK = C::LPK, KPW = C::KPW, U = C::U;
  const int grp = lane / LPK;
  const int col = (lane % LPK) * EPL;
  for (int64_t base = j_begin + first; base < j_end; base += step) {
    uint4 kr[U], vr[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t row = base + u * KPW + grp;
      ok[u] = row < j_end;
      const int64_t r = ok[u] ? row : j_begin;
      const T* kp = Kb + r * stride + col;
      const T* vp = Vb + r * stride + col;
      if (r == sub_row) {
        kp = knew + col;
        vp = vnew + col;
      }
      kr[u] = ld_stream16(kp);
      vr[u] = ld_stream16(vp);
    }
    float s[G][U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float kf[EPL];
      Elt<T>::widen(kr[u], kf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc = fmaf(qf[g * EPL + e], kf[e], acc);
        s[g][u] = acc;
      }
    }
#pragma unroll
    for (int off = LPK / 2; off > 0; off >>= 1) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int u = 0; u < U; ++u)
          s[g][u] += __shfl_xor_sync(0xffffffffu, s[g][u], off);
    }
    float p[G][U];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float mx = st[g].m;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (!ok[u]) s[g][u] = -INFINITY;
        mx = fmaxf(mx, s[g][u]);
      }
      const float ref = (mx == -INFINITY) ? 0.f : mx;
      const float alpha = fast_exp2(st[g].m - ref);
      st[g].l *= alpha;
#pragma unroll
      for (int e = 0; e < EPL; ++e) st[g].acc[e] *= alpha;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        p[g][u] = fast_exp2(s[g][u] - ref);
        st[g].l += p[g][u];
      }
      st[g].m = mx;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float vf[EPL];
      Elt<T>::widen(vr[u], vf);
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < EPL; ++e) st[g].acc[e] = fmaf(p[g][u], vf[e], st[g].acc[e]);
    }
  }
}

// attend_range for G query heads of one KV head with U = LPK / G rows per
// lane group and iteration, so that the G * U partial dot products of a lane
// group are exactly LPK values.  A butterfly reduce-scatter over the LPK
// lanes (offsets LPK/2 .. 1, each level keeping the half of the values
// named by the lane's bit at that offset) leaves lane pos of the group with
// the full score of head pos / U and row pos % U: 15 shuffles for 16 scores
// instead of 64, and one exp2 per lane.  Each lane then keeps the running
// maximum of every head (identical in all lanes), the partial sum l of its
// own (head, row) slot, and its EPL columns of every head's accumulator; the
// probabilities reach all lanes by shuffle for the value update.  Dot
// products and value updates use the packed f32x2 FMA.  On return st[g]
// holds m, l (summed over the head's U lanes) and acc, as attend_range_grouped
// leaves them.
template <typename T, int D, int G>
struct GroupedRsCfg {
  static constexpr int EPL = Elt<T>::kPerVec;
  static constexpr int LPK = D / EPL;
  static constexpr int KPW = 32 / LPK;
  static constexpr int U = LPK / G;
  static constexpr int KEYS_WARP = U * KPW;
  static constexpr bool kUsable = G * U == LPK && U >= 1 && U <= 8 && EPL % 2 == 0;
};

// Per-lane running state of the reduce-scatter loop: packed q pairs and
// accumulators of the G heads, every head's running maximum (identical in
// all lanes) and the maximum and partial sum of this lane's own head.
template <typename T, int D, int G>
struct GroupedRsState {
  static constexpr int NP = GroupedRsCfg<T, D, G>::EPL / 2;
  uint64_t q2[G][NP], a2[G][NP];
  float m[G];
  float m_own, l_own;

  __device__ __forceinline__ void init(const float* qf) {
    constexpr int EPL = GroupedRsCfg<T, D, G>::EPL;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        q2[g][i] = f2_pack(qf[g * EPL + 2 * i], qf[g * EPL + 2 * i + 1]);
        a2[g][i] = 0;
      }
    }
    m_own = -INFINITY;
    l_own = 0.f;
  }

  // One batch: the lane group's U rows (kr, vr: this lane's 16-byte slices;
  // ok[u]: row u is a key; a row that is not has its value taken as 0, so
  // any bits may stand in kr/vr for it).  pos = lane % LPK.
  __device__ __forceinline__ void step(const uint4* kr, uint4* vr,
                                       const bool* ok, int pos) {
    using C = GroupedRsCfg<T, D, G>;
    constexpr int EPL = C::EPL, LPK = C::LPK, U = C::U;
    const int my_u = pos % U;
    float v[G * U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float kf[EPL];
      Elt<T>::widen(kr[u], kf);
      uint64_t k2[NP];
#pragma unroll
      for (int i = 0; i < NP; ++i) k2[i] = f2_pack(kf[2 * i], kf[2 * i + 1]);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        uint64_t acc = 0;
#pragma unroll
        for (int i = 0; i < NP; ++i) acc = f2_fma(q2[g][i], k2[i], acc);
        float lo, hi;
        f2_unpack(acc, lo, hi);
        v[g * U + u] = lo + hi;
      }
    }
    // reduce-scatter: value index g*U+u ends in lane pos = g*U+u
#pragma unroll
    for (int o = LPK / 2, n = LPK; o > 0; o >>= 1, n >>= 1) {
      const bool up = (pos & o) != 0;
#pragma unroll
      for (int j = 0; j < n / 2; ++j) {
        const float send = up ? v[j] : v[j + n / 2];
        const float keep = up ? v[j + n / 2] : v[j];
        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    bool ok_own = ok[0];
#pragma unroll
    for (int u = 1; u < U; ++u)
      if (my_u == u) ok_own = ok[u];
    const float s_own = ok_own ? v[0] : -INFINITY;
    float mx_own = s_own;
#pragma unroll
    for (int o = U / 2; o > 0; o >>= 1)
      mx_own = fmaxf(mx_own, __shfl_xor_sync(0xffffffffu, mx_own, o));
    // every head's new maximum, in every lane; the accumulators are
    // rescaled only when some head's maximum grew (alpha is exactly 1
    // otherwise)
    float mn[G];
    bool grew = false;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      mn[g] = fmaxf(m[g], __shfl_sync(0xffffffffu, mx_own, g * U, LPK));
      grew |= mn[g] > m[g];
    }
    if (__any_sync(0xffffffffu, grew)) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float ref = (mn[g] == -INFINITY) ? 0.f : mn[g];
        const float alpha = fast_exp2(m[g] - ref);
        const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll
        for (int i = 0; i < NP; ++i) a2[g][i] = f2_mul(a2[g][i], al2);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) m[g] = mn[g];
    const float mo = fmaxf(m_own, mx_own);
    const float ref_own = (mo == -INFINITY) ? 0.f : mo;
    const float alpha_own = fast_exp2(m_own - ref_own);
    m_own = mo;
    const float p_own = fast_exp2(s_own - ref_own);
    l_own = l_own * alpha_own + p_own;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!ok[u]) vr[u] = make_uint4(0, 0, 0, 0);
      float vf[EPL];
      Elt<T>::widen(vr[u], vf);
      uint64_t v2[NP];
#pragma unroll
      for (int i = 0; i < NP; ++i) v2[i] = f2_pack(vf[2 * i], vf[2 * i + 1]);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float p = __shfl_sync(0xffffffffu, p_own, g * U + u, LPK);
        const uint64_t p2 = f2_pack(p, p);
#pragma unroll
        for (int i = 0; i < NP; ++i) a2[g][i] = f2_fma(p2, v2[i], a2[g][i]);
      }
    }
  }

  // st[g] = (m, l summed over the head's U lanes, this lane's acc columns).
  __device__ __forceinline__ void finish(SoftmaxState<GroupedRsCfg<T, D, G>::EPL>* st) {
    using C = GroupedRsCfg<T, D, G>;
    constexpr int LPK = C::LPK, U = C::U;
    float l_sum = l_own;
#pragma unroll
    for (int o = U / 2; o > 0; o >>= 1) l_sum += __shfl_xor_sync(0xffffffffu, l_sum, o);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      st[g].m = m[g];
      st[g].l = __shfl_sync(0xffffffffu, l_sum, g * U, LPK);
#pragma unroll
      for (int i = 0; i < NP; ++i)
        f2_unpack(a2[g][i], st[g].acc[2 * i], st[g].acc[2 * i + 1]);
    }
  }
};

// The reduce-scatter loop over a contiguous range of rows read straight
// from global memory (16-byte loads, U rows in flight per lane).
template <typename T, int D, int G>
__device__ __forceinline__ void attend_range_grouped_rs(
    const float* qf, const T* __restrict__ Kb, const T* __restrict__ Vb,
    int64_t stride, int64_t j_begin, int64_t j_end, int64_t first,
    int64_t step, int64_t sub_row, const T* knew, const T* vnew, int lane,
    SoftmaxState<AttendCfg<T, D>::EPL>* st) {
  using C = GroupedRsCfg<T, D, G>;
  constexpr int EPL = C::EPL, LPK = C::LPK, KPW = C::KPW, U = C::U;
  static_assert(C::kUsable, "reduce-scatter shape");
  const int grp = lane / LPK, pos = lane % LPK;
  const int col = pos * EPL;
  GroupedRsState<T, D, G> rs;
  rs.init(qf);
  for (int64_t base = j_begin + first; base < j_end; base += step) {
    uint4 kr[U], vr[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t row = base + u * KPW + grp;
      ok[u] = row < j_end;
      const int64_t r = ok[u] ? row : j_begin;
      const T* kp = Kb + r * stride + col;
      const T* vp = Vb + r * stride + col;
      if (r == sub_row) {
        kp = knew + col;
        vp = vnew + col;
      }
      kr[u] = ld_stream16(kp);
      vr[u] = ld_stream16(vp);
    }
    rs.step(kr, vr, ok, pos);
  }
  rs.finish(st);
}

}  // namespace rswa
