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

// Attend logical rows [j_begin, j_end) of a key/value table whose physical
// row p starts at Kb + p * stride (elements); logical row r maps to
// p = r for r < seg_end and p = r + gap beyond it (two segments of one
// table, e.g. the prefix rows and the ring slots of a cache slab).  This warp
// takes the rows j_begin + first + it * step + (0 .. KEYS_WARP-1).  A row
// whose physical index equals sub_row is read from (knew, vnew) instead.
template <typename T, int D, int UNROLL = RSWA_DECODE_UNROLL>
__device__ __forceinline__ void attend_range(
    const float* qf, const T* __restrict__ Kb, const T* __restrict__ Vb,
    int64_t stride, int64_t j_begin, int64_t j_end, int64_t first,
    int64_t step, int64_t sub_row, const T* knew, const T* vnew, int lane,
    SoftmaxState<AttendCfg<T, D>::EPL>& st, int64_t seg_end = INT64_MAX,
    int64_t gap = 0) {
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
      const int64_t lr = ok[u] ? row : j_begin;
      const int64_t r = lr < seg_end ? lr : lr + gap;
      const T* kp = Kb + r * stride + col;
      const T* vp = Vb + r * stride + col;
      if (r == sub_row) {
        kp = knew + col;
        vp = vnew + col;
      }
      kr[u] = ld_stream16(kp);
      vr[u] = ld_stream16(vp);
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
    float mx = st.m;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!ok[u]) s[u] = -INFINITY;
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
      Elt<T>::widen(vr[u], vf);
#pragma unroll
      for (int e = 0; e < EPL; ++e) st.acc[e] = fmaf(p, vf[e], st.acc[e]);
    }
    st.m = mx;
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

}  // namespace rswa
