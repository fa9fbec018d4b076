// Device helpers shared by the R-SWA kernels.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "rswa_internal.h"

namespace rswa {

// log2(e): logits are pre-scaled by (1/sqrt(d)) * log2(e) so that the softmax
// uses exp2.
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device error codes written to CacheView::err (first one wins).
enum DeviceErr : int32_t {
  kErrNone = 0,
  kErrWaitTimeout = 1,
  kErrLaunchShape = 2,   // a launch whose grid does not cover its work
};

__device__ __forceinline__ void flag_error(int32_t* err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

// 2^x on the special-function unit (ex2.approx.ftz: relative error about
// 2^-22; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Programmatic dependent launch: wait for the preceding grid of the stream
// (a no-op when the kernel was not launched as a dependent), and allow the
// next grid to begin launching.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Thread-block clusters: rank and size of this CTA's cluster, the two halves
// of the cluster barrier, and the cluster address of `p` in CTA `rank`.  An
// arrive with release semantics followed by a wait with acquire semantics
// makes every shared-memory write issued before the arrive (local or remote,
// mbarrier initialisation included) visible to every CTA after the wait.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive without ordering any memory operation (every thread of the CTA
// executes it together), and a wait that a subset of a warp may execute.
// A wait returns once every thread of the cluster that has not exited has
// arrived at the current phase.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_divergent() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_dsmem(const void* p, uint32_t rank) {
  const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}
// Asynchronous 4-byte store into another CTA's shared memory: `dst` and the
// mbarrier `bar` are cluster addresses from map_dsmem; on arrival the store
// completes 4 transaction bytes of that CTA's mbarrier.
__device__ __forceinline__ void st_async_f32(uint32_t dst, uint32_t bar, float v) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
      :: "r"(dst), "r"(__float_as_uint(v)), "r"(bar) : "memory");
}

// Two float32 values in one 64-bit register for the packed f32x2 arithmetic
// of sm_100 and later: each half is rounded like the scalar instruction.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max(a, b, c) in one instruction (sm_100 and later); -inf and NaN operands
// behave as for fmaxf.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Maximum of v over the 32 lanes of the warp, in one instruction (sm_100 and
// later); -inf operands behave as for fmaxf.
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Arrival on a split-K counter: atomically adds 1 with release and acquire
// semantics at GPU scope and returns the old value.  Issued by one thread
// after a CTA barrier, the release orders every store the CTA made before
// the barrier (the CTA's partial) before the increment; the acquire orders
// the increment before the loads that follow, so the last CTA to arrive
// sees every other CTA's partial.  Replaces a fence, a relaxed add and a
// second fence.
__device__ __forceinline__ int arrive_acq_rel(int32_t* counter) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;"
               : "=r"(old)
               : "l"(counter)
               : "memory");
  return old;
}

// 16-byte streaming load through the read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Element traits: how many elements a 16-byte vector holds and how to widen.
template <typename T>
struct Elt;

template <>
struct Elt<float> {
  static constexpr int kPerVec = 4;
  __device__ __forceinline__ static void widen(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static uint4 narrow(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                      __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
};

template <>
struct Elt<__nv_bfloat16> {
  static constexpr int kPerVec = 8;
  // bf16 -> f32 is exact: the bf16 bits are the top half of the f32 bits.
  __device__ __forceinline__ static void widen(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static uint4 narrow(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// Running softmax state in log2 units: max m, sum l (relative to m) and the
// weighted value accumulator acc (relative to m).
template <int E>
struct SoftmaxState {
  float m, l;
  float acc[E];
  __device__ __forceinline__ void init() {
    m = -INFINITY;
    l = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
  }
  // Merge another state into this one.
  __device__ __forceinline__ void merge(float m2, float l2, const float* a2) {
    const float mn = fmaxf(m, m2);
    const float ref = (mn == -INFINITY) ? 0.f : mn;
    const float s1 = fast_exp2(m - ref);
    const float s2 = fast_exp2(m2 - ref);
    l = l * s1 + l2 * s2;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = acc[e] * s1 + a2[e] * s2;
    m = mn;
  }
};

// Online merge of split-K partials (m, l, acc[D]) in log2 units: chunks
// 0..nch-1 of NG heads, head g's chunk k at P0 + g * hs + k * (D + 2); this
// thread's column is col (acc ignored when col >= D).  KB chunks of every
// head are loaded before any of them is used, so a merge costs
// ceil(nch / KB) load round trips rather than two per chunk.  On return
// M[g] is the reference maximum, L[g] the sum and A[g] the column, both
// relative to M[g] (L[g] = 0 for a head with no visible key).
template <int NG, int KB>
__device__ __forceinline__ void merge_partials(const float* P0, size_t hs,
                                               int nch, int D, int col,
                                               int ng, float* M, float* L,
                                               float* A) {
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    M[g] = -INFINITY;
    L[g] = 0.f;
    A[g] = 0.f;
  }
  for (int k0 = 0; k0 < nch; k0 += KB) {
    float mk[NG][KB], lk[NG][KB], ak[NG][KB];
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int u = 0; u < KB; ++u) {
        mk[g][u] = -INFINITY;
        lk[g][u] = 0.f;
        ak[g][u] = 0.f;
        if (g < ng && k0 + u < nch) {
          const float* P = P0 + g * hs + (size_t)(k0 + u) * (D + 2);
          mk[g][u] = __ldcg(P);
          lk[g][u] = __ldcg(P + 1);
          if (col < D) ak[g][u] = __ldcg(P + 2 + col);
        }
      }
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      float mn = M[g];
#pragma unroll
      for (int u = 0; u < KB; ++u) mn = fmaxf(mn, mk[g][u]);
      const float ref = (mn == -INFINITY) ? 0.f : mn;
      const float sc = fast_exp2(M[g] - ref);
      L[g] *= sc;
      A[g] *= sc;
#pragma unroll
      for (int u = 0; u < KB; ++u) {
        const float w = fast_exp2(mk[g][u] - ref);
        L[g] += lk[g][u] * w;
        A[g] += ak[g][u] * w;
      }
      M[g] = mn;
    }
  }
}

}  // namespace rswa
