// R-SWA decode of a block of k consecutive output tokens per sequence.
//
// Output t_b + i (i = 0..k-1) attends to the prefix, to the outputs of its
// window already in the cache, j in [max(0, t_b + i - n + 1), t_b), and to
// block tokens 0..i (k <= n keeps every earlier block token inside the
// window).  The attention kernel reads the ring before the append kernel
// overwrites any slot; both run on the caller's stream in that order.
// This is the shape of a speculative-verification forward or of chunked
// prefill of output text into an existing cache.
#include "attend.cuh"

namespace rswa {

// One warp per (b, i, h); 4 warps per CTA over consecutive (i, h).
template <typename T, int D>
__global__ void __launch_bounds__(128)
decode_block_kernel(CacheView cv, const T* __restrict__ q,
                    const T* __restrict__ kblk, const T* __restrict__ vblk,
                    int64_t k, T* __restrict__ o, float* __restrict__ lse) {
  using C = AttendCfg<T, D>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.y;
  const int64_t qi = (int64_t)blockIdx.x * 4 + warp;
  if (qi >= k * cv.H) return;
  const int64_t i = qi / cv.H;
  const int h = (int)(qi % cv.H);
  const size_t bh = (size_t)b * cv.H + h;
  const int kvh = h / (cv.H / cv.Hkv);
  const size_t bkv = (size_t)b * cv.Hkv + kvh;
  const int64_t m_b = cv.m_dev[b];
  const int64_t t_b = cv.t_dev[bh];
  const int64_t n = cv.n;
  const int64_t row_stride = (int64_t)cv.Hkv * D;        // k, v: [B][k][Hkv][D]
  const size_t qrow = ((size_t)b * k + i) * cv.H + h;    // q, o: [B][k][H][D]

  float qf[C::EPL];
  load_q_frag<T, D>(q + qrow * D, lane, qf);
  SoftmaxState<C::EPL> st;
  st.init();
  const T* Kb = static_cast<const T*>(cv.K) + bkv * cv.slab_rows * D;
  const T* Vb = static_cast<const T*>(cv.V) + bkv * cv.slab_rows * D;
  // prefix
  attend_range<T, D>(qf, Kb, Vb, D, 0, m_b, 0, C::KEYS_WARP, -1, nullptr,
                     nullptr, lane, st);
  // cached outputs of the window: j in [j_lo, t_b), slot j mod n
  const int64_t j_lo = max((int64_t)0, t_b + i - n + 1);
  if (j_lo < t_b) {
    const T* Kr = Kb + cv.m_cap * D;
    const T* Vr = Vb + cv.m_cap * D;
    const int64_t a = j_lo % n, cnt = t_b - j_lo;
    const int64_t first_end = min(n, a + cnt);
    attend_range<T, D>(qf, Kr, Vr, D, a, first_end, 0, C::KEYS_WARP, -1, nullptr,
                       nullptr, lane, st);
    if (a + cnt > n)
      attend_range<T, D>(qf, Kr, Vr, D, 0, a + cnt - n, 0, C::KEYS_WARP, -1,
                         nullptr, nullptr, lane, st);
  }
  // block tokens 0..i (rows of the input, stride H*D)
  const T* Kk = kblk + ((size_t)b * k * cv.Hkv + kvh) * D;
  const T* Vk = vblk + ((size_t)b * k * cv.Hkv + kvh) * D;
  attend_range<T, D>(qf, Kk, Vk, row_stride, 0, i + 1, 0, C::KEYS_WARP, -1,
                     nullptr, nullptr, lane, st);
  merge_groups<T, D>(st);
  if (lane < C::LPK) {
    float out[C::EPL];
    const float inv = 1.f / st.l;
#pragma unroll
    for (int e = 0; e < C::EPL; ++e) out[e] = st.acc[e] * inv;
    *reinterpret_cast<uint4*>(o + qrow * D + lane * C::EPL) = Elt<T>::narrow(out);
    if (lane == 0 && lse) lse[qrow] = (st.m + log2f(st.l)) * kLn2;
  }
}

// One CTA per sequence: block token i -> ring slot (t_b + i) mod n for every
// KV head, then t_b += k for every query head (after every thread has read
// t_b).
template <typename T, int D>
__global__ void __launch_bounds__(128)
append_block_kernel(CacheView cv, const T* __restrict__ kblk,
                    const T* __restrict__ vblk, int64_t k) {
  const int b = blockIdx.x;
  const int H = cv.Hkv;                          // k, v carry the KV heads
  const int64_t t_b = cv.t_dev[(size_t)b * cv.H];
  constexpr int NV = D * sizeof(T) / 16;
  const int64_t total = 2 * k * H * NV;
  for (int64_t x = threadIdx.x; x < total; x += blockDim.x) {
    const int kv = (int)(x / (k * H * NV));
    const int64_t rest = x % (k * H * NV);
    const int64_t i = rest / (H * NV);
    const int h = (int)((rest / NV) % H);
    const int vi = (int)(rest % NV);
    const T* in = (kv ? vblk : kblk) + (((size_t)b * k + i) * H + h) * D;
    const int64_t slot = (t_b + i) % cv.n;
    T* out = static_cast<T*>(kv ? cv.V : cv.K) +
             (((size_t)b * H + h) * cv.slab_rows + cv.m_cap + slot) * D;
    reinterpret_cast<uint4*>(out)[vi] = reinterpret_cast<const uint4*>(in)[vi];
  }
  __syncthreads();
  for (int h = threadIdx.x; h < cv.H; h += blockDim.x)
    cv.t_dev[(size_t)b * cv.H + h] = t_b + k;
}

template <typename T, int D>
static cudaError_t launch_block_t(const CacheView& cv, const void* q,
                                  const void* k, const void* v, int64_t block,
                                  void* o, float* lse, cudaStream_t s) {
  const int64_t nq = block * cv.H;
  dim3 grid((unsigned)((nq + 3) / 4), (unsigned)cv.B);
  decode_block_kernel<T, D><<<grid, 128, 0, s>>>(cv, (const T*)q, (const T*)k,
                                                 (const T*)v, block, (T*)o, lse);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  append_block_kernel<T, D><<<cv.B, 128, 0, s>>>(cv, (const T*)k, (const T*)v, block);
  return cudaGetLastError();
}

cudaError_t launch_decode_block(const CacheView& cv, const void* q, const void* k,
                                const void* v, int64_t block, void* o, float* lse,
                                cudaStream_t s) {
  if (cv.dtype == RSWA_F32) {
    if (cv.d == 64) return launch_block_t<float, 64>(cv, q, k, v, block, o, lse, s);
    return launch_block_t<float, 128>(cv, q, k, v, block, o, lse, s);
  }
  if (cv.d == 64)
    return launch_block_t<__nv_bfloat16, 64>(cv, q, k, v, block, o, lse, s);
  return launch_block_t<__nv_bfloat16, 128>(cv, q, k, v, block, o, lse, s);
}

}  // namespace rswa
