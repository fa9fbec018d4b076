// Cache manager kernels: the prefill KV write and the per-step append.
//
// The cache of sequence b is a slab per head, [m_cap + n][d]: rows
// 0..m_cap-1 hold the static prefix (written once at prefill, "encoded once,
// no state transition", GeekNews, model architecture), rows m_cap..m_cap+n-1
// the ring of output KV, where output j lives in slot j mod n (the queue of
// capacity m + n that evicts its (m+1)-th entry).
#include <vector>

#include "rswa_device.cuh"

namespace rswa {

// One CTA per (4 cache rows, sequence).  Cache row r of sequence b is prefix
// row r (r < m_b) or output j = T - min(n, T) + (r - m_b).
template <typename T>
__global__ void __launch_bounds__(128)
prefill_cache_kernel(CacheView cv, SeqTable st, const T* __restrict__ K,
                     const T* __restrict__ V) {
  const int sl = blockIdx.y;                // sequence within the launch
  const int b = st.seq0 + sl;
  const int64_t m_b = st.m[sl];
  const int64_t T_ = st.T[sl];
  const int64_t keep = min(cv.n, T_);       // outputs kept in the ring
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) cv.m_dev[b] = (int32_t)m_b;
    for (int h = threadIdx.x; h < cv.H; h += blockDim.x) cv.t_dev[(size_t)b * cv.H + h] = T_;
  }
  const int D = cv.d, H = cv.Hkv;           // K and V carry the KV heads
  const int nv = D * (int)sizeof(T) / 16;   // 16-byte vectors per head row
  for (int rr = 0; rr < 4; ++rr) {
    const int64_t r = (int64_t)blockIdx.x * 4 + rr;
    if (r >= m_b + keep) return;
    int64_t src, dst;
    if (r < m_b) {
      src = r;
      dst = r;
    } else {
      const int64_t j = T_ - keep + (r - m_b);
      src = m_b + j;
      dst = cv.m_cap + j % cv.n;
    }
    const int64_t in_row = st.row_off[sl] + src;
    for (int i = threadIdx.x; i < 2 * H * nv; i += blockDim.x) {
      const int kv = i / (H * nv);
      const int h = (i / nv) % H;
      const int vi = i % nv;
      const T* in = (kv ? V : K) + (in_row * H + h) * D;
      T* out = static_cast<T*>(kv ? cv.V : cv.K) +
               (((int64_t)b * H + h) * cv.slab_rows + dst) * D;
      reinterpret_cast<uint4*>(out)[vi] = reinterpret_cast<const uint4*>(in)[vi];
    }
  }
}

// One CTA per sequence: write k, v of every KV head to slot t_b mod n, then
// t_b += 1 for every query head (after every thread has read t_b).
template <typename T>
__global__ void __launch_bounds__(128)
append_kernel(CacheView cv, const T* __restrict__ k, const T* __restrict__ v) {
  const int b = blockIdx.x;
  const int64_t t_b = cv.t_dev[(size_t)b * cv.H];
  const int64_t slot = t_b % cv.n;
  const int D = cv.d, H = cv.Hkv;           // k, v: [B][Hkv][d]
  const int nv = D * (int)sizeof(T) / 16;
  for (int i = threadIdx.x; i < 2 * H * nv; i += blockDim.x) {
    const int kv = i / (H * nv);
    const int h = (i / nv) % H;
    const int vi = i % nv;
    const T* in = (kv ? v : k) + ((int64_t)b * H + h) * D;
    T* out = static_cast<T*>(kv ? cv.V : cv.K) +
             (((int64_t)b * H + h) * cv.slab_rows + cv.m_cap + slot) * D;
    reinterpret_cast<uint4*>(out)[vi] = reinterpret_cast<const uint4*>(in)[vi];
  }
  __syncthreads();
  for (int h = threadIdx.x; h < cv.H; h += blockDim.x)
    cv.t_dev[(size_t)b * cv.H + h] = t_b + 1;
}

cudaError_t launch_prefill_cache(const CacheView& cv, const SeqTable& st,
                                 const void* K, const void* V,
                                 int64_t max_rows, cudaStream_t s) {
  dim3 grid((unsigned)((max_rows + 3) / 4 > 0 ? (max_rows + 3) / 4 : 1),
            (unsigned)st.nseq);
  if (cv.dtype == RSWA_F32)
    prefill_cache_kernel<float><<<grid, 128, 0, s>>>(cv, st, (const float*)K,
                                                     (const float*)V);
  else
    prefill_cache_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(
        cv, st, (const __nv_bfloat16*)K, (const __nv_bfloat16*)V);
  return cudaGetLastError();
}

cudaError_t launch_append(const CacheView& cv, const void* k, const void* v,
                          cudaStream_t s) {
  if (cv.dtype == RSWA_F32)
    append_kernel<float><<<cv.B, 128, 0, s>>>(cv, (const float*)k,
                                              (const float*)v);
  else
    append_kernel<__nv_bfloat16><<<cv.B, 128, 0, s>>>(
        cv, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v);
  return cudaGetLastError();
}

cudaError_t launch_set_t(const CacheView& cv, const int64_t* t_host,
                         cudaStream_t s) {
  // A decode step that flagged an error may have left split-K arrival
  // counters part-way: restoring t_b clears them too.
  cudaError_t e = cudaMemsetAsync(cv.cnt_bh, 0, sizeof(int32_t) * (size_t)cv.B * cv.H, s);
  if (e != cudaSuccess) return e;
  // One copy of t_b per head; the caller synchronises before t_host and this
  // staging array go away.
  static thread_local std::vector<int64_t> per_head;
  per_head.assign((size_t)cv.B * cv.H, 0);
  for (int b = 0; b < cv.B; ++b)
    for (int h = 0; h < cv.H; ++h) per_head[(size_t)b * cv.H + h] = t_host[b];
  return cudaMemcpyAsync(cv.t_dev, per_head.data(), sizeof(int64_t) * per_head.size(),
                         cudaMemcpyHostToDevice, s);
}

}  // namespace rswa
