// R-SWA prefill on CUDA cores: one warp per (row, head).
//
// Row i of a sequence with prefix m attends to keys [0, min(m, i + 1)) and,
// for an output row (i >= m), to the window [max(m, i - n + 1), i]
// ("Unlimited-OCR deep dive", N(t) = P U D_n(t)).  The two key ranges are
// streamed with the same warp routine as the decode step.  This kernel serves
// float32 caches (where tensor-core tf32 would not hold float32 accuracy);
// bf16 caches run on the tcgen05 kernel.
#include "attend.cuh"

namespace rswa {

template <typename T, int D>
__global__ void __launch_bounds__(128)
prefill_rowwise_kernel(CacheView cv, SeqTable st, const T* __restrict__ Q,
                       const T* __restrict__ K, const T* __restrict__ V,
                       T* __restrict__ O, int64_t total_rows) {
  using C = AttendCfg<T, D>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t g = (int64_t)blockIdx.x * 4 + warp;  // row in this launch
  const int h = blockIdx.y;
  if (g >= total_rows) return;
  int sl = 0;
  while (sl + 1 < st.nseq && st.row_off[sl + 1] <= st.row_off[0] + g) ++sl;
  const int64_t grow = st.row_off[0] + g;            // absolute input row
  const int64_t i = grow - st.row_off[sl];           // row within sequence
  const int64_t m = st.m[sl];
  const int H = cv.H;
  const int64_t stride = (int64_t)H * D;          // Q, O: [rows][H][D]
  const int64_t kstride = (int64_t)cv.Hkv * D;    // K, V: [rows][Hkv][D]
  const int kvh = h / (H / cv.Hkv);
  const T* Kb = K + st.row_off[sl] * kstride + (int64_t)kvh * D;
  const T* Vb = V + st.row_off[sl] * kstride + (int64_t)kvh * D;

  float qf[C::EPL];
  load_q_frag<T, D>(Q + grow * stride + (int64_t)h * D, lane, qf);
  SoftmaxState<C::EPL> s;
  s.init();
  attend_range<T, D>(qf, Kb, Vb, kstride, 0, min(m, i + 1), 0, C::KEYS_WARP,
                     -1, nullptr, nullptr, lane, s);
  if (i >= m)
    attend_range<T, D>(qf, Kb, Vb, kstride, max(m, i - cv.n + 1), i + 1, 0,
                       C::KEYS_WARP, -1, nullptr, nullptr, lane, s);
  merge_groups<T, D>(s);
  if (lane < C::LPK) {
    float out[C::EPL];
    const float inv = 1.f / s.l;
#pragma unroll
    for (int e = 0; e < C::EPL; ++e) out[e] = s.acc[e] * inv;
    *reinterpret_cast<uint4*>(O + grow * stride + (int64_t)h * D +
                              lane * C::EPL) = Elt<T>::narrow(out);
  }
}

template <typename T, int D>
static cudaError_t launch_rw(const CacheView& cv, const SeqTable& st,
                             const void* Q, const void* K, const void* V,
                             void* O, int64_t total_rows, cudaStream_t s) {
  dim3 grid((unsigned)((total_rows + 3) / 4), (unsigned)cv.H);
  prefill_rowwise_kernel<T, D><<<grid, 128, 0, s>>>(
      cv, st, (const T*)Q, (const T*)K, (const T*)V, (T*)O, total_rows);
  return cudaGetLastError();
}

cudaError_t launch_prefill_rowwise(const CacheView& cv, const SeqTable& st,
                                   const void* Q, const void* K, const void* V,
                                   void* O, int64_t total_rows,
                                   cudaStream_t s) {
  if (total_rows <= 0) return cudaSuccess;
  if (cv.dtype == RSWA_F32) {
    if (cv.d == 64) return launch_rw<float, 64>(cv, st, Q, K, V, O, total_rows, s);
    return launch_rw<float, 128>(cv, st, Q, K, V, O, total_rows, s);
  }
  if (cv.d == 64)
    return launch_rw<__nv_bfloat16, 64>(cv, st, Q, K, V, O, total_rows, s);
  return launch_rw<__nv_bfloat16, 128>(cv, st, Q, K, V, O, total_rows, s);
}

}  // namespace rswa
