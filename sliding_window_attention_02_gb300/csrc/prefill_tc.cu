// R-SWA prefill on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// One CTA computes one 128-row query tile of one head:
//   O_i = softmax_{j in N(i)}(q_i . k_j / sqrt(d)) . v_j,
//   N(i) = {j <= i}                                   for prefix rows i < m,
//   N(i) = {j < m} U {j : max(m, i - n + 1) <= j <= i} for output rows,
// ("Unlimited-OCR deep dive": N(t) = P U D_n(t); "Unlimited OCR", GeekNews:
// the two-segment window of size m + n).  Key tiles of 128 rows are visited
// only if the mask admits at least one (row, key) pair of the tile: the
// prefix tiles 0 .. ceil(m/128)-1 up to the diagonal, plus the band tiles
// that hold the last n keys of the tile's output rows.  Per-element masking
// runs only on tiles the mask covers partially.
//
// Warp roles (256 threads):
//   warp 0      TMA producer: Q once, then K and V tiles into a 2-stage ring
//   warp 1      TMEM allocator and MMA issuer (one thread):
//                 S_j = Q K_j^T   -> TMEM (two S buffers, ping-pong)
//                 O  += P_j V_j   -> TMEM
//   warps 4..7  softmax: thread r owns query row r (= TMEM lane r); reads
//               S_j from TMEM, masks, exponentiates, writes P_j (bf16) to
//               shared memory, rescales O in TMEM when its running maximum
//               grows by more than 2^8, and finally normalises O.
// Every wait is bounded; on a timeout the CTA drains its own copies and MMAs,
// frees TMEM, sets the cache's device error flag and exits.
#include <cuda.h>

#include "rswa_device.cuh"
#include "tc_ptx.cuh"

namespace rswa {
namespace {

using namespace ptx;

constexpr int BM = 128;                       // query rows per CTA
constexpr int BN = 128;                       // keys per tile
constexpr int HD = 128;                       // head_dim
constexpr int kThreads = 256;
constexpr uint32_t kSub = BM * 64 * 2;        // [128][64] bf16, 128B-swizzled
constexpr uint32_t kTileB = 2 * kSub;         // [128][128] bf16
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + kTileB;    // 2 stages
constexpr uint32_t OFF_V = OFF_K + 2 * kTileB;// 2 stages
constexpr uint32_t OFF_P = OFF_V + 2 * kTileB;
constexpr uint32_t OFF_BAR = OFF_P + kTileB;
constexpr uint32_t kSmemBytes = OFF_BAR + 256 + 1024;  // + 1 KB alignment slack

constexpr uint32_t TM_O = 0, TM_S0 = 128, TM_S1 = 256, TM_COLS = 512;
constexpr float kRescaleThreshold = 8.0f;     // log2 units
constexpr uint64_t kWaitLimitNs = 1000000000ull;

enum Bar { B_Q, B_KF0, B_KF1, B_VF0, B_VF1, B_E0, B_E1, B_S0, B_S1, B_P, B_O, B_FIN, NBAR };

struct TileRange {
  int np;        // prefix tiles 0 .. np-1
  int kb_start;  // first band tile
  int nt;        // tiles visited
};

__device__ __forceinline__ TileRange tile_range(int qt, int m, int n, int L) {
  TileRange r;
  const int q0 = qt * BM;
  const int i_hi = min(q0 + BM - 1, L - 1);
  r.np = min((m + BN - 1) / BN, qt + 1);
  const int i_lo = max(q0, m);
  int nb = 0;
  r.kb_start = r.np;
  if (i_lo <= i_hi) {
    const int band_lo = max(m, i_lo - n + 1);
    r.kb_start = max(band_lo / BN, r.np);
    nb = max(0, i_hi / BN - r.kb_start + 1);
  }
  r.nt = r.np + nb;
  return r;
}

__device__ __forceinline__ int tile_at(const TileRange& r, int j) {
  return j < r.np ? j : r.kb_start + (j - r.np);
}

// 32 TMEM columns of this warp's 32 lanes, completed before returning.
__device__ __forceinline__ void tmem_ld32_sync(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]),
        "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32_sync(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
      "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
      "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]),
      "r"(r[31])
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, CacheView cv,
                  SeqTable st, __nv_bfloat16* __restrict__ O, int total_tiles) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar0 = sb + OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 8 * NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_BAR + 8 * NBAR + 4);
  volatile int* never = reinterpret_cast<volatile int*>(smem + OFF_BAR + 8 * NBAR + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = cv.H;
  const int h = blockIdx.x % H;
  const int g = total_tiles - 1 - (int)(blockIdx.x / H);  // heavy tiles first
  int sl = 0;
  while (sl + 1 < st.nseq && st.tile_off[sl + 1] <= g) ++sl;
  const int qt = g - st.tile_off[sl];
  const int m = st.m[sl];
  const int n = (int)min(cv.n, (int64_t)1 << 30);
  const int L = m + (int)st.T;
  const int64_t row0 = st.row_off[sl];
  const TileRange tr = tile_range(qt, m, n, L);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) mbar_init(bar(i), i == B_P ? 128u : 1u);
    *abort_flag = 0;
    *never = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const int x0 = h * HD;
      const int yq = (int)(row0 + (int64_t)qt * BM);
      mbar_arrive_expect_tx(bar(B_Q), kTileB);
      tma_load_2d(sb + OFF_Q, &tmQ, x0, yq, bar(B_Q));
      tma_load_2d(sb + OFF_Q + kSub, &tmQ, x0 + 64, yq, bar(B_Q));
      int issued = 0;
      for (int j = 0; j < tr.nt; ++j) {
        const int s = j & 1;
        if (j >= 2 && !mbar_wait(bar(B_E0 + s), ((j >> 1) - 1) & 1, abort_flag,
                                 kWaitLimitNs))
          break;
        const int y = (int)(row0 + (int64_t)tile_at(tr, j) * BN);
        mbar_arrive_expect_tx(bar(B_KF0 + s), kTileB);
        tma_load_2d(sb + OFF_K + s * kTileB, &tmK, x0, y, bar(B_KF0 + s));
        tma_load_2d(sb + OFF_K + s * kTileB + kSub, &tmK, x0 + 64, y, bar(B_KF0 + s));
        mbar_arrive_expect_tx(bar(B_VF0 + s), kTileB);
        tma_load_2d(sb + OFF_V + s * kTileB, &tmV, x0, y, bar(B_VF0 + s));
        tma_load_2d(sb + OFF_V + s * kTileB + kSub, &tmV, x0 + 64, y, bar(B_VF0 + s));
        ++issued;
      }
      // Drain: every copy issued has landed before the CTA may exit.
      mbar_wait(bar(B_Q), 0, never, kWaitLimitNs);
      for (int j = max(0, issued - 2); j < issued; ++j) {
        mbar_wait(bar(B_KF0 + (j & 1)), (j >> 1) & 1, never, kWaitLimitNs);
        mbar_wait(bar(B_VF0 + (j & 1)), (j >> 1) & 1, never, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(BM, BN, false);
      constexpr uint32_t idesc_pv = idesc_bf16(BM, HD, true);
      auto issue_qk = [&](int j) -> bool {
        const int s = j & 1;
        if (!mbar_wait(bar(B_KF0 + s), (j >> 1) & 1, abort_flag, kWaitLimitNs))
          return false;
        tc_fence_after();
        const uint32_t d = tmem + (s ? TM_S1 : TM_S0);
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t off = (k >> 2) * kSub + (k & 3) * 32;
          mma_bf16_ss(d, desc_sw128(sb + OFF_Q + off, 16, 1024),
                      desc_sw128(sb + OFF_K + s * kTileB + off, 16, 1024), idesc_qk,
                      k > 0);
        }
        mma_commit(bar(B_S0 + s));
        return true;
      };
      bool ok = mbar_wait(bar(B_Q), 0, abort_flag, kWaitLimitNs);
      if (ok) tc_fence_after();
      if (ok && tr.nt > 0) ok = issue_qk(0);
      for (int j = 0; ok && j < tr.nt; ++j) {
        if (j + 1 < tr.nt && !issue_qk(j + 1)) break;
        const int s = j & 1;
        if (!mbar_wait(bar(B_P), j & 1, abort_flag, kWaitLimitNs)) break;
        if (!mbar_wait(bar(B_VF0 + s), (j >> 1) & 1, abort_flag, kWaitLimitNs)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint32_t aoff = (k >> 2) * kSub + (k & 3) * 32;
          mma_bf16_ss(tmem + TM_O, desc_sw128(sb + OFF_P + aoff, 16, 1024),
                      desc_sw128(sb + OFF_V + s * kTileB + k * 2048, kSub, 1024),
                      idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(bar(B_O));
        mma_commit(bar(B_E0 + s));
      }
      // Drain: all MMAs of this CTA have finished before TMEM is freed.
      mma_commit(bar(B_FIN));
      mbar_wait(bar(B_FIN), 0, never, kWaitLimitNs);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x - 128;                     // row in tile
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int i = qt * BM + r;                           // row in sequence
    const float sl2 = rsqrtf((float)HD) * kLog2e;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < tr.nt; ++j) {
      const int s = j & 1;
      const int k0 = tile_at(tr, j) * BN;
      const int q0 = qt * BM;
      // Tile fully visible: every key <= every row, and every key either in
      // the prefix or inside every row's window.
      const bool full = (k0 + BN - 1 <= q0) &&
                        ((k0 + BN - 1 < m) || (max(k0, m) > q0 + BM - 1 - n));
      if (!mbar_wait(bar(B_S0 + s), (j >> 1) & 1, abort_flag, kWaitLimitNs)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // Pass 1: row maximum of the visible logits (raw q.k; the positive
      // scale is applied afterwards).
      const uint32_t sa = tmem + lane_off + (s ? TM_S1 : TM_S0);
      const int hi = i - k0;          // visible: c <= hi && (c < a || c > b)
      const int a = m - k0;
      const int b = i - n - k0;
      float tmax = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32_sync(sa + c * 32, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int col = c * 32 + e;
          const bool vis = full || (col <= hi && (col < a || col > b));
          tmax = fmaxf(tmax, vis ? __uint_as_float(v[e]) : -INFINITY);
        }
      }
      tmax *= sl2;
      // Lazy rescale: keep the reference maximum unless it grew by > 2^8.
      // Exact either way: O and l share the reference.
      float alpha = 1.f;
      bool resc = false;
      const float m_new = fmaxf(m_run, tmax);
      if (m_run == -INFINITY) {
        m_run = m_new;
      } else if (m_new > m_run + kRescaleThreshold) {
        alpha = ex2(m_run - m_new);
        m_run = m_new;
        l_run *= alpha;
        resc = true;
      }
      const float ref = (m_run == -INFINITY) ? 0.f : m_run;
      // PV of the previous tile must be done: P buffer free, O stable.
      if (j > 0 && !mbar_wait(bar(B_O), (j - 1) & 1, abort_flag, kWaitLimitNs)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t o[32];
          const uint32_t oa = tmem + lane_off + TM_O + c * 32;
          tmem_ld32_sync(oa, o);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32_sync(oa, o);
        }
      }
      // Pass 2: P = exp2(x - ref) -> bf16 -> shared memory, 128B-swizzled
      // K-major as the MMA reads it, in 16-byte chunks of 8 keys.
      uint8_t* prow = smem + OFF_P + (r >> 3) * 1024 + (r & 7) * 128;
      float psum = 0.f;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32_sync(sa + c * 32, v);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c0 = c * 32 + 2 * e;
          const bool v0 = full || (c0 <= hi && (c0 < a || c0 > b));
          const bool v1 = full || (c0 + 1 <= hi && (c0 + 1 < a || c0 + 1 > b));
          const float p0 = v0 ? ex2(fmaf(__uint_as_float(v[2 * e]), sl2, -ref)) : 0.f;
          const float p1 = v1 ? ex2(fmaf(__uint_as_float(v[2 * e + 1]), sl2, -ref)) : 0.f;
          psum += p0 + p1;
          w[e] = pack_bf16(p0, p1);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c16 = c * 4 + q;
          uint8_t* dst = prow + (c16 >> 3) * kSub + (((c16 & 7) ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(dst) =
              make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
      l_run += psum;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_P));
    }
    // Epilogue: O / l -> bf16 -> global.
    if (ok && tr.nt > 0 &&
        mbar_wait(bar(B_O), (tr.nt - 1) & 1, abort_flag, kWaitLimitNs)) {
      tc_fence_after();
      const float inv = 1.f / l_run;
      __nv_bfloat16* orow = O + ((row0 + i) * H + h) * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t o[32];
        tmem_ld32_sync(tmem + lane_off + TM_O + c * 32, o);
        if (i < L) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv,
                             __uint_as_float(o[2 * e + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
  if (threadIdx.x == 0 && *abort_flag) flag_error(cv.err, kErrWaitTimeout);
}

// ---- host: tensor maps through the driver entry point ----------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                  void*, const cuuint64_t*, const cuuint64_t*,
                                  const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// [rows][H*128] bf16 viewed as a 2-D tensor; box 64 columns x 128 rows,
// 128-byte swizzle; rows past `rows` read as zero.
bool make_map(CUtensorMap* map, const void* base, int H, int64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)H * HD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)H * HD * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_tc_supported(const CacheView& cv) {
  return cv.dtype == RSWA_BF16 && cv.d == HD && encode_fn() != nullptr;
}

cudaError_t launch_prefill_tc(const CacheView& cv, const SeqTable& st,
                              const void* Q, const void* K, const void* V,
                              void* O, int64_t total_rows, cudaStream_t s) {
  if (!prefill_tc_supported(cv)) return cudaErrorNotSupported;
  const int64_t end_row = st.row_off[0] + total_rows;
  if (end_row >= (int64_t(1) << 31)) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, Q, cv.H, end_row) || !make_map(&mk, K, cv.H, end_row) ||
      !make_map(&mv, V, cv.H, end_row))
    return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(
        prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int tiles = st.tile_off[st.nseq];
  if (tiles == 0) return cudaSuccess;
  const int64_t grid = (int64_t)tiles * cv.H;
  if (grid >= (int64_t(1) << 31)) return cudaErrorNotSupported;
  prefill_tc_kernel<<<(unsigned)grid, kThreads, kSmemBytes, s>>>(
      mq, mk, mv, cv, st, static_cast<__nv_bfloat16*>(O), tiles);
  return cudaGetLastError();
}

}  // namespace rswa
