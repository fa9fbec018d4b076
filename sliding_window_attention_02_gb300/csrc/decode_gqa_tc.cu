// Grouped-query R-SWA decode on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA).
//
// The G query heads that read one KV head attend the same keys, so one
// decode step for them is a small dense contraction: S = Q_G K^T over the
// visible keys of the KV head ("Unlimited-OCR deep dive": N(t) = P U D_n(t))
// and O_G = softmax(S) V.  With G <= 16 this kernel computes it transposed,
//   S^T  = K Q_G^T    M = 128 keys of a tile, N = 16 (heads, padded), K = d
//   O^T += V^T P^T    M = d = 128, N = 16, K = 128 keys of a tile
// with both accumulators in TMEM, K and V tiles streaming through a TMA ring,
// and the CUDA cores left with the softmax: one key per thread, G scores.
//
// Grid (B * H_kv, max_chunks): one CTA is one split-K chunk (prefix chunk or
// ring chunk, as in decode_kernel) of one KV head and serves every query
// head of that KV head, so the CTA that stores a fused step's new key and
// value in its ring slot is also the only reader of that slot: it writes the
// row, orders the write before the TMA reads (proxy fence), then loads.
// Roles (192 threads):
//   warps 0-3  softmax: thread t owns key t of a tile (TMEM lane t); then the
//              epilogue: thread t owns row d = t of O^T
//   warp 4     TMA producer: K_0, V_0, K_1, V_1, ... into a ring of slots
//   warp 5     TMEM allocator and MMA issuer (one thread)
// TMEM (64 columns): S^T double buffer at columns 0 and 16, O^T at 32.
// The MMA order S(0) S(1) PV(0) S(2) PV(1) ... lets the softmax of tile j run
// while PV(j-1) executes.  O^T is rescaled lazily: only when a head's running
// maximum exceeds the reference the probabilities use by more than 2^8 (the
// reference, not the true maximum, is what the partial reports).
// Rows of a tile past the chunk's end are masked (score -inf, p = 0); the
// cache's K/V regions are zeroed at creation, so such rows hold finite
// values and contribute exactly 0.
// Every wait is bounded (wait_ns, phase_wait_limit_ns(), for the pipeline's
// phases; kWaitLimitNs for the drains); on a timeout the CTA drains its
// copies and MMAs, frees TMEM, sets the cache's device error flag and exits.
#include <cuda.h>

#include "rswa_device.cuh"
#include "rswa_internal.h"
#include "tc_ptx.cuh"

namespace rswa {
namespace {

using namespace ptx;

constexpr int HD = 128;                     // head_dim
constexpr int BN = 128;                     // keys per tile
constexpr int NQ = 16;                      // MMA N: query heads, padded
constexpr int kSoftThreads = 128;
constexpr int kThreads = kSoftThreads + 64;
constexpr int kProducerWarp = 4, kMmaWarp = 5;
#ifndef RSWA_TC_STAGES
#define RSWA_TC_STAGES 3
#endif
constexpr int NS = RSWA_TC_STAGES;          // ring slots (a K or a V tile)
static_assert(NS >= 2, "a chunk's first K and V tiles take slots 0 and 1");
constexpr uint32_t kSub = BN * 64 * 2;      // [128][64] bf16, 128B-swizzled
constexpr uint32_t kTileB = 2 * kSub;       // [128][128] bf16 = 32 KB
constexpr uint32_t kNAtom = NQ * 128;       // [16][64] bf16 atom = 2 KB
constexpr uint32_t OFF_Q = 0;               // Q^T operand: 2 atoms
constexpr uint32_t OFF_P = OFF_Q + 2 * kNAtom;   // P^T double buffer
constexpr uint32_t OFF_RING = OFF_P + 4 * kNAtom;
constexpr uint32_t OFF_BAR = OFF_RING + NS * kTileB;
constexpr int B_FULL = 0;                   // NS
constexpr int B_EMPTY = B_FULL + NS;        // NS
constexpr int B_S = B_EMPTY + NS;           // 2: S^T(j) in TMEM
constexpr int B_SFREE = B_S + 2;            // 2: S^T(j) read (128 arrivals)
constexpr int B_P = B_SFREE + 2;            // 2: P^T(j) in smem (128 arrivals)
constexpr int B_PFREE = B_P + 2;            // 2: PV(j) done
constexpr int B_O = B_PFREE + 2;            // all MMAs done
constexpr int B_SYNC = B_O + 1;             // softmax warps' barrier (128)
constexpr int NBAR = B_SYNC + 1;
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * NBAR;    // tmem slot, flags
constexpr uint32_t OFF_RED = OFF_MISC + 16;          // [2][4][16] + [4][16]
constexpr uint32_t kSmemBytes = OFF_RED + (2 * 4 * NQ + 4 * NQ) * 4 + 1024;
static_assert(OFF_RING % 1024 == 0, "swizzled tiles need 1 KB alignment");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
constexpr uint32_t TM_S = 0, TM_O = 32, TM_COLS = 64;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// PREFETCH: the preceding kernel of the stream writes no prefix row, so a
// prefix slot's first K and V tiles may be requested before the dependency
// wait.
// tmK8 / tmV8: the same slabs with 8-row boxes, for the rows of a chunk's
// last tile (whole 8-row groups; the tile's other rows are not fetched).
// A key or value tile is read once per launch: its TMA loads carry an
// evict-first L2 policy, so the streamed tiles do not displace the partials,
// q and the state.
__device__ __forceinline__ uint64_t stream_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int32_t x,
                                                 int32_t y, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
      : "memory");
}

template <bool FUSED, int G, bool PREFETCH>
__global__ void __launch_bounds__(kThreads, 2)
decode_gqa_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmK8,
                     const __grid_constant__ CUtensorMap tmV8, CacheView cv,
                     const __nv_bfloat16* __restrict__ q,
                     const __nv_bfloat16* __restrict__ knew,
                     const __nv_bfloat16* __restrict__ vnew,
                     __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                     uint64_t wait_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int k) { return sb + OFF_BAR + 8u * (uint32_t)k; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  volatile int* never = reinterpret_cast<volatile int*>(smem + OFF_MISC + 8);
  int* s_last = reinterpret_cast<int*>(smem + OFF_MISC + 12);
  float* red_max = reinterpret_cast<float*>(smem + OFF_RED);     // [2][4][NQ]
  float* red_sum = red_max + 2 * 4 * NQ;                          // [4][NQ]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int b = blockIdx.x / cv.Hkv, kv = blockIdx.x % cv.Hkv;
  const int per_kv = cv.H / cv.Hkv;                 // query heads served (<= G)

  if (tid == 0) {
    for (int k = 0; k < NBAR; ++k)
      mbar_init(bar(k), ((k >= B_SFREE && k < B_PFREE) || k == B_SYNC) ? 128u : 1u);
    *abort_flag = 0;
    *never = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
  }
  // Zero the ring slots: a chunk's last tile fetches only its rows (in
  // 8-row groups), and the rows it leaves keep what the slot held before -
  // zeros, or rows of an earlier tile - finite values that the masked
  // probabilities (p = 0) multiply exactly to 0.
  for (uint32_t i = tid; i < NS * kTileB / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + OFF_RING)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  __syncthreads();                                  // barriers initialised
  // A prefix slot's first K and V tiles start at slab row y * chunk whatever
  // m_b is: request them (ring slots 0 and 1, loads 0 and 1 of the chunk)
  // before the state loads.  A slot past this sequence's prefix drains them
  // unused.
  const int chunk = cv.chunk;
  const int cp_cap = (int)((cv.m_cap + chunk - 1) / chunk);
  const int y = blockIdx.y;
  const size_t bkv = (size_t)b * cv.Hkv + kv;
  const bool spec = y < cp_cap;
  const uint64_t kpol = stream_policy();
  auto spec_loads = [&]() {
    if (warp == kProducerWarp && lane == 0 && spec) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const int yr = (int)((int64_t)bkv * cv.slab_rows + (int64_t)y * chunk);
      mbar_arrive_expect_tx(bar(B_FULL + 0), kTileB);
      tma_load_2d_hint(sb + OFF_RING, &tmK, 0, yr, bar(B_FULL + 0), kpol);
      tma_load_2d_hint(sb + OFF_RING + kSub, &tmK, 64, yr, bar(B_FULL + 0), kpol);
      mbar_arrive_expect_tx(bar(B_FULL + 1), kTileB);
      tma_load_2d_hint(sb + OFF_RING + kTileB, &tmV, 0, yr, bar(B_FULL + 1), kpol);
      tma_load_2d_hint(sb + OFF_RING + kTileB + kSub, &tmV, 64, yr, bar(B_FULL + 1), kpol);
    }
  };
  if (PREFETCH) spec_loads();
  griddep_wait();
  // The next step's CTAs may take SM slots as this grid's CTAs finish (and
  // do their set-up and early tile requests there); they wait for this grid.
  griddep_launch_dependents();
  if (!PREFETCH) spec_loads();

  // The query rows of the KV head's heads (column tid), loaded alongside the
  // state words: their address does not depend on them.
  __nv_bfloat16 qv[G];
  if (tid < kSoftThreads) {
    const size_t bq = (size_t)b * cv.H + (size_t)kv * per_kv;
#pragma unroll
    for (int g = 0; g < G; ++g)
      qv[g] = g < per_kv ? q[(bq + g) * HD + tid] : __float2bfloat16(0.f);
  }

  // This chunk: slab rows [j0, j1) of KV head (b, kv).
  const int64_t m_b = cv.m_dev[b];
  const int cp = (int)((m_b + chunk - 1) / chunk);
  const int nch = cp + (int)((cv.n + chunk - 1) / chunk);
  // Grid slot y: prefix chunk y while y < ceil(m_cap / chunk) (no work past
  // this sequence's prefix), then ring chunk y - ceil(m_cap / chunk).  Slots
  // launch in order, so every sequence's prefix chunks run before the
  // one-tile ring chunks, which fill the last wave.  c is the chunk's index
  // among this sequence's nch partials.
  const bool live = y >= cp_cap || y < cp;
  const int c = y < cp_cap ? y : cp + (y - cp_cap);
  const size_t bh0 = (size_t)b * cv.H + (size_t)kv * per_kv;
  const int64_t t_b = cv.t_dev[bh0];                // equal for the heads
  int64_t j0 = 0, j1 = 0, sub = -1;
  if (live) {
    if (c < cp) {
      j0 = (int64_t)c * chunk;
      j1 = min(j0 + chunk, m_b);
    } else {
      const int64_t s0 = (int64_t)(c - cp) * chunk;
      const int64_t filled = FUSED ? min(cv.n, t_b + 1) : min(cv.n, t_b);
      j0 = cv.m_cap + s0;
      j1 = cv.m_cap + max(s0, min(s0 + chunk, filled));
      if (FUSED) {
        const int64_t w = t_b % cv.n;
        if (w >= s0 && w < s0 + chunk) sub = cv.m_cap + w;
      }
    }
  }
  const int nt = (int)((j1 - j0 + BN - 1) / BN);   // tiles of this chunk
  const int64_t rbase = (int64_t)bkv * cv.slab_rows + j0;
  // Rows of the last tile, rounded up to whole 8-row groups.
  const int last8 = nt > 0 ? (int)((j1 - j0 - (int64_t)(nt - 1) * BN + 7) & ~7) : BN;
  // K_i (even idx) or V_i (odd idx) into ring slot idx % NS; the last tile
  // as 8-row boxes, each landing at its rows' place in the swizzled tile
  // (1 KB-aligned, so the 128-byte swizzle pattern is the full tile's).
  auto load = [&](int idx) {
    const int s = idx % NS;
    const bool isv = idx & 1;
    const int y = (int)(rbase + (int64_t)(idx >> 1) * BN);
    const uint32_t dst = sb + OFF_RING + s * kTileB;
    const int rows = (idx >> 1) == nt - 1 ? last8 : BN;
    if (rows == BN) {
      const CUtensorMap* map = isv ? &tmV : &tmK;
      mbar_arrive_expect_tx(bar(B_FULL + s), kTileB);
      tma_load_2d_hint(dst, map, 0, y, bar(B_FULL + s), kpol);
      tma_load_2d_hint(dst + kSub, map, 64, y, bar(B_FULL + s), kpol);
    } else {
      const CUtensorMap* map = isv ? &tmV8 : &tmK8;
      mbar_arrive_expect_tx(bar(B_FULL + s), (uint32_t)rows * 256u);
      for (int r = 0; r < rows; r += 8) {
        tma_load_2d_hint(dst + r * 128, map, 0, y + r, bar(B_FULL + s), kpol);
        tma_load_2d_hint(dst + kSub + r * 128, map, 64, y + r, bar(B_FULL + s), kpol);
      }
    }
  };
  const int first_loads = min(NS, 2 * nt);

  if (warp == kProducerWarp) {
    // The new key and value of a fused step, stored before any TMA read,
    // then the first ring loads, while the other warps stage Q.
    if (FUSED && sub >= 0) {
      constexpr int NV = HD * 2 / 16;               // 16-byte pieces per row
      const bool isk = lane < NV;
      const int i = isk ? lane : lane - NV;
      uint4* dst = reinterpret_cast<uint4*>(
          static_cast<__nv_bfloat16*>(isk ? cv.K : cv.V) +
          (bkv * cv.slab_rows + sub) * HD);
      const uint4* src = reinterpret_cast<const uint4*>((isk ? knew : vnew) + bkv * HD);
      dst[i] = src[i];
      fence_proxy_async_global();
    }
    __syncwarp();
    if (lane == 0 && live) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      // A live prefix chunk starts at slab row y * chunk: its loads 0 and 1
      // are the ones requested above.
      for (int idx = spec ? 2 : 0; idx < first_loads; ++idx) load(idx);
    }
  } else if (tid < kSoftThreads) {
    // Q_G^T as the MMA's B operand: row g = query head g, K-major over d.
#pragma unroll
    for (int g = 0; g < NQ; ++g) {
      const __nv_bfloat16 v = (live && g < G) ? qv[g < G ? g : 0] : __float2bfloat16(0.f);
      *reinterpret_cast<__nv_bfloat16*>(smem + OFF_Q + sw128_off(g, tid, kNAtom)) = v;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const float scale = rsqrtf((float)HD) * kLog2e;

  float m_ref[G], l_t[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m_ref[g] = -INFINITY;
    l_t[g] = 0.f;
  }

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && live) {
      int issued = first_loads;
      for (int idx = first_loads; idx < 2 * nt; ++idx) {
        if (!mbar_wait(bar(B_EMPTY + idx % NS), ((idx / NS) - 1) & 1, abort_flag,
                       wait_ns))
          break;
        load(idx);
        ++issued;
      }
      // Drain: every copy issued has landed before the CTA may exit.
      for (int idx = max(0, issued - NS); idx < issued; ++idx)
        mbar_wait(bar(B_FULL + idx % NS), (idx / NS) & 1, never, kWaitLimitNs);
    } else if (lane == 0 && spec) {
      // A prefix slot past this sequence's prefix: its two early loads.
      mbar_wait(bar(B_FULL + 0), 0, never, kWaitLimitNs);
      mbar_wait(bar(B_FULL + 1), 0, never, kWaitLimitNs);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_ab(BN, NQ, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_ab(HD, NQ, true, false);
      auto full = [&](int idx) {
        return mbar_wait(bar(B_FULL + idx % NS), (idx / NS) & 1, abort_flag,
                         wait_ns);
      };
      // S^T(j) = K_j Q^T: A = K tile (K-major over d), B = Q^T.
      auto issue_s = [&](int j) {
        const uint32_t kb = sb + OFF_RING + ((2 * j) % NS) * kTileB;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k)
          mma_bf16_ss(tmem + TM_S + 16 * (j & 1),
                      desc_sw128(kb + (k >> 2) * kSub + (k & 3) * 32, 16, 1024),
                      desc_sw128(sb + OFF_Q + (k >> 2) * kNAtom + (k & 3) * 32, 16, 1024),
                      idesc_s, k > 0);
        mma_commit(bar(B_S + (j & 1)));
        mma_commit(bar(B_EMPTY + (2 * j) % NS));
      };
      // O^T += V_j^T P_j^T: A = V tile read MN-major (d contiguous), B = P^T.
      auto issue_pv = [&](int j) {
        const uint32_t vb = sb + OFF_RING + ((2 * j + 1) % NS) * kTileB;
        const uint32_t pb = sb + OFF_P + (j & 1) * 2 * kNAtom;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_bf16_ss(tmem + TM_O, desc_sw128(vb + k * 2048, kSub, 1024),
                      desc_sw128(pb + (k >> 2) * kNAtom + (k & 3) * 32, 16, 1024),
                      idesc_o, (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(bar(B_PFREE + (j & 1)));
        mma_commit(bar(B_EMPTY + (2 * j + 1) % NS));
      };
      auto pv_ready = [&](int j) {
        return mbar_wait(bar(B_P + (j & 1)), (j >> 1) & 1, abort_flag, wait_ns) &&
               full(2 * j + 1);
      };
      bool ok = live;
      for (int j = 0; ok && j < nt; ++j) {
        ok = full(2 * j) &&
             (j < 2 || mbar_wait(bar(B_SFREE + (j & 1)), ((j - 2) >> 1) & 1,
                                 abort_flag, wait_ns));
        if (!ok) break;
        tc_fence_after();
        issue_s(j);
        if (j >= 1) {
          ok = pv_ready(j - 1);
          if (!ok) break;
          tc_fence_after();
          issue_pv(j - 1);
        }
      }
      if (ok && nt > 0 && pv_ready(nt - 1)) {
        tc_fence_after();
        issue_pv(nt - 1);
      }
      // Arrives once every MMA issued above has completed.
      mma_commit(bar(B_O));
    }
  } else {
    // ------------------------------------------------------------ softmax
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    // Waits agreed by the whole warp (lanes stay converged for the
    // warp-collective TMEM loads and shuffles), and a barrier over the four
    // softmax warps on an mbarrier: bounded, so a warp that gives up cannot
    // leave the others blocked.
    auto wait_all = [&](int k, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar(k), parity, abort_flag, wait_ns));
    };
    int n_sync = 0;
    auto soft_sync = [&]() {
      mbar_arrive(bar(B_SYNC));
      const bool r = mbar_wait(bar(B_SYNC), n_sync & 1, abort_flag, wait_ns);
      ++n_sync;
      return __all_sync(0xffffffffu, r);
    };
    for (int j = 0; live && j < nt; ++j) {
      if (!wait_all(B_S + (j & 1), (j >> 1) & 1)) break;
      tc_fence_after();
      uint32_t r[16];
      tmem_ld16(tmem + lane_off + TM_S + 16 * (j & 1), r);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(B_SFREE + (j & 1)));
      const bool valid = j0 + (int64_t)j * BN + tid < j1;
      float s[G];
#pragma unroll
      for (int g = 0; g < G; ++g)
        s[g] = (valid && g < per_kv) ? __uint_as_float(r[g]) * scale : -INFINITY;
      // tile maximum of every head over the 128 keys
      float* rm = red_max + (j & 1) * 4 * NQ;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float v = warp_max(s[g]);
        if (lane == 0) rm[warp * NQ + g] = v;
      }
      if (!soft_sync()) break;
      bool grow = false;
      float mt[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        mt[g] = fmaxf(fmaxf(rm[g], rm[NQ + g]), fmaxf(rm[2 * NQ + g], rm[3 * NQ + g]));
        grow |= mt[g] > m_ref[g] + kRescaleThreshold ||
                (m_ref[g] == -INFINITY && mt[g] > -INFINITY);
      }
      if (grow) {
        // New references: every head's maximum so far.  O^T holds PV(0..j-1)
        // and is rescaled once PV(j-1) has completed.
        float alpha[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float mn = fmaxf(m_ref[g], mt[g]);
          alpha[g] = (mn == -INFINITY) ? 1.f : fast_exp2(m_ref[g] - mn);
          m_ref[g] = mn;
          l_t[g] *= alpha[g];
        }
        if (j >= 1) {
          if (!wait_all(B_PFREE + ((j - 1) & 1), ((j - 1) >> 1) & 1)) break;
          tc_fence_after();
          uint32_t ov[16];
          tmem_ld16(tmem + lane_off + TM_O, ov);
          tmem_wait_ld();
#pragma unroll
          for (int g = 0; g < G; ++g)
            ov[g] = __float_as_uint(__uint_as_float(ov[g]) * alpha[g]);
          tmem_st16(tmem + lane_off + TM_O, ov);
          tmem_wait_st();
        }
      }
      // P^T(j): buffer j & 1 is free once PV(j-2) has completed.
      if (j >= 2 && !wait_all(B_PFREE + (j & 1), ((j - 2) >> 1) & 1)) break;
      uint8_t* pbuf = smem + OFF_P + (j & 1) * 2 * kNAtom;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float ref = (m_ref[g] == -INFINITY) ? 0.f : m_ref[g];
        const float p = fast_exp2(s[g] - ref);
        l_t[g] += p;
        if (g < per_kv)
          *reinterpret_cast<__nv_bfloat16*>(pbuf + sw128_off(g, tid, kNAtom)) =
              __float2bfloat16(p);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(B_P + (j & 1)));
    }
  }

  // ------------------------------------------------------------ epilogue
  // Partial (m_ref, l, O^T column) of every query head of this chunk.
  bool have_o = false;
  uint32_t ov[16];
  if (tid < kSoftThreads && live && nt > 0 && !*abort_flag &&
      __all_sync(0xffffffffu, mbar_wait(bar(B_O), 0, abort_flag, wait_ns))) {
    tc_fence_after();
    tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + TM_O, ov);
    tmem_wait_ld();
    have_o = true;
  }
  if (tid < kSoftThreads) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float v = l_t[g];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) red_sum[warp * NQ + g] = v;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (live && tid < kSoftThreads) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (g >= per_kv) break;
      float* P = cv.part + ((bh0 + g) * cv.max_chunks + c) * (HD + 2);
      P[2 + tid] = have_o ? __uint_as_float(ov[g]) : 0.f;
      if (tid == 0) {
        P[0] = m_ref[g];
        P[1] = red_sum[g] + red_sum[NQ + g] + red_sum[2 * NQ + g] + red_sum[3 * NQ + g];
      }
    }
  }
  __syncthreads();
  if (tid == 0) *s_last = live && arrive_acq_rel(&cv.cnt_bh[bh0]) == nch - 1;
  __syncthreads();
  if (*s_last && tid < kSoftThreads) {
    float M[G], L[G], A[G];
    merge_partials<G, (G <= 2 ? 2 : 1)>(
        cv.part + bh0 * cv.max_chunks * (HD + 2), (size_t)cv.max_chunks * (HD + 2),
        nch, HD, tid, per_kv, M, L, A);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (g >= per_kv) break;
      o[(bh0 + g) * HD + tid] = __float2bfloat16(L[g] > 0.f ? A[g] / L[g] : 0.f);
      if (tid == 0) {
        if (lse) lse[bh0 + g] = L[g] > 0.f ? (M[g] + log2f(L[g])) * kLn2 : -INFINITY;
        // Every CTA of this KV head read t_b before its own arrival.
        if (FUSED) cv.t_dev[bh0 + g] = t_b + 1;
      }
    }
    if (tid == 0) cv.cnt_bh[bh0] = 0;
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    // Every MMA this CTA issued has completed before TMEM is released.
    if (lane == 0) mbar_wait(bar(B_O), 0, never, kWaitLimitNs);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
  if (tid == 0 && *abort_flag) flag_error(cv.err, kErrWaitTimeout);
}

template <bool FUSED, int G, bool PREFETCH>
cudaError_t launch_tc(const CacheView& cv, const CUtensorMap& mk,
                      const CUtensorMap& mv, const CUtensorMap& mk8,
                      const CUtensorMap& mv8, const void* q, const void* k,
                      const void* v, void* o, float* lse, cudaStream_t s) {
  auto kern = decode_gqa_tc_kernel<FUSED, G, PREFETCH>;
  // Per device (the attribute belongs to the current device's context).
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cv.B * cv.Hkv, cv.max_chunks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  using BF = __nv_bfloat16;
  return cudaLaunchKernelEx(&cfg, kern, mk, mv, mk8, mv8, cv, (const BF*)q,
                            (const BF*)(FUSED ? k : nullptr),
                            (const BF*)(FUSED ? v : nullptr), (BF*)o, lse,
                            phase_wait_limit_ns());
}

template <bool FUSED, bool PREFETCH>
cudaError_t launch_tc_g(const CacheView& cv, const CUtensorMap* m, const void* q,
                        const void* k, const void* v, void* o, float* lse,
                        cudaStream_t s) {
  const int per_kv = cv.H / cv.Hkv;
  if (per_kv <= 2)
    return launch_tc<FUSED, 2, PREFETCH>(cv, m[0], m[1], m[2], m[3], q, k, v, o, lse, s);
  if (per_kv <= 4)
    return launch_tc<FUSED, 4, PREFETCH>(cv, m[0], m[1], m[2], m[3], q, k, v, o, lse, s);
  if (per_kv <= 8)
    return launch_tc<FUSED, 8, PREFETCH>(cv, m[0], m[1], m[2], m[3], q, k, v, o, lse, s);
  return launch_tc<FUSED, 16, PREFETCH>(cv, m[0], m[1], m[2], m[3], q, k, v, o, lse, s);
}

}  // namespace

bool gqa_tc_supported(const CacheView& cv) {
  if (!gqa_tc_shape(cv.H, cv.Hkv, cv.d, cv.dtype)) return false;
  if ((int64_t)cv.B * cv.Hkv * cv.slab_rows + BN >= (int64_t(1) << 31)) return false;
  CUtensorMap probe;
  return make_tmap_rows_bf16(&probe, cv.K, HD, 128);
}

cudaError_t launch_decode_gqa_tc(const CacheView& cv, const void* q,
                                 const void* k, const void* v, void* o,
                                 float* lse, bool fused, bool prefetch_prefix,
                                 cudaStream_t s) {
  const uint64_t rows = (uint64_t)cv.B * cv.Hkv * cv.slab_rows;
  CUtensorMap m[4];                                 // K, V; K, V in 8-row boxes
  if (!make_tmap_rows_bf16(&m[0], cv.K, HD, rows) ||
      !make_tmap_rows_bf16(&m[1], cv.V, HD, rows) ||
      !make_tmap_rows_bf16(&m[2], cv.K, HD, rows, 8) ||
      !make_tmap_rows_bf16(&m[3], cv.V, HD, rows, 8))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if (prefetch_prefix)
    e = fused ? launch_tc_g<true, true>(cv, m, q, k, v, o, lse, s)
              : launch_tc_g<false, true>(cv, m, q, k, v, o, lse, s);
  else
    e = fused ? launch_tc_g<true, false>(cv, m, q, k, v, o, lse, s)
              : launch_tc_g<false, false>(cv, m, q, k, v, o, lse, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace rswa
