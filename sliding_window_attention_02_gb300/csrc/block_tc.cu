// R-SWA attention for a block of C consecutive output tokens appended to an
// existing cache, on the 5th-generation tensor cores (tcgen05 + TMEM + TMA):
// chunked prefill of output text longer than the window, and the
// verification forward of drafted tokens.
//
// Output t_b + i of sequence b (i = 0..C-1) attends to
//   the prefix          keys 0..m_b-1            (cache slab rows 0..m_b-1)
//   cached outputs      j in [t_b + i - n + 1, t_b) (ring slot j mod n)
//   the block's tokens  i' in (i - n, i]          (rows of the block's K, V)
// which is N(t) = P U D_n(t) of the "Unlimited-OCR deep dive" (R-SWA
// pseudo-code block) for t = t_b + i.  Slot s of the ring holds output
// t_b - 1 - a_s, a_s = (t_b - 1 - s) mod n steps old; it is a key of row i
// iff a_s <= min(t_b - 1, n - 2 - i).
//
// A work unit is two adjacent 128-row query tiles ("halves") of the block of
// one (b, h); one CTA per unit.  Its key tiles come from three sources: the
// prefix tiles of the cache slab, the ring tiles (only while some row of the
// unit still sees a cached output), and the block tiles of the band
// (i - n, i].  The pipeline is the prefill kernel's (prefill_tc.cu): roles
// (320 threads) warps 0-3 / 4-7 softmax of half 0 / 1 (thread r owns row r =
// TMEM lane r), warp 8 TMA producer (Q0, Q1, then K_j, V_j into a 4-slot
// ring), warp 9 TMEM allocator and MMA issuer; TMEM S0 | S1 | O0 | O1; the
// issue order QK0(0) QK1(0) | PV0(j) QK0(j+1) PV1(j) QK1(j+1) | ... keeps
// the tensor core on one half while the other half's softmax runs; P_h
// overwrites S_h in TMEM and feeds the PV MMA from there; O is rescaled
// lazily.  Every wait is bounded; on a timeout the CTA drains its copies and
// MMAs, frees TMEM, sets the cache's device error flag and exits.
//
// When pairs of tiles would not fill the SMs once, a unit is one query tile
// instead, split: both halves take its rows, half 0 the even and half 1 the
// odd key tiles, so the two halves still alternate on the tensor core and
// each CTA's chain of tiles is half as long; at the end half 1 hands its
// (m, l, O) to half 0 through shared memory and half 0 writes the merged
// rows.  So is the last unit of a pair grid whose second tile holds no row.
// Single-page cache, per call with the append kernel: blocks of 64 / 256 /
// 1024 tokens 20.7 / 26.1 / 26.9 us as pairs, 16.3 / 16.8 / 17.8 split.
//
// The cache is only read here; the append of the block's last min(n, C)
// tokens runs afterwards (decode_block.cu), once this kernel has finished
// with the ring slots it overwrites.
#include <cuda.h>

#include <algorithm>

#include "rswa_device.cuh"
#include "tc_ptx.cuh"

namespace rswa {
namespace {

using namespace ptx;

constexpr int BM = 128;                        // rows per half
constexpr int BN = 128;                        // keys per tile
constexpr int HD = 128;                        // head_dim
constexpr int kSoftmaxThreads = 256;
constexpr int kThreads = kSoftmaxThreads + 64;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int NS = 4;                          // K/V ring slots
constexpr uint32_t kSub = BM * 64 * 2;         // [128][64] bf16, 128B-swizzled
constexpr uint32_t kTileB = 2 * kSub;          // [128][128] bf16 = 32 KB
constexpr uint32_t OFF_Q = 0;                  // Q0, Q1
constexpr uint32_t OFF_RING = 2 * kTileB;
constexpr uint32_t OFF_BAR = OFF_RING + NS * kTileB;
constexpr uint32_t kSmemBytes = OFF_BAR + 256 + 1024;  // + 1 KB alignment slack

__host__ __device__ constexpr uint32_t tm_s(int half) { return half ? 128u : 0u; }
__host__ __device__ constexpr uint32_t tm_o(int half) { return half ? 384u : 256u; }
constexpr uint32_t TM_COLS = 512;
constexpr float kRescaleThreshold = 8.0f;      // log2 units
constexpr uint64_t kWaitLimitNs = 1000000000ull;

constexpr int B_Q = 0;
constexpr int B_FULL = 1;                      // NS slots
constexpr int B_EMPTY = B_FULL + NS;           // NS slots
constexpr int B_S = B_EMPTY + NS;              // 2 halves
constexpr int B_P = B_S + 2;                   // 2 halves
constexpr int B_O = B_P + 2;                   // 2 halves
constexpr int B_FIN = B_O + 2;
constexpr int B_MERGE = B_FIN + 1;             // split unit: half 1's (m, l, O) in smem
constexpr int NBAR = B_MERGE + 1;

enum TileKind { kPrefix = 0, kRing = 1, kBlock = 2 };

// The key tiles of one unit: prefix tiles 0..np-1 of the slab, ring tiles
// 0..nr-1 (slots 128 r ..), block tiles kb0..kb0+nb-1 (block rows 128 k ..).
struct Tiles {
  int np, nr, kb0, nb;
  __device__ int count() const { return np + nr + nb; }
  __device__ void at(int j, int& kind, int& idx) const {
    if (j < np) {
      kind = kPrefix;
      idx = j;
    } else if (j < np + nr) {
      kind = kRing;
      idx = j - np;
    } else {
      kind = kBlock;
      idx = kb0 + (j - np - nr);
    }
  }
};

// Unit u: head u % H, then (sequence, tile or tile pair) of the block.
// split: the unit's second half holds no row of the block.
struct Unit {
  int b, h, kvh, q0;
  bool split;
  int64_t m_b, t_b;
  Tiles tl;
};

// rows: 2 BM (a pair of query tiles per unit) or BM (one tile per unit, split
// into the two halves).
__device__ __forceinline__ Unit unit_at(int u, const CacheView& cv, int C, int rows) {
  Unit w;
  const int per_head = (C + rows - 1) / rows;
  w.h = u % cv.H;
  const int rest = u / cv.H;
  w.b = rest / per_head;
  w.q0 = (rest % per_head) * rows;
  w.split = rows == BM || w.q0 + BM >= C;       // no second tile in this unit
  w.kvh = w.h / (cv.H / cv.Hkv);
  w.m_b = cv.m_dev[w.b];
  w.t_b = cv.t_dev[(size_t)w.b * cv.H + w.h];
  const int64_t n = cv.n;
  w.tl.np = (int)((w.m_b + BN - 1) / BN);
  // Rows i <= n - 2 see cached outputs (while t_b >= 1): all filled slots.
  const int64_t filled = min(n, w.t_b);
  w.tl.nr = (w.q0 <= n - 2 && filled > 0) ? (int)((filled + BN - 1) / BN) : 0;
  const int q_hi = min(w.q0 + rows - 1, C - 1);
  const int64_t lo = max((int64_t)0, (int64_t)w.q0 - n + 1);
  w.tl.kb0 = (int)(lo / BN);
  w.tl.nb = q_hi / BN - w.tl.kb0 + 1;
  return w;
}

// wait_ns bounds every wait for a pipeline phase (phase_wait_limit_ns());
// the drains before exit keep kWaitLimitNs.
__global__ void __launch_bounds__(kThreads, 1)
block_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                const __grid_constant__ CUtensorMap tmKc,
                const __grid_constant__ CUtensorMap tmVc,
                const __grid_constant__ CUtensorMap tmKb,
                const __grid_constant__ CUtensorMap tmVb, CacheView cv, int C,
                int unit_rows, __nv_bfloat16* __restrict__ O, float* __restrict__ lse,
                uint64_t wait_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar0 = sb + OFF_BAR;
  auto bar = [&](int k) { return bar0 + 8u * (uint32_t)k; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_BAR + 8 * NBAR);
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(smem + OFF_BAR + 8 * NBAR + 4);
  volatile int* never = reinterpret_cast<volatile int*>(smem + OFF_BAR + 8 * NBAR + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int k = 0; k < NBAR; ++k)
      mbar_init(bar(k), (k == B_P || k == B_P + 1 || k == B_MERGE) ? 128u : 1u);
    *abort_flag = 0;
    *never = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Unit w = unit_at(blockIdx.x, cv, C, unit_rows);
  const int nt = w.tl.count();                  // >= 1: every row sees itself

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmKc);
      prefetch_tmap(&tmVc);
      prefetch_tmap(&tmKb);
      prefetch_tmap(&tmVb);
      const int x0 = w.h * HD;                                  // Q column
      const int xb = w.kvh * HD;                                // block K, V column
      const int yq = w.b * C + w.q0;
      mbar_arrive_expect_tx(bar(B_Q), (w.split ? 1 : 2) * kTileB);
      tma_load_2d(sb + OFF_Q, &tmQ, x0, yq, bar(B_Q));
      tma_load_2d(sb + OFF_Q + kSub, &tmQ, x0 + 64, yq, bar(B_Q));
      if (!w.split) {
        tma_load_2d(sb + OFF_Q + kTileB, &tmQ, x0, yq + BM, bar(B_Q));
        tma_load_2d(sb + OFF_Q + kTileB + kSub, &tmQ, x0 + 64, yq + BM, bar(B_Q));
      }
      const int64_t slab0 = ((int64_t)w.b * cv.Hkv + w.kvh) * cv.slab_rows;
      uint32_t gi = 0;
      for (; gi < 2u * (uint32_t)nt; ++gi) {
        const uint32_t s = gi % NS;
        if (gi >= (uint32_t)NS &&
            !mbar_wait(bar(B_EMPTY + s), ((gi / NS) - 1) & 1, abort_flag, wait_ns))
          break;
        int kind, idx;
        w.tl.at((int)(gi >> 1), kind, idx);
        const bool isv = gi & 1;
        const CUtensorMap* map;
        int x, y;
        if (kind == kBlock) {
          map = isv ? &tmVb : &tmKb;
          x = xb;
          y = w.b * C + idx * BN;
        } else {
          map = isv ? &tmVc : &tmKc;
          x = 0;
          y = (int)(slab0 + (kind == kRing ? cv.m_cap : 0) + (int64_t)idx * BN);
        }
        const uint32_t dst = sb + OFF_RING + s * kTileB;
        mbar_arrive_expect_tx(bar(B_FULL + s), kTileB);
        tma_load_2d(dst, map, x, y, bar(B_FULL + s));
        tma_load_2d(dst + kSub, map, x + 64, y, bar(B_FULL + s));
      }
      // Drain: every copy issued has landed before the CTA may exit.
      mbar_wait(bar(B_Q), 0, never, kWaitLimitNs);
      for (uint32_t k = gi > (uint32_t)NS ? gi - NS : 0; k < gi; ++k)
        mbar_wait(bar(B_FULL + k % NS), (k / NS) & 1, never, kWaitLimitNs);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(BM, BN, false);
      constexpr uint32_t idesc_pv = idesc_bf16(BM, HD, true);
      auto wait = [&](int k, uint32_t phase) {
        return mbar_wait(bar(k), phase & 1, abort_flag, wait_ns);
      };
      auto wait_slot = [&](uint32_t gi) { return wait(B_FULL + gi % NS, gi / NS); };
      // S_half = Q K^T with the query rows of Q tile qt (qt = half, or 0 in a
      // split unit).
      auto qk = [&](int half, uint32_t gi, int qt) {
        const uint32_t kb = sb + OFF_RING + (gi % NS) * kTileB;
        const uint32_t qb = sb + OFF_Q + qt * kTileB;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t off = (k >> 2) * kSub + (k & 3) * 32;
          mma_bf16_ss(tmem + tm_s(half), desc_sw128(qb + off, 16, 1024),
                      desc_sw128(kb + off, 16, 1024), idesc_qk, k > 0);
        }
        mma_commit(bar(B_S + half));
      };
      auto pv = [&](int half, uint32_t gi, bool acc) {
        const uint32_t vb = sb + OFF_RING + (gi % NS) * kTileB;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_bf16_ts(tmem + tm_o(half), tmem + tm_s(half) + k * 8,
                      desc_sw128(vb + k * 2048, kSub, 1024), idesc_pv,
                      (acc || k > 0) ? 1u : 0u);
      };
      if (w.split) {
        // Tile t: K load 2 t, V load 2 t + 1; half 0 takes t = 2 j, half 1
        // t = 2 j + 1.  Every load is used once and its slot released after.
        const int nt0 = (nt + 1) / 2, nt1 = nt / 2;
        bool ok = wait(B_Q, 0) && wait_slot(0);
        if (ok) {
          tc_fence_after();
          qk(0, 0, 0);
          mma_commit(bar(B_EMPTY + 0));
          if (nt1 > 0 && (ok = wait_slot(2))) {
            tc_fence_after();
            qk(1, 2, 0);
            mma_commit(bar(B_EMPTY + 2 % NS));
          }
        }
        for (int j = 0; ok && j < nt0; ++j) {
          const uint32_t v0 = 4 * j + 1, k0 = 4 * j + 4;
          if (!wait(B_P + 0, j) || !wait_slot(v0)) break;
          tc_fence_after();
          pv(0, v0, j > 0);
          mma_commit(bar(B_EMPTY + v0 % NS));
          if (j + 1 < nt0) {
            if (!wait_slot(k0)) break;
            tc_fence_after();
            qk(0, k0, 0);
            mma_commit(bar(B_EMPTY + k0 % NS));
          } else {
            mma_commit(bar(B_O + 0));
          }
          if (j < nt1) {
            const uint32_t v1 = 4 * j + 3, k1 = 4 * j + 6;
            if (!wait(B_P + 1, j) || !wait_slot(v1)) break;
            tc_fence_after();
            pv(1, v1, j > 0);
            mma_commit(bar(B_EMPTY + v1 % NS));
            if (j + 1 < nt1) {
              if (!wait_slot(k1)) break;
              tc_fence_after();
              qk(1, k1, 0);
              mma_commit(bar(B_EMPTY + k1 % NS));
            } else {
              mma_commit(bar(B_O + 1));
            }
          }
        }
      } else if (wait(B_Q, 0) && wait_slot(0)) {
        tc_fence_after();
        qk(0, 0, 0);
        qk(1, 0, 1);
        mma_commit(bar(B_EMPTY + 0));
        for (int j = 0; j < nt; ++j) {
          const uint32_t vi = 2 * j + 1, ki = 2 * j + 2;
          const bool more = j + 1 < nt;
          if (!wait(B_P + 0, j) || !wait_slot(vi)) break;
          tc_fence_after();
          pv(0, vi, j > 0);
          if (more) {
            if (!wait_slot(ki)) break;
            tc_fence_after();
            qk(0, ki, 0);
          } else {
            mma_commit(bar(B_O + 0));
          }
          if (!wait(B_P + 1, j)) break;
          tc_fence_after();
          pv(1, vi, j > 0);
          mma_commit(bar(B_EMPTY + vi % NS));
          if (more) {
            qk(1, ki, 1);
            mma_commit(bar(B_EMPTY + ki % NS));
          } else {
            mma_commit(bar(B_O + 1));
          }
        }
      }
      // Drain: all MMAs of this CTA have finished before TMEM is freed.
      mma_commit(bar(B_FIN));
      mbar_wait(bar(B_FIN), 0, never, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int half = warp >> 2;
    const int r = threadIdx.x & 127;                    // row in half
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = rsqrtf((float)HD) * kLog2e;
    const uint32_t s_addr = tmem + lane_off + tm_s(half);
    const uint32_t o_addr = tmem + lane_off + tm_o(half);
    const int qh = w.q0 + (w.split ? 0 : half * BM);    // first row of half
    const int i = qh + r;                               // row in the block
    // Key tiles of this half: all of the unit's, or every other one.
    const int nth = w.split ? (nt + 1 - half) / 2 : nt;
    const int n = (int)min(cv.n, (int64_t)1 << 30);
    const int m_b = (int)w.m_b;
    // Ring: slot s is a key of row i iff its age (r0 - s) mod n <= lim, i.e.
    // s in [r0 - lim, r0] taken mod n (r0: slot of output t_b - 1).
    const int lim = (int)min(w.t_b - 1, (int64_t)n - 2 - i);
    const int r0 = w.t_b > 0 ? (int)((w.t_b - 1) % n) : 0;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nth; ++j) {
      int kind, idx;
      w.tl.at(w.split ? 2 * j + half : j, kind, idx);
      const int k0 = idx * BN;
      // Tile fully visible for every row of this half.
      const bool full =
          kind == kPrefix ? k0 + BN <= m_b
                          : (kind == kBlock && k0 + BN - 1 <= qh && k0 > qh + BM - 1 - n &&
                             k0 + BN <= C);
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_S + half), j & 1, abort_flag,
                                             wait_ns))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // This row's keys in the tile: columns [a1, b1] and [a2, b2].
      int a1, b1, a2 = 1, b2 = 0;
      if (kind == kPrefix) {
        a1 = 0;
        b1 = m_b - 1 - k0;
      } else if (kind == kBlock) {
        a1 = max(i - n + 1, 0) - k0;
        b1 = min(i, C - 1) - k0;
      } else if (lim < 0) {
        a1 = 1;
        b1 = 0;
      } else if (r0 >= lim) {
        a1 = r0 - lim - k0;
        b1 = r0 - k0;
      } else {
        a1 = -k0;
        b1 = r0 - k0;
        a2 = r0 - lim + n - k0;
        b2 = n - 1 - k0;
      }
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      uint32_t va[32], vb[32];
      auto max_chunk = [&](uint32_t* v, int c0) {
        if (!full) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int c = c0 + e;
            if (!((c >= a1 && c <= b1) || (c >= a2 && c <= b2)))
              v[e] = 0xff800000u;                          // -inf
          }
          tmem_st32(s_addr + c0, v);
        }
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          mx[0] = fmax3(mx[0], __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
          mx[1] = fmax3(mx[1], __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
          mx[2] = fmax3(mx[2], __uint_as_float(v[e + 4]), __uint_as_float(v[e + 5]));
          mx[3] = fmax3(mx[3], __uint_as_float(v[e + 6]), __uint_as_float(v[e + 7]));
        }
      };
      tmem_ld32(s_addr, va);
      tmem_wait_ld32(va);
      tmem_ld32(s_addr + 32, vb);
      max_chunk(va, 0);
      tmem_wait_ld32(vb);
      tmem_ld32(s_addr + 64, va);
      max_chunk(vb, 32);
      tmem_wait_ld32(va);
      tmem_ld32(s_addr + 96, vb);
      max_chunk(va, 64);
      tmem_wait_ld32(vb);
      max_chunk(vb, 96);
      if (!full) tmem_wait_st();
      const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
      // Lazy rescale (exact: O and l share the reference).  O_h is stable
      // here: S_h(j) completing implies PV_h(j-1) completed.
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
      const float nref = (m_run == -INFINITY) ? 0.f : -m_run;
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32_sync(o_addr + c * 32, ov);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st32(o_addr + c * 32, ov);
        }
      }
      uint32_t pk[2][32];
      const uint64_t sl2x2 = f2_pack(sl2, sl2), nref2 = f2_pack(nref, nref);
      uint64_t ps2[2] = {0, 0};
      auto exp_chunk = [&](const uint32_t* v, uint32_t* out) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int e = 2 * c;
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                           sl2x2, nref2),
                    x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          ps2[c & 1] = f2_add(ps2[c & 1], f2_pack(p0, p1));
          out[c] = pack_bf16(p0, p1);
        }
      };
      tmem_ld32(s_addr, va);
      tmem_wait_ld32(va);
      tmem_ld32(s_addr + 32, vb);
      exp_chunk(va, pk[0]);
      tmem_wait_ld32(vb);
      tmem_ld32(s_addr + 64, va);
      exp_chunk(vb, pk[0] + 16);
      tmem_wait_ld32(va);
      tmem_ld32(s_addr + 96, vb);
      exp_chunk(va, pk[1]);
      tmem_wait_ld32(vb);
      exp_chunk(vb, pk[1] + 16);
      float s0, s1, s2, s3;
      f2_unpack(ps2[0], s0, s1);
      f2_unpack(ps2[1], s2, s3);
      tmem_st32(s_addr, pk[0]);
      tmem_st32(s_addr + 32, pk[1]);
      l_run += (s0 + s1) + (s2 + s3);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_P + half));
    }
    if (w.split) {
      // Split unit: half 1 leaves (m, l) and its unnormalised O rows in the
      // K/V ring's shared memory once every MMA of the unit has completed
      // (the last PVs read V tiles there); half 0 merges them with its own.
      float* o1 = reinterpret_cast<float*>(smem + OFF_RING);   // [BM][HD]
      float* ml1 = o1 + BM * HD;                               // m [BM], l [BM]
      const int nt1 = nt / 2;
      auto wait_o = [&](int h) {
        return __all_sync(0xffffffffu, mbar_wait(bar(B_O + h), 0, abort_flag, wait_ns));
      };
      if (half == 1) {
        // Half 0's MMAs read ring slots too: wait for them even when half 1
        // had no tile.
        bool have = ok && wait_o(0) && nt1 > 0 && wait_o(1);
        if (have) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32_sync(o_addr + c * 32, ov);
#pragma unroll
            for (int e = 0; e < 32; ++e)
              o1[r * HD + ((c * 32 + e + r) & (HD - 1))] = __uint_as_float(ov[e]);
          }
        }
        ml1[r] = have ? m_run : -INFINITY;
        ml1[BM + r] = have ? l_run : 0.f;
        mbar_arrive(bar(B_MERGE));
      } else if (ok && wait_o(0) &&
                 __all_sync(0xffffffffu, mbar_wait(bar(B_MERGE), 0, abort_flag, wait_ns))) {
        tc_fence_after();
        const float m1 = ml1[r], l1 = ml1[BM + r];
        const float M = fmaxf(m_run, m1);
        const float a0 = ex2(m_run - M), a1 = l1 > 0.f ? ex2(m1 - M) : 0.f;
        const float L = l_run * a0 + l1 * a1;
        const float inv = 1.f / L;
        const size_t row = (size_t)w.b * C + i;
        __nv_bfloat16* orow = O + (row * cv.H + w.h) * HD;
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32_sync(o_addr + c * 32, ov);
          if (i < C) {
            uint32_t wv[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int c0 = c * 32 + 2 * e;
              const float x0 = __uint_as_float(ov[2 * e]) * a0 +
                               (a1 > 0.f ? o1[r * HD + ((c0 + r) & (HD - 1))] * a1 : 0.f);
              const float x1 = __uint_as_float(ov[2 * e + 1]) * a0 +
                               (a1 > 0.f ? o1[r * HD + ((c0 + 1 + r) & (HD - 1))] * a1 : 0.f);
              wv[e] = pack_bf16(x0 * inv, x1 * inv);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[e] = make_uint4(wv[4 * e], wv[4 * e + 1], wv[4 * e + 2], wv[4 * e + 3]);
          }
        }
        if (lse && i < C) lse[row * cv.H + w.h] = (M + log2f(L)) * kLn2;
      }
    } else if (ok && __all_sync(0xffffffffu,
                                mbar_wait(bar(B_O + half), 0, abort_flag, wait_ns))) {
      // Epilogue: O / l -> bf16 -> global; lse in natural log units.
      tc_fence_after();
      const float inv = 1.f / l_run;
      const size_t row = (size_t)w.b * C + i;
      __nv_bfloat16* orow = O + (row * cv.H + w.h) * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32_sync(o_addr + c * 32, ov);
        if (i < C) {
          uint32_t wv[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            wv[e] = pack_bf16(__uint_as_float(ov[2 * e]) * inv,
                              __uint_as_float(ov[2 * e + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(wv[4 * e], wv[4 * e + 1], wv[4 * e + 2], wv[4 * e + 3]);
        }
      }
      if (lse && i < C) lse[row * cv.H + w.h] = (m_run + log2f(l_run)) * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
  if (threadIdx.x == 0 && *abort_flag) flag_error(cv.err, kErrWaitTimeout);
}

}  // namespace

bool block_tc_supported(const CacheView& cv, int64_t block) {
  return cv.dtype == RSWA_BF16 && cv.d == HD && block >= kBlockTcMin &&
         (int64_t)cv.B * block < (int64_t(1) << 30) &&
         (int64_t)cv.B * cv.Hkv * cv.slab_rows + cv.n < (int64_t(1) << 31);
}

// Launched in stream order: an early start with the first prefix tiles
// requested before a dependency wait measured no faster for 64-256 tokens and
// 1.1 us slower for 1024 on the single-page cache.
cudaError_t launch_block_tc(const CacheView& cv, const void* q, const void* k,
                            const void* v, int64_t block, void* o, float* lse,
                            cudaStream_t s) {
  if (!block_tc_supported(cv, block)) return cudaErrorNotSupported;
  const int C = (int)block;
  const uint64_t brows = (uint64_t)cv.B * C;
  const uint64_t crows = (uint64_t)cv.B * cv.Hkv * cv.slab_rows;
  CUtensorMap mq, mkc, mvc, mkb, mvb;
  if (!make_tmap_rows_bf16(&mq, q, (uint64_t)cv.H * HD, brows) ||
      !make_tmap_rows_bf16(&mkc, cv.K, HD, crows) ||
      !make_tmap_rows_bf16(&mvc, cv.V, HD, crows) ||
      !make_tmap_rows_bf16(&mkb, k, (uint64_t)cv.Hkv * HD, brows) ||
      !make_tmap_rows_bf16(&mvb, v, (uint64_t)cv.Hkv * HD, brows))
    return cudaErrorInvalidValue;
  // Per device (the attribute belongs to the current device's context).
  cudaError_t e = cudaFuncSetAttribute(
      block_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  // Units of one query tile (each split over the two halves) while pairs of
  // tiles would not fill the SMs once: twice the CTAs, each with half the
  // key-tile chain.
  const int64_t pair_units = (int64_t)cv.B * ((C + 2 * BM - 1) / (2 * BM)) * cv.H;
  const int unit_rows = pair_units < cv.sms ? BM : 2 * BM;
  const int64_t units = (int64_t)cv.B * ((C + unit_rows - 1) / unit_rows) * cv.H;
  block_tc_kernel<<<(unsigned)units, kThreads, kSmemBytes, s>>>(
      mq, mkc, mvc, mkb, mvb, cv, C, unit_rows, static_cast<__nv_bfloat16*>(o), lse,
      phase_wait_limit_ns());
  return cudaGetLastError();
}

}  // namespace rswa
