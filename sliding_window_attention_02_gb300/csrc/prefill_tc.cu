// R-SWA prefill on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Computes, for every row i of every sequence and head,
//   O_i = softmax_{j in N(i)}(q_i . k_j / sqrt(d)) . v_j,
//   N(i) = {j <= i}                                   for prefix rows i < m,
//   N(i) = {j < m} U {j : max(m, i - n + 1) <= j <= i} for output rows,
// ("Unlimited-OCR deep dive": N(t) = P U D_n(t); "Unlimited OCR", GeekNews:
// the two-segment window of size m + n).
//
// A work unit is two adjacent 128-row query tiles ("halves") of one head; it
// walks the union of their key tiles: the prefix tiles 0 .. ceil(m/128)-1 up
// to the diagonal, then the band tiles that hold the last n keys of the
// output rows.  Tiles the mask excludes entirely are never loaded.  Both
// halves share every K and V tile.  Per-element masking runs only on tiles
// the mask covers partially for that half.  A CTA takes one unit per round
// of gridDim.x units of the heavy-first order (a snake order, see
// snake_unit), and its producer loads the next unit's Q and first K/V tiles
// while the current unit's last tiles and epilogue run.  The host launches
// one CTA per SM when units are short (few key tiles: band-dominated
// sequences), else one CTA per unit.
//
// Roles (320 threads):
//   warps 0-3   softmax of half 0 (thread r owns row r = TMEM lane r)
//   warps 4-7   softmax of half 1
//   warp 8      TMA producer: Q0, Q1, then K_j, V_j into a 4-slot ring
//   warp 9      TMEM allocator and MMA issuer (one thread)
// TMEM (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each; P_h (bf16,
// two per column) overwrites the first 64 columns of S_h once S_h is read,
// and feeds the PV MMA straight from TMEM.  The issue order
//   QK0(0) QK1(0) | PV0(j) QK0(j+1) PV1(j) QK1(j+1) | ...
// keeps the tensor core on one half while the other half's softmax runs, and
// relies on the in-order execution of one thread's tcgen05.mma stream for
// S_h being rewritten only after PV_h has read P_h.
// Across units: Q is reloaded once the last QK MMA of the unit has completed
// (B_QFREE), and PV_h of a unit's first tile overwrites O_h only after the
// softmax warps of half h have read the previous unit's O_h (B_OFREE).
// Every wait is bounded; on a timeout the CTA drains its own copies and MMAs,
// frees TMEM, sets the cache's device error flag and exits.
#include <cuda.h>

#include <algorithm>
#include <climits>

#include "rswa_device.cuh"
#include "tc_ptx.cuh"

namespace rswa {
namespace {

using namespace ptx;

constexpr int BM = 128;                        // rows per half
constexpr int BN = 128;                        // keys per tile
constexpr int HD = 128;                        // largest head_dim (smem layout)
constexpr int kSoftmaxThreads = 256;
constexpr int kThreads = kSoftmaxThreads + 64;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int NS = 4;                          // K/V ring slots
constexpr uint32_t kSub = BM * 64 * 2;         // [128][64] bf16, 128B-swizzled
constexpr uint32_t kTileB = BM * HD * 2;       // [128][128] bf16 = 32 KB (2 kSub)
constexpr uint32_t OFF_Q = 0;                  // Q0, Q1
constexpr uint32_t OFF_RING = 2 * kTileB;
constexpr uint32_t OFF_BAR = OFF_RING + NS * kTileB;
constexpr uint32_t kSmemBytes = OFF_BAR + 256 + 1024;  // + 1 KB alignment slack
static_assert(kTileB == 2 * kSub, "a tile is two 64-column swizzled halves");

__host__ __device__ constexpr uint32_t tm_s(int half) { return half ? 128u : 0u; }
__host__ __device__ constexpr uint32_t tm_o(int half) { return half ? 384u : 256u; }
constexpr uint32_t TM_COLS = 512;
constexpr float kRescaleThreshold = 8.0f;      // log2 units
constexpr uint64_t kWaitLimitNs = 1000000000ull;
// Below this mean number of key tiles per unit the launch is persistent.
constexpr int64_t kPersistentTilesPerUnit = 16;

// barrier indices
constexpr int B_Q = 0;
constexpr int B_FULL = 1;                      // NS slots
constexpr int B_EMPTY = B_FULL + NS;           // NS slots
constexpr int B_S = B_EMPTY + NS;              // 2 halves
constexpr int B_P = B_S + 2;                   // 2 halves
constexpr int B_O = B_P + 2;                   // 2 halves
constexpr int B_FIN = B_O + 2;
constexpr int B_QFREE = B_FIN + 1;             // Q buffer may be reloaded
constexpr int B_OFREE = B_QFREE + 1;           // 2 halves: O_h read out
constexpr int NBAR = B_OFREE + 2;

struct TileRange {
  int np;        // prefix tiles 0 .. np-1
  int kb_start;  // first band tile
  int nt;        // tiles visited
};

// Key tiles visited by rows [r_lo, r_hi] of a sequence with prefix m,
// window n and length L.
__device__ __forceinline__ TileRange tile_range(int r_lo, int r_hi, int m, int n,
                                                int L) {
  TileRange t;
  const int i_hi = min(r_hi, L - 1);
  t.np = min((m + BN - 1) / BN, i_hi / BN + 1);
  const int i_lo = max(r_lo, m);
  int nb = 0;
  t.kb_start = t.np;
  if (i_lo <= i_hi) {
    const int band_lo = max(m, i_lo - n + 1);
    t.kb_start = max(band_lo / BN, t.np);
    nb = max(0, i_hi / BN - t.kb_start + 1);
  }
  t.nt = t.np + nb;
  return t;
}

__device__ __forceinline__ int tile_at(const TileRange& t, int j) {
  return j < t.np ? j : t.kb_start + (j - t.np);
}

// Whether key tile k0 .. k0+BN-1 holds a key that some row of the 128-row
// query tile at qh sees (sequence with prefix m, window n, length L).
// Prefix keys are seen by every output row and causally by prefix rows;
// keys at or past m only by output rows i with i - n + 1 <= key <= i, of
// which the first output row reaches furthest back.  A (query tile, key
// tile) product that fails this is skipped: both tiles of a unit walk the
// union of their key tiles, and e.g. a band-only unit has two such
// products out of six (the persistent form skips them).
__device__ __forceinline__ bool tile_touches(int k0, int qh, int m, int n, int L) {
  const int i_hi = min(qh + BM - 1, L - 1);     // last row of the tile
  if (k0 > i_hi) return false;                  // above the diagonal
  if (k0 < m) return true;                      // prefix keys, k0 <= i_hi
  const int i_lo = max(qh, m);                  // first output row
  if (i_lo > i_hi) return false;                // prefix rows only
  return k0 + BN - 1 >= i_lo - n + 1;
}

// The k-th unit of CTA b out of G: rounds of G units, walked forward in even
// rounds and backward in odd ones, so that with units in heavy-first order
// every CTA's sum of work is near the mean (as list scheduling would give,
// with no shared counter).  -1 past the last unit.
__device__ __forceinline__ int snake_unit(int k, int b, int G, int units) {
  const int u = k * G + ((k & 1) ? G - 1 - b : b);
  return u < units ? u : -1;
}

// Work unit u: head u % H, tile pair total_pairs - 1 - u / H (heavy pairs
// first: a pair's work grows with its position in the sequence).
struct Unit {
  int h, kvh, m, L, q0;
  int64_t row0;
  TileRange tr;
};

__device__ __forceinline__ Unit unit_at(int u, const CacheView& cv,
                                        const SeqTable& st, int total_pairs) {
  Unit w;
  const int H = cv.H;
  w.h = u % H;
  const int g = total_pairs - 1 - u / H;
  int sl = 0;
  while (sl + 1 < st.nseq && st.tile_off[sl + 1] <= g) ++sl;
  const int pr = g - st.tile_off[sl];                      // pair in sequence
  w.m = st.m[sl];
  const int n = (int)min(cv.n, (int64_t)1 << 30);
  w.L = w.m + (int)st.T[sl];
  w.kvh = w.h / (H / cv.Hkv);                              // KV head read
  w.row0 = st.row_off[sl];
  w.q0 = pr * 2 * BM;
  w.tr = tile_range(w.q0, w.q0 + 2 * BM - 1, w.m, n, w.L);
  return w;
}

// Tile bytes of a head_dim-D operand: D / 64 swizzle atoms of 128 rows.
template <int D>
constexpr uint32_t tile_bytes() { return (uint32_t)(D / 64) * kSub; }

// D: head_dim, 64 or 128 (one or two 64-column atoms per Q/K/V tile; the
// shared-memory layout is the head_dim-128 one either way).
// wait_ns bounds every wait for a pipeline phase (phase_wait_limit_ns());
// the drains before exit keep kWaitLimitNs.
// PERSIST: a CTA may take several units (one per round of gridDim units)
// and skips (query tile, key tile) products the mask excludes entirely;
// otherwise exactly one unit, blockIdx.x, the cross-unit barriers (B_QFREE,
// B_OFREE) and phase counters fold away, and every product of the unit's
// tile list runs.
template <bool PERSIST, int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, CacheView cv,
                  SeqTable st, __nv_bfloat16* __restrict__ O, int total_pairs,
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
  const int H = cv.H;
  const int units = total_pairs * H;
  constexpr int kMaxRounds = PERSIST ? INT_MAX : 1;

  if (threadIdx.x == 0) {
    for (int k = 0; k < NBAR; ++k) {
      const bool per_row = k == B_P || k == B_P + 1 || k == B_OFREE || k == B_OFREE + 1;
      mbar_init(bar(k), per_row ? 128u : 1u);
    }
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

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      uint32_t gi = 0, nq = 0;                  // K/V loads, Q loads issued
      bool ok = true;
      for (int k = 0, u; ok && k < kMaxRounds && (u = snake_unit(k, blockIdx.x, gridDim.x, units)) >= 0;
           ++k) {
        const Unit w = unit_at(u, cv, st, total_pairs);
        if (w.tr.nt == 0) continue;
        // Q of the previous unit is read by its last QK MMA.
        if (nq > 0 && !mbar_wait(bar(B_QFREE), (nq - 1) & 1, abort_flag, wait_ns))
          break;
        const int x0 = w.h * D;                                // Q column
        const int xk = w.kvh * D;                              // K, V column
        const int yq = (int)(w.row0 + w.q0);
        mbar_arrive_expect_tx(bar(B_Q), 2 * tile_bytes<D>());
        tma_load_2d(sb + OFF_Q, &tmQ, x0, yq, bar(B_Q));
        if (D > 64) tma_load_2d(sb + OFF_Q + kSub, &tmQ, x0 + 64, yq, bar(B_Q));
        tma_load_2d(sb + OFF_Q + kTileB, &tmQ, x0, yq + BM, bar(B_Q));
        if (D > 64) tma_load_2d(sb + OFF_Q + kTileB + kSub, &tmQ, x0 + 64, yq + BM, bar(B_Q));
        ++nq;
        for (int idx = 0; idx < 2 * w.tr.nt; ++idx, ++gi) {
          const uint32_t s = gi % NS;
          if (gi >= (uint32_t)NS &&
              !mbar_wait(bar(B_EMPTY + s), ((gi / NS) - 1) & 1, abort_flag,
                         wait_ns)) {
            ok = false;
            break;
          }
          const CUtensorMap* map = (idx & 1) ? &tmV : &tmK;
          const int y = (int)(w.row0 + (int64_t)tile_at(w.tr, idx >> 1) * BN);
          const uint32_t dst = sb + OFF_RING + s * kTileB;
          mbar_arrive_expect_tx(bar(B_FULL + s), tile_bytes<D>());
          tma_load_2d(dst, map, xk, y, bar(B_FULL + s));
          if (D > 64) tma_load_2d(dst + kSub, map, xk + 64, y, bar(B_FULL + s));
        }
      }
      // Drain: every copy issued has landed before the CTA may exit (older
      // loads of a ring slot completed before the slot was reissued).
      if (nq > 0) mbar_wait(bar(B_Q), (nq - 1) & 1, never, kWaitLimitNs);
      for (uint32_t idx = gi > (uint32_t)NS ? gi - NS : 0; idx < gi; ++idx)
        mbar_wait(bar(B_FULL + idx % NS), (idx / NS) & 1, never, kWaitLimitNs);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(BM, BN, false);
      constexpr uint32_t idesc_pv = idesc_bf16(BM, D, true);
      auto wait = [&](int k, uint32_t phase) {
        return mbar_wait(bar(k), phase & 1, abort_flag, wait_ns);
      };
      auto wait_slot = [&](uint32_t gi) { return wait(B_FULL + gi % NS, gi / NS); };
      // S_h = Q_h K^T from the K tile in the ring slot of load gi.
      auto qk = [&](int half, uint32_t gi) {
        const uint32_t kb = sb + OFF_RING + (gi % NS) * kTileB;
        const uint32_t qb = sb + OFF_Q + half * kTileB;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kSub + (k & 3) * 32;
          mma_bf16_ss(tmem + tm_s(half), desc_sw128(qb + off, 16, 1024),
                      desc_sw128(kb + off, 16, 1024), idesc_qk, k > 0);
        }
        mma_commit(bar(B_S + half));
      };
      // O_h (+)= P_h V from TMEM P_h and the V tile of load gi.
      auto pv = [&](int half, uint32_t gi, bool acc) {
        const uint32_t vb = sb + OFF_RING + (gi % NS) * kTileB;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_bf16_ts(tmem + tm_o(half), tmem + tm_s(half) + k * 8,
                      desc_sw128(vb + k * 2048, kSub, 1024), idesc_pv,
                      (acc || k > 0) ? 1u : 0u);
      };
      const int nwin = (int)min(cv.n, (int64_t)1 << 30);
      uint32_t gi = 0, gt = 0, kq = 0;          // loads, tiles, units done
      bool ok = true;
      for (int k = 0, u; ok && k < kMaxRounds && (u = snake_unit(k, blockIdx.x, gridDim.x, units)) >= 0;
           ++k) {
        const Unit w = unit_at(u, cv, st, total_pairs);
        const int nt = w.tr.nt;
        if (nt == 0) continue;
        if (!wait(B_Q, kq) || !wait_slot(gi)) break;
        tc_fence_after();
        if constexpr (!PERSIST) {
          // Long units: every product of the unit's tile list runs.  (This
          // issuing thread sits on the critical path: a per-tile skip test
          // here measured 1-6 % slower on the multi-page prefill.)
          qk(0, gi);
          qk(1, gi);
          mma_commit(bar(B_EMPTY + gi % NS));
          if (nt == 1) mma_commit(bar(B_QFREE));
          for (int j = 0; j < nt; ++j) {
            const uint32_t vi = gi + 2 * j + 1, ki = gi + 2 * j + 2;
            const bool more = j + 1 < nt;
            if (!wait(B_P + 0, gt + j) || !wait_slot(vi)) {
              ok = false;
              break;
            }
            tc_fence_after();
            pv(0, vi, j > 0);
            if (more) {
              if (!wait_slot(ki)) {
                ok = false;
                break;
              }
              tc_fence_after();
              qk(0, ki);
            } else {
              mma_commit(bar(B_O + 0));
            }
            if (!wait(B_P + 1, gt + j)) {
              ok = false;
              break;
            }
            tc_fence_after();
            pv(1, vi, j > 0);
            mma_commit(bar(B_EMPTY + vi % NS));
            if (more) {
              qk(1, ki);
              mma_commit(bar(B_EMPTY + ki % NS));
              if (j + 2 == nt) mma_commit(bar(B_QFREE));   // last QK of the unit
            } else {
              mma_commit(bar(B_O + 1));
            }
          }
        } else {
          // Short units: products the mask excludes entirely are skipped.
          // A skipped QK still completes S_h's barrier (the softmax warps
          // hand P_h back at once); the unit's first PV of a half that runs
          // overwrites O_h.
          auto use = [&](int half, int j) {
            return tile_touches(tile_at(w.tr, j) * BN, w.q0 + half * BM, w.m, nwin, w.L);
          };
          bool pv_done[2] = {false, false};
          auto qk_if = [&](int half, uint32_t g, bool on) {
            if (on)
              qk(half, g);
            else
              mma_commit(bar(B_S + half));
          };
          auto pv_if = [&](int half, uint32_t g, bool on) {
            if (!on) return;
            pv(half, g, pv_done[half]);
            pv_done[half] = true;
          };
          bool u0 = use(0, 0), u1 = use(1, 0);
          qk_if(0, gi, u0);
          qk_if(1, gi, u1);
          mma_commit(bar(B_EMPTY + gi % NS));
          if (nt == 1) mma_commit(bar(B_QFREE));
          for (int j = 0; j < nt; ++j) {
            const uint32_t vi = gi + 2 * j + 1, ki = gi + 2 * j + 2;
            const bool more = j + 1 < nt;
            const bool n0 = more && use(0, j + 1), n1 = more && use(1, j + 1);
            // PV_h of the unit's first tile overwrites O_h: the previous
            // unit's epilogue must have read it.
            if (!wait(B_P + 0, gt + j) || !wait_slot(vi) ||
                (j == 0 && kq > 0 && !wait(B_OFREE + 0, kq - 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
            pv_if(0, vi, u0);
            if (more) {
              if (!wait_slot(ki)) {
                ok = false;
                break;
              }
              tc_fence_after();
              qk_if(0, ki, n0);
            } else {
              mma_commit(bar(B_O + 0));
            }
            if (!wait(B_P + 1, gt + j) ||
                (j == 0 && kq > 0 && !wait(B_OFREE + 1, kq - 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
            pv_if(1, vi, u1);
            mma_commit(bar(B_EMPTY + vi % NS));
            if (more) {
              qk_if(1, ki, n1);
              mma_commit(bar(B_EMPTY + ki % NS));
              if (j + 2 == nt) mma_commit(bar(B_QFREE));   // last QK of the unit
            } else {
              mma_commit(bar(B_O + 1));
            }
            u0 = n0;
            u1 = n1;
          }
        }
        gi += 2 * nt;
        gt += nt;
        ++kq;
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
    const float sl2 = rsqrtf((float)D) * kLog2e;
    const uint32_t s_addr = tmem + lane_off + tm_s(half);
    const uint32_t o_addr = tmem + lane_off + tm_o(half);
    uint32_t gt = 0, kq = 0;                            // tiles, units done
    bool ok = true;
    for (int k = 0, u; ok && k < kMaxRounds && (u = snake_unit(k, blockIdx.x, gridDim.x, units)) >= 0;
           ++k) {
      const Unit w = unit_at(u, cv, st, total_pairs);
      const TileRange& tr = w.tr;
      if (tr.nt == 0) continue;
      const int m = w.m;
      const int n = (int)min(cv.n, (int64_t)1 << 30);
      const int qh = w.q0 + half * BM;                  // first row of half
      const int i = qh + r;                             // row in sequence
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < tr.nt; ++j) {
        const int k0 = tile_at(tr, j) * BN;
        // Tile fully visible for this half: every key <= every row, and every
        // key either in the prefix or inside every row's window.
        const bool full = (k0 + BN - 1 <= qh) &&
                          ((k0 + BN - 1 < m) || (max(k0, m) > qh + BM - 1 - n));
        // The warp agrees on the outcome, so no lane reaches the warp-wide
        // TMEM loads alone.
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_S + half), (gt + j) & 1,
                                               abort_flag, wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (PERSIST && !tile_touches(k0, qh, m, n, w.L)) {
          // No MMA wrote S_h for this tile: P_h is "ready" at once.
          tc_fence_before();
          mbar_arrive(bar(B_P + half));
          continue;
        }
        // Pass 1: row maximum over the visible logits, 32 columns at a time.
        const int hi = i - k0;   // visible: c <= hi && (c < a || c > b)
        const int a = m - k0;
        const int b = i - n - k0;
        // The load of chunk c + 1 is in flight while chunk c is reduced.
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        uint32_t va[32], vb[32];
        auto max_chunk = [&](uint32_t* v, int c0) {
          if (!full) {
            // Mask in place and write back, so pass 2 reads masked logits.
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int c = c0 + e;
              if (!(c <= hi && (c < a || c > b))) v[e] = 0xff800000u;  // -inf
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
        // Lazy rescale: keep the reference maximum unless it grew by > 2^8.
        // Exact either way: O and l share the reference.  O_h is stable here:
        // S_h(j) completing implies PV_h(j-1) completed (one MMA stream).
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
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32_sync(o_addr + c * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e)
              o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(o_addr + c * 32, o);
          }
        }
        // Pass 2: P_h = exp2(x - ref) as bf16 -> TMEM over the first 64
        // columns of S_h (two bf16 per column), 64 logits at a time.  Columns
        // 0..63 of S_h are read before any P column is written.
        uint32_t pk[2][32];
        // Two logits per packed f32x2 FMA and sum; the load of chunk c + 1
        // is in flight while chunk c is exponentiated.
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
        const float psum = (s0 + s1) + (s2 + s3);
        tmem_st32(s_addr, pk[0]);
        tmem_st32(s_addr + 32, pk[1]);
        l_run += psum;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(B_P + half));
      }
      if (!ok) break;
      // Epilogue: O / l -> bf16 -> global, then O_h is free for the next unit.
      if (!__all_sync(0xffffffffu,
                      mbar_wait(bar(B_O + half), kq & 1, abort_flag, wait_ns)))
        break;
      tc_fence_after();
      const float inv = 1.f / l_run;
      __nv_bfloat16* orow = O + ((w.row0 + i) * H + w.h) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32_sync(o_addr + c * 32, o);
        if (i < w.L) {
          uint32_t wv[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            wv[e] = pack_bf16(__uint_as_float(o[2 * e]) * inv,
                              __uint_as_float(o[2 * e + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(wv[4 * e], wv[4 * e + 1], wv[4 * e + 2], wv[4 * e + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(B_OFREE + half));
      gt += tr.nt;
      ++kq;
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

// ---- host: tensor maps through the driver entry point ----------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                  void*, const cuuint64_t*, const cuuint64_t*,
                                  const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  // Looked up once (thread-safe static initialisation).
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return nullptr;
  }();
  return fn;
}

// [rows][heads*d] bf16 viewed as a 2-D tensor; box 64 columns x 128 rows,
// 128-byte swizzle; rows past `rows` read as zero.
bool make_map(CUtensorMap* map, const void* base, int H, int d, int64_t rows) {
  return make_tmap_rows_bf16(map, base, (uint64_t)H * d, (uint64_t)rows);
}

}  // namespace

bool make_tmap_rows_bf16(CUtensorMap* map, const void* base, uint64_t cols,
                         uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Key tiles visited by all tile pairs of the launch (one head): the host
// twin of tile_range, summed over the pairs.
static int64_t host_tiles(const SeqTable& st, int64_t n_window) {
  const int64_t n = std::min<int64_t>(n_window, int64_t(1) << 30);
  int64_t total = 0;
  for (int sq = 0; sq < st.nseq; ++sq) {
    const int64_t m = st.m[sq], L = m + st.T[sq];
    for (int64_t q0 = 0; q0 < L; q0 += 2 * BM) {
      const int64_t i_hi = std::min(q0 + 2 * BM - 1, L - 1);
      const int64_t np = std::min((m + BN - 1) / BN, i_hi / BN + 1);
      const int64_t i_lo = std::max(q0, m);
      int64_t nb = 0;
      if (i_lo <= i_hi) {
        const int64_t band_lo = std::max(m, i_lo - n + 1);
        const int64_t kb = std::max(band_lo / BN, np);
        nb = std::max<int64_t>(0, i_hi / BN - kb + 1);
      }
      total += np + nb;
    }
  }
  return total;
}

bool prefill_tc_supported(const CacheView& cv) {
  return cv.dtype == RSWA_BF16 && (cv.d == 64 || cv.d == 128) && encode_fn() != nullptr;
}

template <int D>
static cudaError_t launch_d(const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, const CacheView& cv,
                            const SeqTable& st, void* O, int pairs, bool persist,
                            int64_t grid, cudaStream_t s) {
  // Per device (the attribute belongs to the current device's context).
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<true, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(prefill_tc_kernel<false, D>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const uint64_t wait_ns = phase_wait_limit_ns();
  if (persist)
    prefill_tc_kernel<true, D><<<(unsigned)grid, kThreads, kSmemBytes, s>>>(
        mq, mk, mv, cv, st, static_cast<__nv_bfloat16*>(O), pairs, wait_ns);
  else
    prefill_tc_kernel<false, D><<<(unsigned)grid, kThreads, kSmemBytes, s>>>(
        mq, mk, mv, cv, st, static_cast<__nv_bfloat16*>(O), pairs, wait_ns);
  return cudaGetLastError();
}

cudaError_t launch_prefill_tc(const CacheView& cv, const SeqTable& st_in,
                              const void* Q, const void* K, const void* V,
                              void* O, int64_t total_rows, cudaStream_t s) {
  if (!prefill_tc_supported(cv)) return cudaErrorNotSupported;
  const int64_t end_row = st_in.row_off[0] + total_rows;
  if (end_row >= (int64_t(1) << 31)) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, Q, cv.H, cv.d, end_row) || !make_map(&mk, K, cv.Hkv, cv.d, end_row) ||
      !make_map(&mv, V, cv.Hkv, cv.d, end_row))
    return cudaErrorInvalidValue;
  // Work units are pairs of 128-row tiles: tile_off counts pairs here.
  SeqTable st = st_in;
  int pairs = 0;
  st.tile_off[0] = 0;
  for (int i = 0; i < st.nseq; ++i) {
    const int64_t L = st.m[i] + st.T[i];
    pairs += (int)((L + 2 * BM - 1) / (2 * BM));
    st.tile_off[i + 1] = pairs;
  }
  if (pairs == 0) return cudaSuccess;
  const int64_t units = (int64_t)pairs * cv.H;
  if (units >= (int64_t(1) << 31)) return cudaErrorNotSupported;
  // One CTA per SM fits (shared memory, 512 TMEM columns).  Units of few key
  // tiles (band-dominated sequences) run persistently, one unit per round of
  // gridDim units, so that the next unit's loads overlap this one's tail;
  // long units run one per CTA, left to the hardware's dynamic scheduling.
  const bool persist = host_tiles(st, cv.n) < kPersistentTilesPerUnit * pairs;
  const int64_t grid = persist ? std::min<int64_t>(units, std::max(cv.sms, 1)) : units;
  if (cv.d == 64) return launch_d<64>(mq, mk, mv, cv, st, O, pairs, persist, grid, s);
  return launch_d<128>(mq, mk, mv, cv, st, O, pairs, persist, grid, s);
}

}  // namespace rswa
