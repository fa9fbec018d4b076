// Grouped-query R-SWA decode on the tensor cores, stream-K form.
//
// What it computes is decode_gqa_tc.cu's: for every KV head (b, kv) the G
// query heads that read it attend its visible keys, the prefix rows 0..m_b-1
// and the filled ring slots ("Unlimited-OCR deep dive": N(t) = P U D_n(t)),
// as S^T = K Q_G^T and O^T += V^T P^T on tcgen05 with TMEM accumulators.
// How the work is laid out differs: the key tiles of all KV heads form one
// list, head after head (a head's ceil(m_b / 128) prefix tiles, then its
// ceil(n / 128) ring tiles), and a grid of persistent CTAs (two per SM)
// splits that list into equal ranges.  A CTA streams its range through one
// TMA ring without draining between heads; each head it touches is a
// segment whose partial (m, l, O) it publishes, and the last of the head's
// CTAs merges them (a head inside one CTA writes o directly).  The split
// depends on m_b only (never on t_b), so a fused step may advance t_b while
// other CTAs of the launch still start.
//
// Roles (320 threads):
//   warps 0-3  softmax: thread t owns key t of a tile (TMEM lane t)
//   warps 4-7  segment epilogue: thread e owns row d = e of O^T; reads the
//              segment's O^T out of TMEM, publishes or merges, and stages
//              the next segment's Q^T
//   warp 8     TMA producer: K and V tiles into a 3-slot ring
//   warp 9     TMEM allocator and MMA issuer (one thread)
// TMEM (64 columns): S^T double buffer at columns 0 and 16, O^T double
// buffer (by segment) at 32 and 48, so the next segment's PV MMAs run while
// the epilogue warps read the previous one out.  The MMA order S(0) S(1)
// PV(0) S(2) PV(1) ... lets the softmax of tile j run while PV(j-1)
// executes; at a segment boundary the last PV of the old segment is issued
// before the first S of the new one, while its Q^T is staged.  O^T is
// rescaled lazily (threshold 2^8).  A head's last prefix tile and its ring
// tiles are fetched as 8-row TMA boxes covering their rows; the ring slots
// are zeroed at CTA start, so rows a clamped load leaves hold finite values
// that masked probabilities (p = 0) multiply to exactly 0.
// Every wait is bounded (wait_ns for the pipeline's phases, kWaitLimitNs for
// the drains); on a timeout the CTA drains its copies and MMAs, frees TMEM
// and sets the cache's device error flag.
#include <cuda.h>

#include <algorithm>

#include "rswa_device.cuh"
#include "rswa_internal.h"
#include "tc_ptx.cuh"

namespace rswa {
namespace {

using namespace ptx;

constexpr int HD = 128;                     // head_dim
constexpr int BN = 128;                     // keys per tile
constexpr int NQ = 16;                      // MMA N: query heads, padded
constexpr int kEpiWarp0 = 4;                // warps 4-7
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr int NS = 3;                       // ring slots (a K or a V tile)
constexpr uint32_t kSub = BN * 64 * 2;      // [128][64] bf16, 128B-swizzled
constexpr uint32_t kTileB = 2 * kSub;       // [128][128] bf16 = 32 KB
constexpr uint32_t kNAtom = NQ * 128;       // [16][64] bf16 atom = 2 KB
constexpr uint32_t OFF_RING = 0;            // NS tiles, 1 KB aligned
constexpr uint32_t OFF_Q = OFF_RING + NS * kTileB;   // Q^T: 2 atoms
constexpr uint32_t OFF_P = OFF_Q + 2 * kNAtom;       // P^T double buffer
constexpr uint32_t OFF_BAR = OFF_P + 4 * kNAtom;
constexpr int B_FULL = 0;                   // NS
constexpr int B_EMPTY = B_FULL + NS;        // NS
constexpr int B_S = B_EMPTY + NS;           // 2: S^T(j) in TMEM
constexpr int B_SFREE = B_S + 2;            // 2: S^T(j) read (128)
constexpr int B_P = B_SFREE + 2;            // 2: P^T(j) in smem (128)
constexpr int B_PFREE = B_P + 2;            // 2: PV(j) done
constexpr int B_QFULL = B_PFREE + 2;        // Q^T of the next segment staged (128)
constexpr int B_QFREE = B_QFULL + 1;        // a segment's last S done
constexpr int B_OREADY = B_QFREE + 1;       // 2: a segment's last PV done
constexpr int B_OFREE = B_OREADY + 2;       // 2: its O^T read out (128)
constexpr int B_ML = B_OFREE + 2;           // 2: its m, l written (128)
constexpr int B_MLFREE = B_ML + 2;          // 2: m, l read (128)
constexpr int B_SYNCS = B_MLFREE + 2;       // softmax warps' barrier (128)
constexpr int B_SYNCE = B_SYNCS + 1;        // epilogue warps' barrier (128)
constexpr int B_FIN = B_SYNCE + 1;          // every MMA done
constexpr int NBAR = B_FIN + 1;
constexpr int kMaxSeg = 48;                 // segments per CTA
struct Seg {
  int bkv;        // b * H_kv + kv
  int np;         // prefix tiles of the head
  int i0, i1;     // this CTA's tiles of the head's list
  int slot;       // this CTA's partial slot of the head
  int nparts;     // CTAs sharing the head
  int m_b;
  int pad;
};
constexpr uint32_t OFF_SEG = (OFF_BAR + 8 * NBAR + 15) & ~15u;
constexpr uint32_t OFF_ML = OFF_SEG + kMaxSeg * sizeof(Seg);  // [2][NQ] m, [2][4][NQ] l
constexpr uint32_t OFF_RED = OFF_ML + (2 * NQ + 2 * 4 * NQ) * 4;  // [2][4][NQ] max
constexpr uint32_t OFF_MISC = OFF_RED + 2 * 4 * NQ * 4;
constexpr uint32_t kSmemBytes = OFF_MISC + 32 + 1024;          // + alignment slack
static_assert(OFF_SEG % 16 == 0, "segment table alignment");
static_assert(kSmemBytes + 1024 <= 233472 / 2, "two CTAs per SM");
constexpr uint32_t TM_S = 0, TM_O = 32, TM_COLS = 64;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Stores v at a with the L2 eviction priority of `pol` (a createpolicy
// descriptor).
__device__ __forceinline__ void st_hint(float* a, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(a), "f"(v), "l"(pol)
               : "memory");
}
// Evict-last priority for a split-K partial: kept in L2 while the streamed
// keys pass through, until the merge reads and discards it.
__device__ __forceinline__ uint64_t partial_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

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

// Drops, without write-back, the L2 lines that lie wholly inside [lo, hi):
// merged split-K partials, which nothing reads again before a later launch
// rewrites them, would otherwise go back to DRAM when the streamed keys
// evict them.  The lines at the two ends may hold another head's partials
// and are kept.  Thread t of nt takes lines t, t + nt, ...; the caller has
// made every read of the range complete (a barrier after the merge).
__device__ __forceinline__ void discard_l2_inside(const void* lo, const void* hi, int t,
                                                  int nt) {
  const uintptr_t a = (reinterpret_cast<uintptr_t>(lo) + 127) & ~uintptr_t(127);
  const uintptr_t e = reinterpret_cast<uintptr_t>(hi) & ~uintptr_t(127);
  for (uintptr_t p = a + (uintptr_t)t * 128; p < e; p += (uintptr_t)nt * 128)
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// The CTA of `P` whose range holds tile t of `tot` (ranges [c tot / P,
// (c + 1) tot / P)).
__device__ __forceinline__ int owner(int64_t t, int64_t tot, int P) {
  int c = (int)((t * P) / tot);
  while (c + 1 < P && ((int64_t)(c + 1) * tot) / P <= t) ++c;
  while (c > 0 && ((int64_t)c * tot) / P > t) --c;
  return c;
}

// Segment table of CTA c, built by one warp from m_b: the heads whose tiles
// overlap the CTA's range.  Returns the number of segments, or -1 when they
// do not fit the table.
__device__ int build_segments(const CacheView& cv, int c, int P, Seg* segs, int lane) {
  const int Hkv = cv.Hkv;
  const int rt = (int)((cv.n + BN - 1) / BN);
  int64_t tot = 0;
  for (int b0 = 0; b0 < cv.B; b0 += 32) {
    const int b = b0 + lane;
    int64_t tb = 0;
    if (b < cv.B) tb = (int64_t)Hkv * ((cv.m_dev[b] + BN - 1) / BN + rt);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tb += __shfl_xor_sync(0xffffffffu, tb, off);
    tot += tb;
  }
  const int64_t t0 = ((int64_t)c * tot) / P, t1 = ((int64_t)(c + 1) * tot) / P;
  if (t1 <= t0) return 0;                             // fewer tiles than CTAs
  int nseg = 0;
  int64_t base = 0;                                   // tiles before sequence b0
  for (int b0 = 0; b0 < cv.B && base < t1; b0 += 32) {
    const int b = b0 + lane;
    const int m_b = b < cv.B ? cv.m_dev[b] : 0;
    const int th = (m_b + BN - 1) / BN + rt;          // tiles per head
    const int64_t tb = b < cv.B ? (int64_t)Hkv * th : 0;
    int64_t inc = tb;                                  // inclusive scan
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t x = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += x;
    }
    const int64_t sb = base + inc - tb;               // first tile of sequence b
    int kv_lo = 0, kv_hi = -1;
    if (tb > 0 && sb < t1 && sb + tb > t0) {
      kv_lo = (int)(max(t0 - sb, (int64_t)0) / th);
      kv_hi = (int)min((int64_t)Hkv - 1, (t1 - 1 - sb) / th);
    }
    const int cnt = kv_hi - kv_lo + 1;
    int ex = cnt;                                      // exclusive scan of counts
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, ex, off);
      if (lane >= off) ex += x;
    }
    const int total = __shfl_sync(0xffffffffu, ex, 31);
    ex -= cnt;
    if (nseg + total > kMaxSeg) return -1;
    for (int kv = kv_lo; kv <= kv_hi; ++kv) {
      const int64_t hs = sb + (int64_t)kv * th;
      Seg& s = segs[nseg + ex + (kv - kv_lo)];
      s.bkv = b * Hkv + kv;
      s.np = (m_b + BN - 1) / BN;
      s.i0 = (int)max(t0 - hs, (int64_t)0);
      s.i1 = (int)min(t1 - hs, (int64_t)th);
      if (tot >= P) {
        // every CTA's range holds a tile: the head's CTAs are consecutive
        const int c0 = owner(hs, tot, P), c1 = owner(hs + th - 1, tot, P);
        s.slot = c - c0;
        s.nparts = c1 - c0 + 1;
      } else {
        // ranges of 0 or 1 tile: one partial per tile of the head
        s.slot = s.i0;
        s.nparts = th;
      }
      s.m_b = m_b;
    }
    nseg += total;
    base += __shfl_sync(0xffffffffu, inc, 31);
  }
  return nseg;
}

template <bool FUSED, int G, bool PREFETCH>
__global__ void __launch_bounds__(kThreads, 2)
decode_gqa_sk_kernel(const __grid_constant__ CUtensorMap tmK,
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
  Seg* segs = reinterpret_cast<Seg*>(smem + OFF_SEG);
  float* ml_m = reinterpret_cast<float*>(smem + OFF_ML);           // [2][NQ]
  float* ml_l = ml_m + 2 * NQ;                                     // [2][4][NQ]
  float* red_max = reinterpret_cast<float*>(smem + OFF_RED);       // [2][4][NQ]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  volatile int* never = reinterpret_cast<volatile int*>(smem + OFF_MISC + 8);
  int* s_nseg = reinterpret_cast<int*>(smem + OFF_MISC + 12);
  int* s_last = reinterpret_cast<int*>(smem + OFF_MISC + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int per_kv = cv.H / cv.Hkv;                 // query heads per KV head (<= G)
  const int64_t n = cv.n;

  if (tid == 0) {
    for (int k = 0; k < NBAR; ++k) {
      const bool cnt128 = (k >= B_SFREE && k < B_PFREE) || (k >= B_OFREE && k < B_FIN) ||
                          k == B_QFULL;
      mbar_init(bar(k), cnt128 ? 128u : 1u);
    }
    *abort_flag = 0;
    *never = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tmem_relinquish();
  }
  for (uint32_t i = tid; i < NS * kTileB / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + OFF_RING)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Segment table: from m_b, before the dependency wait when the preceding
  // kernel of the stream writes no m_b of this cache.
  auto build = [&]() {
    if (warp == 0) {
      const int ns = build_segments(cv, blockIdx.x, gridDim.x, segs, lane);
      if (lane == 0) {
        *s_nseg = ns < 0 ? 0 : ns;
        if (ns < 0) flag_error(cv.err, kErrLaunchShape);
      }
    }
    __syncthreads();
  };
  if (PREFETCH) build();
  const int nseg_pre = PREFETCH ? *s_nseg : 0;

  // Producer state: loads are numbered idx = 2 j (+ 1 for V) over the CTA's
  // tiles j; walk (segment, tile) in order.
  int p_seg = 0, p_i = 0, p_idx = 0;
  auto p_valid = [&]() { return p_seg < *s_nseg; };
  auto p_advance = [&]() {
    if (p_idx & 1) {
      if (++p_i >= segs[p_seg].i1) {
        ++p_seg;
        if (p_seg < *s_nseg) p_i = segs[p_seg].i0;
      }
    }
    ++p_idx;
  };
  // Issues load p_idx (K or V of tile p_i of segment p_seg): whole tiles,
  // except a head's last prefix tile and its ring tiles, fetched as 8-row
  // boxes up to the last row that holds a key (at least one box).
  const uint64_t kpol = stream_policy();
  auto p_issue = [&](int64_t filled) {
    const Seg& sg = segs[p_seg];
    const int s = p_idx % NS;
    const bool isv = p_idx & 1;
    const bool ring = p_i >= sg.np;
    const int64_t row0 = (int64_t)sg.bkv * cv.slab_rows +
                         (ring ? cv.m_cap + (int64_t)(p_i - sg.np) * BN : (int64_t)p_i * BN);
    int rows = BN;
    if (ring) {
      const int64_t v = filled - (int64_t)(p_i - sg.np) * BN;
      rows = (int)max((int64_t)8, min((int64_t)BN, (v + 7) & ~(int64_t)7));
    } else if (p_i == sg.np - 1) {
      rows = (int)((sg.m_b - (int64_t)p_i * BN + 7) & ~7);
    }
    const uint32_t dst = sb + OFF_RING + s * kTileB;
    const int y = (int)row0;
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
  if (PREFETCH && warp == kProducerWarp && lane == 0 && nseg_pre > 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    p_i = segs[0].i0;
    // Loads of prefix tiles into free slots: their rows are fixed until the
    // next prefill.
    while (p_valid() && p_idx < NS && p_i < segs[p_seg].np) {
      p_issue(0);
      p_advance();
    }
  }
  griddep_wait();
  // The next launch's CTAs may take SM slots as this grid's CTAs finish;
  // they wait for this grid.
  griddep_launch_dependents();
  if (!PREFETCH) build();
  const int nseg = *s_nseg;
  const float scale = rsqrtf((float)HD) * kLog2e;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nseg > 0) {
      if (!PREFETCH) p_i = segs[0].i0;
      auto t_b_of = [&](const Seg& sg) {
        return cv.t_dev[(size_t)(sg.bkv / cv.Hkv) * cv.H + (size_t)(sg.bkv % cv.Hkv) * per_kv];
      };
      // The new key and value of a head whose ring tile holding slot w is in
      // this CTA's range go to that slot before any TMA read of the tile (no
      // other CTA reads the head's ring tiles).
      auto append = [&](const Seg& sg, int64_t t_b) {
        const int64_t w = t_b % n;
        const int wt = sg.np + (int)(w / BN);
        if (wt < sg.i0 || wt >= sg.i1) return;
        const int64_t row = (int64_t)sg.bkv * cv.slab_rows + cv.m_cap + w;
        uint4* dk = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(cv.K) + row * HD);
        uint4* dv = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(cv.V) + row * HD);
        const uint4* sk = reinterpret_cast<const uint4*>(knew + (size_t)sg.bkv * HD);
        const uint4* sv = reinterpret_cast<const uint4*>(vnew + (size_t)sg.bkv * HD);
#pragma unroll 4
        for (int i = 0; i < HD * 2 / 16; ++i) {
          dk[i] = sk[i];
          dv[i] = sv[i];
        }
        fence_proxy_async_global();
      };
      int64_t filled = 0;
      int f_seg = -1;
      while (p_valid()) {
        if (f_seg != p_seg) {
          f_seg = p_seg;
          const int64_t t_b = t_b_of(segs[p_seg]);
          filled = FUSED ? min(n, t_b + 1) : min(n, t_b);
          if (FUSED) append(segs[p_seg], t_b);
        }
        if (p_idx >= NS && !mbar_wait(bar(B_EMPTY + p_idx % NS), ((p_idx / NS) - 1) & 1,
                                      abort_flag, wait_ns))
          break;
        p_issue(filled);
        p_advance();
      }
      // A wait that gave up: the segments never reached still get the
      // step's key and value, so the ring holds what t_b will name.
      if (FUSED)
        for (int s = f_seg + 1; s < nseg; ++s) append(segs[s], t_b_of(segs[s]));
      // Drain: every copy issued has landed before the CTA may exit.
      for (int k = max(0, p_idx - NS); k < p_idx; ++k)
        mbar_wait(bar(B_FULL + k % NS), (k / NS) & 1, never, kWaitLimitNs);
    } else if (PREFETCH && lane == 0) {
      for (int k = 0; k < p_idx; ++k)
        mbar_wait(bar(B_FULL + k % NS), (k / NS) & 1, never, kWaitLimitNs);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nseg > 0) {
      constexpr uint32_t idesc_s = idesc_bf16_ab(BN, NQ, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_ab(HD, NQ, true, false);
      auto full = [&](int idx) {
        return mbar_wait(bar(B_FULL + idx % NS), (idx / NS) & 1, abort_flag, wait_ns);
      };
      auto issue_s = [&](int j, bool last) {
        const uint32_t kb = sb + OFF_RING + ((2 * j) % NS) * kTileB;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k)
          mma_bf16_ss(tmem + TM_S + 16 * (j & 1),
                      desc_sw128(kb + (k >> 2) * kSub + (k & 3) * 32, 16, 1024),
                      desc_sw128(sb + OFF_Q + (k >> 2) * kNAtom + (k & 3) * 32, 16, 1024),
                      idesc_s, k > 0);
        mma_commit(bar(B_S + (j & 1)));
        mma_commit(bar(B_EMPTY + (2 * j) % NS));
        if (last) mma_commit(bar(B_QFREE));
      };
      // PV(j) of segment s into O^T buffer s & 1; the segment's first PV
      // overwrites it (after the epilogue read out segment s - 2).
      auto issue_pv = [&](int j, int s, bool first, bool last) {
        if (!mbar_wait(bar(B_P + (j & 1)), (j >> 1) & 1, abort_flag, wait_ns) ||
            !full(2 * j + 1))
          return false;
        if (first && s >= 2 &&
            !mbar_wait(bar(B_OFREE + (s & 1)), ((s >> 1) - 1) & 1, abort_flag, wait_ns))
          return false;
        tc_fence_after();
        const uint32_t vb = sb + OFF_RING + ((2 * j + 1) % NS) * kTileB;
        const uint32_t pb = sb + OFF_P + (j & 1) * 2 * kNAtom;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          mma_bf16_ss(tmem + TM_O + 16 * (s & 1), desc_sw128(vb + k * 2048, kSub, 1024),
                      desc_sw128(pb + (k >> 2) * kNAtom + (k & 3) * 32, 16, 1024),
                      idesc_o, (!first || k > 0) ? 1u : 0u);
        mma_commit(bar(B_PFREE + (j & 1)));
        mma_commit(bar(B_EMPTY + (2 * j + 1) % NS));
        if (last) mma_commit(bar(B_OREADY + (s & 1)));
        return true;
      };
      bool ok = true;
      int j = 0;
      int ps = -1;                                   // previous tile's segment
      bool pfirst = false, plast = false;
      for (int s = 0; ok && s < nseg; ++s) {
        const int i0 = segs[s].i0, i1 = segs[s].i1;
        for (int i = i0; i < i1; ++i, ++j) {
          const bool first = i == i0, last = i == i1 - 1;
          // At a segment boundary the old segment's last PV goes first.
          if (first && j >= 1 && !(ok = issue_pv(j - 1, ps, pfirst, plast))) break;
          ok = (!first || mbar_wait(bar(B_QFULL), s & 1, abort_flag, wait_ns)) &&
               full(2 * j) &&
               (j < 2 || mbar_wait(bar(B_SFREE + (j & 1)), ((j - 2) >> 1) & 1,
                                   abort_flag, wait_ns));
          if (!ok) break;
          tc_fence_after();
          issue_s(j, last);
          if (!first && !(ok = issue_pv(j - 1, ps, pfirst, plast))) break;
          ps = s;
          pfirst = first;
          plast = last;
        }
      }
      if (ok && j >= 1) issue_pv(j - 1, ps, pfirst, plast);
      // Arrives once every MMA issued above has completed.
      mma_commit(bar(B_FIN));
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ softmax
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    auto wait_all = [&](int k, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar(k), parity, abort_flag, wait_ns));
    };
    int n_sync = 0;
    auto soft_sync = [&]() {
      mbar_arrive(bar(B_SYNCS));
      const bool r = mbar_wait(bar(B_SYNCS), n_sync & 1, abort_flag, wait_ns);
      ++n_sync;
      return __all_sync(0xffffffffu, r);
    };
    bool ok = true;
    int j = 0;
    for (int s = 0; ok && s < nseg; ++s) {
      const Seg sg = segs[s];
      const size_t bh0 = (size_t)(sg.bkv / cv.Hkv) * cv.H + (size_t)(sg.bkv % cv.Hkv) * per_kv;
      const int64_t t_b = cv.t_dev[bh0];
      const int64_t filled = FUSED ? min(n, t_b + 1) : min(n, t_b);
      float m_ref[G], l_t[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m_ref[g] = -INFINITY;
        l_t[g] = 0.f;
      }
      for (int i = sg.i0; i < sg.i1; ++i, ++j) {
        if (!wait_all(B_S + (j & 1), (j >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t r[16];
        tmem_ld16(tmem + lane_off + TM_S + 16 * (j & 1), r);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(B_SFREE + (j & 1)));
        const bool valid = i < sg.np ? (int64_t)i * BN + tid < sg.m_b
                                     : (int64_t)(i - sg.np) * BN + tid < filled;
        float sc[G];
#pragma unroll
        for (int g = 0; g < G; ++g)
          sc[g] = (valid && g < per_kv) ? __uint_as_float(r[g]) * scale : -INFINITY;
        float* rm = red_max + (j & 1) * 4 * NQ;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float v = warp_max(sc[g]);
          if (lane == 0) rm[warp * NQ + g] = v;
        }
        if (!soft_sync()) {
          ok = false;
          break;
        }
        bool grow = false;
        float mt[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          mt[g] = fmaxf(fmaxf(rm[g], rm[NQ + g]), fmaxf(rm[2 * NQ + g], rm[3 * NQ + g]));
          grow |= mt[g] > m_ref[g] + kRescaleThreshold ||
                  (m_ref[g] == -INFINITY && mt[g] > -INFINITY);
        }
        if (grow) {
          float alpha[G];
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float mn = fmaxf(m_ref[g], mt[g]);
            alpha[g] = (mn == -INFINITY) ? 1.f : fast_exp2(m_ref[g] - mn);
            m_ref[g] = mn;
            l_t[g] *= alpha[g];
          }
          if (i > sg.i0) {
            // O^T holds PV of this segment's earlier tiles: rescale it once
            // PV(j - 1) has completed.
            if (!wait_all(B_PFREE + ((j - 1) & 1), ((j - 1) >> 1) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            uint32_t ov[16];
            tmem_ld16(tmem + lane_off + TM_O + 16 * (s & 1), ov);
            tmem_wait_ld();
#pragma unroll
            for (int g = 0; g < G; ++g)
              ov[g] = __float_as_uint(__uint_as_float(ov[g]) * alpha[g]);
            tmem_st16(tmem + lane_off + TM_O + 16 * (s & 1), ov);
            tmem_wait_st();
          }
        }
        // P^T(j): buffer j & 1 is free once PV(j - 2) has completed.
        if (j >= 2 && !wait_all(B_PFREE + (j & 1), ((j - 2) >> 1) & 1)) {
          ok = false;
          break;
        }
        uint8_t* pbuf = smem + OFF_P + (j & 1) * 2 * kNAtom;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float ref = (m_ref[g] == -INFINITY) ? 0.f : m_ref[g];
          const float p = fast_exp2(sc[g] - ref);
          l_t[g] += p;
          if (g < per_kv)
            *reinterpret_cast<__nv_bfloat16*>(pbuf + sw128_off(g, tid, kNAtom)) =
                __float2bfloat16(p);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(B_P + (j & 1)));
      }
      if (!ok) break;
      // The segment's reference maxima and per-warp sums for the epilogue.
      if (s >= 2 && !wait_all(B_MLFREE + (s & 1), ((s >> 1) - 1) & 1)) break;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float v = l_t[g];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) ml_l[((s & 1) * 4 + warp) * NQ + g] = v;
        if (tid == 0) ml_m[(s & 1) * NQ + g] = m_ref[g];
      }
      mbar_arrive(bar(B_ML + (s & 1)));
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = tid - kEpiWarp0 * 32;               // row d of O^T
    const int ew = warp - kEpiWarp0;                  // TMEM lane quarter
    const uint32_t lane_off = (uint32_t)(ew * 32) << 16;
    auto wait_all = [&](int k, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar(k), parity, abort_flag, wait_ns));
    };
    int n_sync = 0;
    auto epi_sync = [&]() {
      mbar_arrive(bar(B_SYNCE));
      const bool r = mbar_wait(bar(B_SYNCE), n_sync & 1, abort_flag, wait_ns);
      ++n_sync;
      return __all_sync(0xffffffffu, r);
    };
    auto head0 = [&](const Seg& sg) {
      return (size_t)(sg.bkv / cv.Hkv) * cv.H + (size_t)(sg.bkv % cv.Hkv) * per_kv;
    };
    // Q^T of segment s as the S MMA's B operand: row g = query head g,
    // K-major over d (column e).
    __nv_bfloat16 qv[G];
    auto load_q = [&](int s) {
      const size_t bq = head0(segs[s]);
#pragma unroll
      for (int g = 0; g < G; ++g)
        qv[g] = g < per_kv ? q[(bq + g) * HD + e] : __float2bfloat16(0.f);
    };
    auto stage_q = [&]() {
#pragma unroll
      for (int g = 0; g < NQ; ++g)
        *reinterpret_cast<__nv_bfloat16*>(smem + OFF_Q + sw128_off(g, e, kNAtom)) =
            g < G ? qv[g < G ? g : 0] : __float2bfloat16(0.f);
      fence_proxy_async_smem();
      mbar_arrive(bar(B_QFULL));
    };
    bool ok = true;
    if (nseg > 0) {
      load_q(0);
      stage_q();
      if (nseg > 1) load_q(1);
    }
    for (int s = 0; ok && s < nseg; ++s) {
      const Seg sg = segs[s];
      const size_t bh0 = head0(sg);
      const int64_t t_b = cv.t_dev[bh0];
      if (s + 1 < nseg) {
        // Q^T is free once segment s's last S MMA has completed.
        if (!wait_all(B_QFREE, s & 1)) {
          ok = false;
          break;
        }
        stage_q();
        if (s + 2 < nseg) load_q(s + 2);
      }
      if (!wait_all(B_OREADY + (s & 1), (s >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t ov[16];
      tmem_ld16(tmem + lane_off + TM_O + 16 * (s & 1), ov);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(B_OFREE + (s & 1)));
      if (!wait_all(B_ML + (s & 1), (s >> 1) & 1)) {
        ok = false;
        break;
      }
      float mg[G], lg[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        mg[g] = ml_m[(s & 1) * NQ + g];
        const float* lw = ml_l + (s & 1) * 4 * NQ;
        lg[g] = lw[g] + lw[NQ + g] + lw[2 * NQ + g] + lw[3 * NQ + g];
      }
      mbar_arrive(bar(B_MLFREE + (s & 1)));
      if (sg.nparts == 1) {
        // The whole head in this CTA: no partials.
#pragma unroll
        for (int g = 0; g < G; ++g) {
          if (g >= per_kv) break;
          o[(bh0 + g) * HD + e] =
              __float2bfloat16(lg[g] > 0.f ? __uint_as_float(ov[g]) / lg[g] : 0.f);
          if (e == 0) {
            if (lse) lse[bh0 + g] = lg[g] > 0.f ? (mg[g] + log2f(lg[g])) * kLn2 : -INFINITY;
            if (FUSED) cv.t_dev[bh0 + g] = t_b + 1;
          }
        }
        continue;
      }
      const size_t stride = (size_t)cv.part_slots * (HD + 2);
      const uint64_t pol = partial_policy();
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (g >= per_kv) break;
        float* P = cv.part + (bh0 + g) * stride + (size_t)sg.slot * (HD + 2);
        st_hint(P + 2 + e, __uint_as_float(ov[g]), pol);
        if (e == 0) {
          st_hint(P, mg[g], pol);
          st_hint(P + 1, lg[g], pol);
        }
      }
      if (!epi_sync()) {
        ok = false;
        break;
      }
      if (e == 0) *s_last = arrive_acq_rel(&cv.cnt_bh[bh0]) == sg.nparts - 1;
      if (!epi_sync()) {
        ok = false;
        break;
      }
      const bool merged = *s_last;
      if (merged) {
        float M[G], L[G], A[G];
        merge_partials<G, (G <= 2 ? 2 : 1)>(cv.part + bh0 * stride, stride, sg.nparts, HD,
                                            e, per_kv, M, L, A);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          if (g >= per_kv) break;
          o[(bh0 + g) * HD + e] = __float2bfloat16(L[g] > 0.f ? A[g] / L[g] : 0.f);
          if (e == 0) {
            if (lse) lse[bh0 + g] = L[g] > 0.f ? (M[g] + log2f(L[g])) * kLn2 : -INFINITY;
            // Every CTA of this KV head read t_b before its own arrival.
            if (FUSED) cv.t_dev[bh0 + g] = t_b + 1;
          }
        }
        if (e == 0) cv.cnt_bh[bh0] = 0;
      }
      // s_last is read again only after the next arrival's barrier.
      if (!epi_sync()) {
        ok = false;
        break;
      }
      if (merged)
        for (int g = 0; g < per_kv; ++g) {
          const float* P0 = cv.part + (bh0 + g) * stride;
          discard_l2_inside(P0, P0 + (size_t)sg.nparts * (HD + 2), e, 128);
        }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    // Every MMA this CTA issued has completed before TMEM is released.
    if (lane == 0 && nseg > 0) mbar_wait(bar(B_FIN), 0, never, kWaitLimitNs);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TM_COLS);
  }
  if (tid == 0 && *abort_flag) flag_error(cv.err, kErrWaitTimeout);
}

// Persistent CTAs: RSWA_SK_GRID_PCT percent of two per SM; 95 measured best on
// GB300, batched GQA step (53.6-53.9 us; 100: 54.5, 90: 54.9, 80: 57.8):
// a few free slots let the next launch's CTAs become resident and request
// their first tiles while this launch's last CTAs finish.
#ifndef RSWA_SK_GRID_PCT
#define RSWA_SK_GRID_PCT 95
#endif
int sk_grid(const CacheView& cv) {
  return std::max(1, (int)((int64_t)2 * cv.sms * RSWA_SK_GRID_PCT / 100));
}

template <bool FUSED, int G, bool PREFETCH>
cudaError_t launch_sk(const CacheView& cv, const CUtensorMap* m, const void* q,
                      const void* k, const void* v, void* o, float* lse, cudaStream_t s) {
  auto kern = decode_gqa_sk_kernel<FUSED, G, PREFETCH>;
  // Per device (the attribute belongs to the current device's context).
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sk_grid(cv));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  using BF = __nv_bfloat16;
  return cudaLaunchKernelEx(&cfg, kern, m[0], m[1], m[2], m[3], cv, (const BF*)q,
                            (const BF*)(FUSED ? k : nullptr),
                            (const BF*)(FUSED ? v : nullptr), (BF*)o, lse,
                            phase_wait_limit_ns());
}

template <bool FUSED, bool PREFETCH>
cudaError_t launch_sk_g(const CacheView& cv, const CUtensorMap* m, const void* q,
                        const void* k, const void* v, void* o, float* lse,
                        cudaStream_t s) {
  const int per_kv = cv.H / cv.Hkv;
  if (per_kv <= 2) return launch_sk<FUSED, 2, PREFETCH>(cv, m, q, k, v, o, lse, s);
  if (per_kv <= 4) return launch_sk<FUSED, 4, PREFETCH>(cv, m, q, k, v, o, lse, s);
  if (per_kv <= 8) return launch_sk<FUSED, 8, PREFETCH>(cv, m, q, k, v, o, lse, s);
  return launch_sk<FUSED, 16, PREFETCH>(cv, m, q, k, v, o, lse, s);
}

}  // namespace

// The stream-K form when its segment table fits: sequences for one warp to
// scan (B <= 256), ranges of at most kMaxSeg - 2 tiles on the largest cache,
// and partial slots for a head shared by every CTA that may touch it (at
// most one per tile of the head's list).
bool gqa_sk_supported(const CacheView& cv) {
  // up to 8 query heads per KV head (16 would spill at two CTAs per SM)
  if (!gqa_tc_supported(cv) || cv.H / cv.Hkv > 8 || cv.B > 256 || cv.sms < 1)
    return false;
  const int64_t th = (cv.m_cap + BN - 1) / BN + (cv.n + BN - 1) / BN;
  const int64_t tot = (int64_t)cv.B * cv.Hkv * th;
  const int64_t P = sk_grid(cv);
  return (tot + P - 1) / P + 2 <= kMaxSeg && th + 1 <= cv.part_slots;
}

cudaError_t launch_decode_gqa_sk(const CacheView& cv, const void* q, const void* k,
                                 const void* v, void* o, float* lse, bool fused,
                                 bool prefetch_prefix, cudaStream_t s) {
  const uint64_t rows = (uint64_t)cv.B * cv.Hkv * cv.slab_rows;
  CUtensorMap m[4];                                 // K, V; K, V in 8-row boxes
  if (!make_tmap_rows_bf16(&m[0], cv.K, HD, rows) ||
      !make_tmap_rows_bf16(&m[1], cv.V, HD, rows) ||
      !make_tmap_rows_bf16(&m[2], cv.K, HD, rows, 8) ||
      !make_tmap_rows_bf16(&m[3], cv.V, HD, rows, 8))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if (prefetch_prefix)
    e = fused ? launch_sk_g<true, true>(cv, m, q, k, v, o, lse, s)
              : launch_sk_g<false, true>(cv, m, q, k, v, o, lse, s);
  else
    e = fused ? launch_sk_g<true, false>(cv, m, q, k, v, o, lse, s)
              : launch_sk_g<false, false>(cv, m, q, k, v, o, lse, s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace rswa
