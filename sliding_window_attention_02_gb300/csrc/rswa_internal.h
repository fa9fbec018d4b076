// Internal declarations shared by the host API and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/rswa.h"

namespace rswa {

constexpr int kMaxSeqPerLaunch = 128;   // sequences per prefill launch
constexpr int kDecodeThreads = 128;     // threads per grouped split-K decode CTA

// Device view of a cache buffer.  All regions live in the caller's buffer.
// H query heads share Hkv key/value heads (H % Hkv == 0): query head h reads
// KV head h / (H / Hkv); Hkv == H is standard multi-head attention.
//   K, V    slabs [B][Hkv][slab_rows][d], slab_rows = m_cap + n: rows
//           0..m_cap-1 are the prefix region, rows m_cap..m_cap+n-1 the ring.
//   m_dev   int32 [B]     prefix length m_b
//   t_dev   int64 [B][H]  outputs appended t_b, one copy per head so that a
//                         fused decode step advances each head's copy
//                         without cross-head synchronisation; all copies
//                         of a sequence are equal between calls
//   err     int32 [1]     first device-side error code (0 = none)
//   part    float [B][H][max_chunks][d + 2]  split-K partials (m, l, acc);
//           the region is sized for the smallest chunk, so it may be larger
//   cnt_bh  int32 [B][H]  CTAs of (b, h) that have published a partial
struct CacheView {
  void* K;
  void* V;
  int32_t* m_dev;
  int64_t* t_dev;
  int32_t* err;
  float* part;
  int32_t* cnt_bh;
  int B, H, Hkv, d, dtype;
  int64_t m_cap, n, slab_rows;
  int chunk;       // keys per decode CTA
  int max_chunks;  // ceil(m_cap / chunk) + ceil(n / chunk)
  int sms;         // streaming multiprocessors of the cache's device
  int part_slots;  // partial slots per (b, h) in `part` (>= max_chunks)
};

// Per-launch sequence table for prefill (passed by value as a kernel param).
struct SeqTable {
  int nseq;                              // sequences in this launch
  int seq0;                              // index of the first one
  int64_t T[kMaxSeqPerLaunch];           // outputs per sequence
  int64_t row_off[kMaxSeqPerLaunch];     // first row of each sequence
  int32_t m[kMaxSeqPerLaunch];           // prefix lengths
  int32_t tile_off[kMaxSeqPerLaunch + 1];// cumulative 128-row q-tiles
};

// Bound on the pipelined kernels' waits for a pipeline phase (tensor-core
// prefill, block, grouped decode; streaming decode): 1 s, or what
// rswa_debug_set_wait_limit_ns set (test hook).
uint64_t phase_wait_limit_ns();

// ---- launchers (each returns the cudaError_t of its launch) ----
cudaError_t launch_prefill_cache(const CacheView& cv, const SeqTable& st,
                                 const void* K, const void* V, int64_t max_rows,
                                 cudaStream_t s);
cudaError_t launch_append(const CacheView& cv, const void* k, const void* v,
                          cudaStream_t s);
cudaError_t launch_set_t(const CacheView& cv, const int64_t* t_host,
                         cudaStream_t s);
bool decode_use_small(const CacheView& cv);
// Few heads with long caches (decode_stream.cu): S CTAs per head stream the
// head's keys through shared memory; S <= part_slots.
bool decode_use_stream(const CacheView& cv);
int decode_stream_splits(const CacheView& cv);
cudaError_t launch_decode_stream(const CacheView& cv, const void* q,
                                 const void* k, const void* v, void* o,
                                 float* lse, bool fused, bool prefetch_prefix,
                                 cudaStream_t s);
// Partial slots per (b, h) the decode path chosen for this view uses.
int decode_part_slots(const CacheView& cv);
// Grouped split-K decode (decode_gqa.cu): used for grouped caches whose query
// heads per KV head are a multiple of 2 when the cluster path is not taken.
// Query heads one CTA serves (4, 2, or 1 = not grouped); the chunk heuristic
// counts the K/V streams this leaves, H / heads_per_cta per sequence.
inline int gqa_heads_per_cta(int heads, int kv_heads) {
  const int per_kv = heads / kv_heads;
  if (per_kv % 4 == 0) return 4;
  if (per_kv % 2 == 0) return 2;
  return 1;
}
int decode_gqa_heads_per_cta(const CacheView& cv);
// Grouped decode on the tensor cores (decode_gqa_tc.cu): bf16, d 128, 2..16
// query heads per KV head; one CTA serves every query head of its KV head.
inline bool gqa_tc_shape(int heads, int kv_heads, int head_dim, int dtype) {
  const int per_kv = heads / kv_heads;
  return dtype == RSWA_BF16 && head_dim == 128 && per_kv >= 2 && per_kv <= 16;
}
bool gqa_tc_supported(const CacheView& cv);
// Stream-K form of the grouped tensor-core decode (decode_gqa_sk.cu):
// persistent CTAs split the key tiles of all KV heads evenly.
bool gqa_sk_supported(const CacheView& cv);
cudaError_t launch_decode_gqa_sk(const CacheView& cv, const void* q, const void* k,
                                 const void* v, void* o, float* lse, bool fused,
                                 bool prefetch_prefix, cudaStream_t s);
// prefetch_prefix: the stream's preceding kernel writes no prefix row of
// this cache (the first K/V tiles of prefix chunks load before its end).
cudaError_t launch_decode_gqa_tc(const CacheView& cv, const void* q,
                                 const void* k, const void* v, void* o,
                                 float* lse, bool fused, bool prefetch_prefix,
                                 cudaStream_t s);
// [rows][cols] bf16, row-major, as a 2-D TMA map: box 64 columns x box_rows
// rows, 128-byte swizzle; rows past `rows` read as zero.
bool make_tmap_rows_bf16(CUtensorMap* map, const void* base, uint64_t cols,
                         uint64_t rows, uint32_t box_rows = 128);
cudaError_t launch_decode_gqa(const CacheView& cv, const void* q, const void* k,
                              const void* v, void* o, float* lse, bool fused,
                              cudaStream_t s);
// prefetch: the preceding kernel of the stream writes no prefix row and no
// m_b of this cache (the kernels may read them before the dependency wait).
cudaError_t launch_decode_block(const CacheView& cv, const void* q, const void* k,
                                const void* v, int64_t block, void* o, float* lse,
                                bool prefetch, cudaStream_t s);
// Blocks of at least kBlockTcMin tokens of a bf16, head_dim 128 cache run
// their attention on the tensor cores (block_tc.cu); smaller blocks, and
// other caches, one CTA per query on the CUDA cores (decode_block.cu), which
// measured faster below 64 tokens on GB300 (single-page cache, 16 / 32
// tokens: 10.2 / 15.5 against 16.5 / 16.8 us).
constexpr int64_t kBlockTcMin = 64;
bool block_tc_supported(const CacheView& cv, int64_t block);
cudaError_t launch_block_tc(const CacheView& cv, const void* q, const void* k,
                            const void* v, int64_t block, void* o, float* lse,
                            cudaStream_t s);
// prefetch_prefix: the preceding kernel of the stream writes no prefix row
// and no m_b of this cache (every decode launch but the first after a
// prefill); the cluster path then loads them before its dependency wait.
cudaError_t launch_decode(const CacheView& cv, const void* q, const void* k,
                          const void* v, void* o, float* lse, bool fused,
                          bool prefetch_prefix, cudaStream_t s);
cudaError_t launch_prefill_rowwise(const CacheView& cv, const SeqTable& st,
                                   const void* Q, const void* K, const void* V,
                                   void* O, int64_t total_rows, cudaStream_t s);
// tcgen05 prefill (bf16, head_dim 128).  Returns cudaErrorNotSupported when
// the shape is outside what the kernel handles.
cudaError_t launch_prefill_tc(const CacheView& cv, const SeqTable& st,
                              const void* Q, const void* K, const void* V,
                              void* O, int64_t total_rows, cudaStream_t s);
bool prefill_tc_supported(const CacheView& cv);

// Fused decode step with split-K scratch in the library's static device array
// (decode_static.cu).  Fails with cudaErrorInvalidValue when the cache needs
// more than static_scratch_capacity() bytes of scratch.
size_t static_scratch_need(const CacheView& cv, size_t* part_bytes,
                           size_t* cnt_bytes);
size_t static_scratch_capacity();
cudaError_t launch_decode_fused_static(const CacheView& cv, int dev,
                                       const void* q, const void* k,
                                       const void* v, void* o, float* lse,
                                       bool prefetch_prefix, cudaStream_t s);

}  // namespace rswa
