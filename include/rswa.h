/*
 * rswa.h - C ABI of the R-SWA (Reference Sliding Window Attention) library
 * for GB300 (sm_103a).
 *
 * The method.  Every output token attends to the whole fixed reference prefix
 * P of length m (visual tokens plus prompt, always visible) and to the last n
 * output tokens, itself included (a causal sliding window; n = 128 by
 * default).  The KV cache is therefore bounded: after T outputs it holds
 * C(T) = m + min(n, T) <= m + n tokens, a queue of capacity m + n in which
 * each new output evicts the oldest output, the (m+1)-th entry.
 *   - "Unlimited-OCR deep dive" (ai-news-5min-kr): R-SWA pseudo-code block
 *     N(t) = P U D_n(t) and C_R-SWA(T) = L_m + min(n, T); data-flow steps 2-4.
 *   - "Unlimited OCR - Baidu's one-shot long-document parsing model"
 *     (GeekNews): sections "Reference Sliding Window Attention (R-SWA)",
 *     "KV cache management" and "Model architecture".
 * Readings where the pages are silent: prefix rows attend causally among
 * themselves; the window of n includes the current token; the softmax scale
 * is 1/sqrt(head_dim); positions are applied by the caller (RoPE etc. before
 * Q/K reach this library); one KV head per query head (standard MHA, the
 * pages' baseline) unless the cache is created by rswa_cache_create_gqa,
 * which lets several query heads share one KV head.
 *
 * Conventions shared by every call.
 *   - All device pointers are plain CUDA device addresses owned by the
 *     caller.  The library allocates no device memory: the cache lives in a
 *     caller-provided buffer of rswa_cache_footprint() bytes.
 *   - dtype is RSWA_F32 (float) or RSWA_BF16 (bfloat16) and applies to every
 *     Q/K/V/O tensor of a cache; arithmetic is float32 in both cases.
 *   - Token-major tensors: a "[rows][H][d]" tensor is contiguous with d
 *     fastest.  Per-step tensors q, k, v, o are "[B][H][d]".
 *   - Work is enqueued on the caller's stream (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream) and returns immediately.
 *     Arguments are validated on the host before anything is launched; an
 *     invalid call launches nothing and changes no state.
 *   - Every call returns an rswa_status.  RSWA_ECUDA reports a CUDA error
 *     from a launch or copy; errors raised inside kernels (a bounded wait
 *     that ran out) set a device flag that rswa_sync_status() returns.
 *   - Calls on one cache must be ordered (same stream, or the caller orders
 *     the streams); the cache state (m_b, t_b) is kept on the device and is
 *     read and advanced by the kernels, so a captured CUDA graph replays
 *     correctly.
 */
#ifndef RSWA_H
#define RSWA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define RSWA_API __attribute__((visibility("default")))
#else
#define RSWA_API
#endif

/* Opaque host handle.  Holds the layout of the caller's device buffer. */
typedef struct rswa_cache rswa_cache;

enum rswa_status {
  RSWA_OK = 0,
  RSWA_EINVAL = 1,    /* bad argument: null pointer, size or shape */
  RSWA_ECAPACITY = 2, /* a prefix longer than the cache's prefix capacity,
                         or a buffer smaller than the footprint */
  RSWA_EDTYPE = 3,    /* unsupported dtype / head_dim combination */
  RSWA_EHANDLE = 4,   /* NULL, destroyed or foreign handle */
  RSWA_ECUDA = 5,     /* a CUDA runtime call or launch failed */
  RSWA_EDEVICE = 6    /* a kernel flagged an error (bounded wait ran out, or a
                        launch shape that does not cover its work) */
};

enum rswa_dtype { RSWA_F32 = 0, RSWA_BF16 = 1 };

/* Static message for a status code; never NULL. */
RSWA_API const char* rswa_strerror(int status);

/*
 * Bytes of device memory a cache needs (written to *out_bytes).
 *   m         prefix capacity per sequence (>= 0): the largest m_b a prefill
 *             may store ("the prefix window m is fixed per inference",
 *             GeekNews, R-SWA section).
 *   n         output window (>= 1); the ring holds n output tokens.
 *   heads     H >= 1, head_dim in {64, 128}, batch B >= 1.
 * The footprint covers the prefix region K,V [B][H][m][d], the ring
 * K,V [B][H][n][d], the per-sequence state (m_b, t_b) and the decode
 * split-K scratch.  Errors: RSWA_EINVAL, RSWA_EDTYPE.
 */
RSWA_API int rswa_cache_footprint(int64_t m, int64_t n, int heads,
                                  int head_dim, int batch, int dtype,
                                  size_t* out_bytes);

/*
 * Create a cache over the caller's device buffer (>= footprint bytes,
 * 256-byte aligned).  The buffer stays owned by the caller and must outlive
 * the handle.  Creation zeroes the per-sequence state (every sequence empty:
 * m_b = t_b = 0) and the key/value slabs with a synchronous memset on the
 * current device.
 * Errors: RSWA_EINVAL (null/misaligned buffer, bad sizes), RSWA_ECAPACITY
 * (buffer too small), RSWA_EDTYPE, RSWA_ECUDA.
 */
RSWA_API int rswa_cache_create(int64_t m, int64_t n, int heads, int head_dim,
                               int batch, int dtype, void* device_buf,
                               size_t buf_bytes, rswa_cache** out);

/*
 * Grouped-query variants (not on the pages, which name standard MHA as the
 * baseline): `heads` query heads share `kv_heads` key/value heads
 * (heads % kv_heads == 0); query head h reads KV head h / (heads / kv_heads).
 * The cache then stores kv_heads slabs, and every K/V tensor of the other
 * calls has kv_heads heads ([rows][kv_heads][d], [B][kv_heads][d]) while
 * Q, O, q, o, lse keep `heads`.  kv_heads == heads is exactly
 * rswa_cache_footprint / rswa_cache_create.  Errors as theirs, plus
 * RSWA_EINVAL when kv_heads does not divide heads.
 */
RSWA_API int rswa_cache_footprint_gqa(int64_t m, int64_t n, int heads,
                                      int kv_heads, int head_dim, int batch,
                                      int dtype, size_t* out_bytes);
RSWA_API int rswa_cache_create_gqa(int64_t m, int64_t n, int heads,
                                   int kv_heads, int head_dim, int batch,
                                   int dtype, void* device_buf,
                                   size_t buf_bytes, rswa_cache** out);

/* Free the host handle (not the device buffer).  Later use of the handle
 * returns RSWA_EHANDLE. */
RSWA_API int rswa_cache_destroy(rswa_cache* cache);

/*
 * Prefill: store every sequence's prefix and its last min(n, T) outputs in the
 * cache, then (if O != NULL) compute R-SWA attention for every row.
 *   Q, K, V   token-major packed rows [sum_b (m_b + T)][H][d]; sequence b
 *             occupies rows off_b .. off_b + m_b + T - 1 with
 *             off_b = sum_{b' < b} (m_b' + T).  Q may be NULL when O is NULL.
 *   O         output rows, same layout as Q, or NULL (fill the cache only).
 *   m_per_seq HOST array of B prefix lengths, 0 <= m_b <= m (capacity).
 *   T         number of output rows per sequence already produced (>= 0).
 * Row i of sequence b attends to keys j <= i with j < m_b (the prefix) or
 * j > i - n (the window; "Unlimited-OCR deep dive", N(t) = P U D_n(t)).
 * Cache effect: prefix rows 0..m_b-1 go to the static prefix region (encoded
 * once, "no state transition", GeekNews, model architecture); output j goes
 * to ring slot j mod n for j >= T - n; m_b and t_b = T are set.
 * Inputs may contain no Inf/NaN: rows past a sequence's end are read but
 * masked.  Errors: RSWA_EINVAL, RSWA_ECAPACITY (some m_b > m), RSWA_ECUDA.
 */
RSWA_API int rswa_prefill(rswa_cache* cache, const void* Q, const void* K,
                          const void* V, void* O, const int64_t* m_per_seq,
                          int64_t T, void* stream);

/*
 * rswa_prefill with a number of output rows per sequence: t_per_seq is a
 * HOST array of B values T_b >= 0, and sequence b occupies rows
 * off_b .. off_b + m_b + T_b - 1 with off_b = sum_{b' < b} (m_b' + T_b').
 * Several documents of different lengths packed into one call, each with its
 * own R-SWA mask (as multi-page training packs documents into one 32K
 * sequence, GeekNews "Unlimited OCR", training setup).  Sets t_b = T_b.
 * Errors as rswa_prefill.
 */
RSWA_API int rswa_prefill_varlen(rswa_cache* cache, const void* Q,
                                 const void* K, const void* V, void* O,
                                 const int64_t* m_per_seq,
                                 const int64_t* t_per_seq, void* stream);

/*
 * Append output t_b's key and value for every sequence: k, v are [B][H][d].
 * Writes ring slot t_b mod n - once t_b >= n this overwrites the oldest
 * output, the (m+1)-th entry of the pages' queue (GeekNews, model
 * architecture) - then advances t_b by one on the device.
 * Errors: RSWA_EINVAL, RSWA_EHANDLE, RSWA_ECUDA.
 */
RSWA_API int rswa_append_kv(rswa_cache* cache, const void* k, const void* v,
                            void* stream);

/*
 * One decode step: o = attention of q over the cache's m_b + min(n, t_b)
 * keys for every (b, h).  q, o are [B][H][d]; lse (may be NULL) receives
 * [B][H] float32 natural-log log-sum-exp of the scaled logits.  The caller
 * appends token t's k, v before decoding q_t, so the token sees itself.
 * Split-K over the prefix with a log-sum-exp combine inside the same launch;
 * per-step cost depends on m_b + min(n, t_b) only, not on t_b (GeekNews,
 * kernel analysis: constant decode-step duration under R-SWA).
 * An empty cache yields o = 0 and lse = -inf.
 * Ordering: decode kernels use programmatic dependent launch and may start
 * while the preceding kernel of the stream still runs.  Every decode call
 * except the first after rswa_prefill, rswa_prefill_varlen or
 * rswa_cache_set_t on this cache may read the cache's prefix rows and m_b
 * before that kernel has finished, so between two such calls the prefix
 * rows are read-only: write them only through the prefill calls, or before
 * rswa_cache_set_t (which synchronises its stream).
 * Errors: RSWA_EINVAL, RSWA_EHANDLE, RSWA_ECUDA.
 */
RSWA_API int rswa_decode_step(rswa_cache* cache, const void* q, void* o,
                              float* lse, void* stream);

/*
 * rswa_append_kv(k, v) followed by rswa_decode_step(q) in one launch: the new
 * key/value is attended straight from k, v and written to its ring slot by
 * the same kernel; t_b advances once every head of the sequence is done.
 * Same layouts and errors as the two calls it replaces.
 */
RSWA_API int rswa_decode_step_fused(rswa_cache* cache, const void* q,
                                    const void* k, const void* v, void* o,
                                    float* lse, void* stream);

/*
 * Decode a block of `block` consecutive output tokens per sequence in one
 * call (1 <= block <= 2^24): q, o are [B][block][H][d] and k, v are
 * [B][block][H_kv][d] for outputs t_b .. t_b + block - 1; lse (may be NULL)
 * is [B][block][H] float32.
 * Output t_b + i attends to the prefix, to the cached outputs of its window
 * j in [max(0, t_b + i - n + 1), t_b), and to the block's tokens of its
 * window, i' in [max(0, i - n + 1), i] - exactly what `block` single steps
 * would give (N(t) = P U D_n(t), "Unlimited-OCR deep dive" pseudo-code
 * block).  Afterwards the ring holds the last n outputs (slot j mod n; a
 * block longer than n replaces the whole ring with its last n tokens) and
 * t_b has advanced by `block`.  For verifying drafted tokens (a few tokens)
 * or prefilling output text into an existing cache (any length).
 * block == 1 runs rswa_decode_step_fused (same layouts), so the prefix
 * ordering rule of rswa_decode_step holds for every block size.  The append
 * follows every read of the ring (the slots it overwrites are read by the
 * block's earlier outputs): blocks of 64 or more on a bf16, head_dim 128
 * cache take two kernels on `stream`, attention on the tensor cores and then
 * the append, which waits for it; shorter blocks (and other caches) take one
 * kernel on the CUDA cores whose last CTA per KV head appends.
 * Errors: RSWA_EINVAL (block outside 1..2^24, batch above 65535, null or
 * misaligned pointers), RSWA_EHANDLE, RSWA_ECUDA.
 */
RSWA_API int rswa_decode_block(rswa_cache* cache, const void* q, const void* k,
                               const void* v, int64_t block, void* o,
                               float* lse, void* stream);

/*
 * rswa_decode_step_fused without scratch from the cache buffer.  (Not part of
 * the method on the pages: it has no counterpart there.)
 *
 * Who needs it: a caller whose device memory is fixed up front and who must
 * not allocate once decoding runs - for example a serving loop that keeps a
 * set budget of buffers, because cudaMalloc can stall the whole device while
 * it synchronises and can fail when memory is fragmented, or a plug-in whose
 * host application owns every device byte.  The split-K partials and arrival
 * counters of this call live in a fixed 4 MiB array inside the library's own
 * device memory (allocated when the library's device code is loaded and held
 * by every GPU that loads it until the process exits).  The call itself
 * allocates nothing and calls no allocating routine.
 *
 * Same arguments, layouts and result as rswa_decode_step_fused; the scratch
 * region of the cache buffer goes unused by this call.
 *   - Limit: the cache must need at most 4 MiB of scratch,
 *     B * H * max_chunks * (d + 2) * 4 bytes of partials plus B * H * 4
 *     bytes of counters, each rounded up to 256 bytes; a larger cache is
 *     rejected with RSWA_ECAPACITY before anything runs.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current) and keeps it for the life of
 *     the process.  Make that first call before any stream capture, and do
 *     not use this call across a device reset (cudaDeviceReset), which
 *     reloads the library's device code and moves the array.
 *   - Every call shares the one array and it keeps the previous call's
 *     contents; each call clears its counters on the caller's stream first.
 *     Calls that overlap on the GPU (other streams, other caches, other
 *     threads) race on the array: order them.
 * Errors: RSWA_EHANDLE, RSWA_EINVAL, RSWA_ECAPACITY, RSWA_ECUDA.
 */
RSWA_API int rswa_decode_step_fused_static(rswa_cache* cache, const void* q,
                                           const void* k, const void* v,
                                           void* o, float* lse, void* stream);

/*
 * Live cache size of sequence b in bytes: C(t_b) * H_kv * d * 2 (K and V) *
 * element size (H_kv = heads unless created with kv_heads), with
 * C(t) = m_b + min(n, t) ("Unlimited-OCR deep dive",
 * cache-size line; GeekNews, KV cache management).  Synchronous: waits for
 * the device (cudaDeviceSynchronize) and reads m_b, t_b.  A test and
 * reporting helper, not a hot-path call.  Errors: RSWA_EINVAL, RSWA_ECUDA.
 */
RSWA_API int rswa_cache_bytes(rswa_cache* cache, int b, size_t* out);

/* Token count C(t_b) = m_b + min(n, t_b) of sequence b.  Synchronous like
 * rswa_cache_bytes. */
RSWA_API int rswa_cache_len(rswa_cache* cache, int b, int64_t* out);

/* Number of outputs t_b appended so far to sequence b.  Synchronous. */
RSWA_API int rswa_cache_get_t(rswa_cache* cache, int b, int64_t* out);

/*
 * Restore t_b for every sequence (t_per_seq: HOST array of B values >= 0),
 * e.g. when resuming a saved cache.  The ring is taken to hold outputs
 * t_b - min(n, t_b) .. t_b - 1 in slots j mod n; the call rewrites no
 * key/value data.  It also clears the decode kernels' split-K arrival
 * counters.  Copies from host memory and synchronises the stream before
 * returning (not for use inside stream capture).
 * After a decode step that reported RSWA_EDEVICE (rswa_sync_status), its
 * outputs are undefined and t_b may be advanced for some heads and not for
 * others, though the step's key and value were appended: call
 * rswa_cache_set_t with the intended t_b (the old one + 1) before the next
 * step.
 * Errors: RSWA_EINVAL, RSWA_ECUDA.
 */
RSWA_API int rswa_cache_set_t(rswa_cache* cache, const int64_t* t_per_seq,
                              void* stream);

/*
 * Byte offsets of the K and V slabs inside the cache buffer.  Each slab is
 * [B][H_kv][m + n][d] in the cache dtype: rows 0..m-1 of a (b, h) slab hold the
 * prefix, rows m..m+n-1 the ring, output j in row m + (j mod n).  For
 * inspection and checkpointing; host-only, no CUDA call.  Prefix rows written
 * here must be followed by rswa_cache_set_t before the next decode call (see
 * the ordering rule of rswa_decode_step).
 * Errors: RSWA_EINVAL, RSWA_EHANDLE.
 */
RSWA_API int rswa_cache_kv_offsets(rswa_cache* cache, size_t* k_offset,
                                   size_t* v_offset);

/*
 * Wait for all work on the current device, then report the first error a
 * kernel flagged on this cache (RSWA_EDEVICE) or a CUDA error (RSWA_ECUDA),
 * else RSWA_OK.  Clears the device flag.
 */
RSWA_API int rswa_sync_status(rswa_cache* cache);

/*
 * Host-side fault injection for tests: the next `count` calls that would
 * touch CUDA fail with RSWA_ECUDA before launching anything.  No GPU fault is
 * involved.
 */
RSWA_API void rswa_debug_fail_next_cuda(int count);

/*
 * Test hook: bound, in nanoseconds, on each wait for a pipeline phase (a
 * tile landing, a tensor core result, a softmax hand-off) of the pipelined
 * kernels - the tensor-core prefill, block decode and grouped-head decode,
 * and the shared-memory streaming decode; 0 restores the default of one
 * second.
 * Kernels launched with a bound that runs out stop, drain their own copies
 * and tensor-core work (those waits keep the default bound), free their
 * tensor memory and set the device flag that rswa_sync_status() reports as
 * RSWA_EDEVICE.  Applies to launches made after the call; process-wide.
 */
RSWA_API void rswa_debug_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* RSWA_H */
