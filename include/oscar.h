/*
 * oscar.h - C ABI of the GB300 (sm_103a) OScaR INT2 KV-cache library.
 *
 * The method ("OScaR: The Occam's Razor for Extreme KV Cache Quantization in
 * LLMs and Beyond", arXiv 2605.19660, Abstract; ai-papers.net summary,
 * section "OScaRの提案手法"): every key vector k is rotated by the normalised
 * Walsh-Hadamard matrix H_d ("Canalized Rotation"), its L2 norm n is stored and
 * the rotated key divided by it ("Omni-Token Scaling"), and the result is
 * quantised to INT2 per channel.  Values are quantised to INT2 per token (the
 * KIVI convention cited in the qiita.com NOVA-KV article, section
 * "KV キャッシュを「読む」時間が、計算そのものより長い").  Decoding reads the
 * packed cache directly (the pages compare against BF16 FlashDecoding-v2,
 * ai-papers.net section "実験結果").
 *
 * Fixed configuration of this library:
 *   d  = 128  head dimension
 *   G  = 128  tokens per key quantisation group; groups cover absolute
 *             positions [128 g, 128 g + 128)
 *   Gv = 32   channels per value quantisation group
 *   H_d[i][j] = (-1)^popcount(i & j) / sqrt(128)  (Sylvester order)
 *   s = (max - min) / 3, z = min (float32); code = clamp(rne((x - z) / s), 0, 3);
 *   s == 0 gives code 0.  Dequantised value: code * s + z.
 *   The L mod 128 most recent tokens of a sequence stay in bf16 (the
 *   residual window) until their group fills; then the whole group is
 *   quantised from the bf16 originals.
 *
 * Conventions
 *   - Ownership: the caller owns every device buffer (arena, inputs, outputs,
 *     workspace).  The library never allocates device memory; the opaque
 *     oscar_cache object is a small host allocation.
 *   - Asynchrony: compute calls enqueue kernels on `stream` (a cudaStream_t,
 *     NULL = legacy default stream) and return without synchronising.  The
 *     per-sequence lengths live on the host, so launch shapes are computed
 *     without device read-back.  All calls on one cache must use one stream
 *     (or be ordered by the caller).
 *   - Errors: every call returns an oscar_status.  Arguments are validated
 *     on the host before anything is enqueued; on error nothing is enqueued
 *     and the cache is unchanged.  oscar_last_error() returns a
 *     thread-local message for the last failing call.  No C++ exception or
 *     abort crosses this boundary.
 *   - GQA: query head h reads KV head h / (num_q_heads / num_kv_heads).
 *   - dtypes: k, v, q and out are bf16 (uint16 storage), row-major.
 */
#ifndef OSCAR_H
#define OSCAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct oscar_cache oscar_cache;

typedef enum oscar_status {
  OSCAR_OK = 0,
  OSCAR_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad sequence id    */
  OSCAR_ERR_CAPACITY = 2,      /* would exceed max_seq_len / arena / plan    */
  OSCAR_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed       */
  OSCAR_ERR_UNSUPPORTED = 4,   /* head_dim != 128, G != 128, Gv != 32, ...   */
  OSCAR_ERR_DEVICE_TIMEOUT = 5 /* a kernel's bounded wait gave up (see
                                  oscar_cache_check)                          */
} oscar_status;

typedef struct oscar_cache_config {
  int32_t max_batch;     /* number of sequence slots, >= 1                   */
  int32_t num_kv_heads;  /* Hkv, >= 1                                        */
  int32_t head_dim;      /* must be 128                                      */
  int32_t max_seq_len;   /* capacity in tokens per slot, >= 1                */
  int32_t group_size;    /* must be 128 (G)                                  */
  int32_t value_group;   /* must be 32 (Gv)                                  */
  int32_t device;        /* CUDA device ordinal of the arena                 */
  int32_t meta_bits;     /* 32 (default; 0 also means 32): float32 scales,   */
                         /* zeros and norms, 13,824-byte blocks; 16: float16 */
                         /* (rounded to nearest even; codes decided against  */
                         /* the rounded values), 11,008-byte blocks          */
} oscar_cache_config;

/* Kinds for oscar_cache_bytes. */
enum {
  OSCAR_BYTES_USED = 0,            /* packed groups + bf16 window in use     */
  OSCAR_BYTES_BF16_EQUIVALENT = 1, /* bytes of a plain bf16 K+V cache       */
  OSCAR_BYTES_ARENA = 2            /* arena size the configuration needs    */
};

/*
 * Device arena layout (all offsets in bytes from the arena base; the arena
 * must be 256-byte aligned):
 *
 *   [0, 256)                       status words; word 0 = device error flags
 *   [256, 256 + 4 S H)             per (slot, kv head): float32 bit pattern of
 *                                  the largest value scale s_v quantised so
 *                                  far (4 bytes each; S = max_batch, H = Hkv)
 *   [256 + 4 S H, M)               per (slot, kv head): float32 bit pattern of
 *                                  the largest |value zero| z_v quantised so
 *                                  far, M = 256-aligned end
 *   blocks  (base = M)             one block of B bytes per
 *                                  (slot, kv head, group g):
 *                                  base + ((slot*Hkv + head)*max_groups + g)*B,
 *                                  max_groups = ceil(max_seq_len / 128),
 *                                  B = 13,824 (meta_bits 32) or 11,008 (16)
 *   windows (after the blocks,     65,536 bytes per (slot, kv head): 128 bf16
 *            256-aligned)          key rows (slot p mod 128) then 128 bf16
 *                                  value rows, 256 bytes per row
 *
 * One group block (the unit the decode kernel streams), meta_bits 32:
 *   +0      K codes, 4,096 B, "fragment order" of the 128x128 matrix
 *           X[row = token][col = channel]
 *   +4096   K scale s_c, float32 [128] (per channel)
 *   +4608   K zero  z_c, float32 [128]
 *   +5120   K norm  n_t, float32 [128] (per token, position order)
 *   +5632   V codes, 4,096 B, fragment words of X[row = channel][col = token]
 *           in "V order"
 *   +9728   V scale s[t][0..3], float32 [128][4] (per token, one per
 *           32-channel group), token t in row t ^ ((t >> 3) & 1)
 *           (neighbouring tokens swap rows where bit 3 of t is set)
 *   +11776  V zero  z[t][0..3], float32 [128][4], rows as the V scale
 * meta_bits 16: the same sections with float16 metadata:
 *   +0 K codes, +4096 K scale, +4352 K zero, +4608 K norm (float16 [128]
 *   each), +4864 V codes, +8960 V scale, +9984 V zero (float16 [128][4]
 *   each); 11,008 bytes, 86 per token and head.
 *
 * Fragment words of a 128x128 matrix of 2-bit codes X[row][col]: the 32-bit
 * word F(mt, lane, j, r) holds the 16 codes with
 *   row = 16*mt + (lane >> 2) + 8*r,
 *   col = 16*(4*j + kk) + 8*hf + 2*(lane & 3) + e,   kk in 0..3, hf, e in {0,1},
 * code at bits [b, b+1] with b = 16*e + 4*kk + 2*hf
 * (mt in 0..7, lane in 0..31, r, j in {0,1}; words are little-endian).
 * "Fragment order" (K codes) stores F(mt, lane, j, r) as word
 *   w = (mt*32 + lane)*4 + 2*j + r,
 * "V order" (V codes) as word
 *   w = ((mt*2 + j)*32 + lane)*2 + r.
 */

/* Arena bytes needed by `cfg`.  Pure host arithmetic. */
oscar_status oscar_cache_required_bytes(const oscar_cache_config* cfg, size_t* out_bytes);

/* Create a cache over a caller-owned device arena of `arena_bytes` (at least
 * oscar_cache_required_bytes) on cfg->device.  Zeroes the status and
 * metadata region (a blocking cudaMemset of a few KB); all sequence lengths
 * start at 0.  *out receives a host object to pass to the other calls. */
oscar_status oscar_cache_create(const oscar_cache_config* cfg, void* device_arena,
                                size_t arena_bytes, oscar_cache** out);

/* Free the host object (never the arena). NULL is accepted. */
oscar_status oscar_cache_destroy(oscar_cache* cache);

/* Set the length of slot `seq` to 0 (or every slot if seq == -1) and clear its
 * value-scale maxima, enqueued on `stream`. */
oscar_status oscar_cache_reset(oscar_cache* cache, int32_t seq, void* stream);

/* Current length (tokens) of slot `seq`. */
oscar_status oscar_cache_length(const oscar_cache* cache, int32_t seq, int32_t* out_len);

/*
 * Append new tokens to `n_seqs` sequences (prefill chunks or single decode
 * tokens; the method's compression step, OScaR abstract / ai-papers.net
 * "OScaRの提案手法").
 *   seq_ids  host int32 [n_seqs], distinct slot ids in [0, max_batch)
 *   cu_new   host int32 [n_seqs + 1], cu_new[0] = 0, non-decreasing;
 *            sequence i appends rows cu_new[i] .. cu_new[i+1]-1
 *   k, v     device bf16 [cu_new[n_seqs], Hkv, 128] (rows of the raw, i.e.
 *            unrotated, keys and values; 16-byte aligned, and read with
 *            32-byte loads, which are faster, when both are 32-byte
 *            aligned); host memory fails with OSCAR_ERR_INVALID_ARG
 * Every 128-token group that fills is rotated, norm-scaled and quantised
 * (keys) and quantised (values) from its bf16 tokens (earlier ones from the
 * window, new ones from k/v) into its block; the remaining tokens go to the
 * window.  Fails with OSCAR_ERR_CAPACITY if a length would exceed
 * max_seq_len.  Lengths are updated on the host when the call returns.
 */
oscar_status oscar_quantize_append(oscar_cache* cache, int32_t n_seqs, const int32_t* seq_ids,
                                   const int32_t* cu_new, const void* k, const void* v,
                                   void* stream);

/* Workspace bytes oscar_decode_attention needs for up to `n_seqs` sequences
 * and `num_q_heads` query heads (an upper bound independent of lengths). */
oscar_status oscar_decode_workspace_bytes(const oscar_cache* cache, int32_t n_seqs,
                                          int32_t num_q_heads, size_t* out_bytes);

/*
 * Single-query decode attention over the packed cache (split-K flash
 * decoding, GQA, ragged batch).
 *   seq_ids      host int32 [n_seqs]; every slot must have length >= 1
 *   q            bf16 [n_seqs, num_q_heads, 128] (unrotated queries), 16-byte
 *                aligned, in device memory or page-locked host memory
 *   num_q_heads  any multiple of Hkv; the kernels serve up to 8 query heads
 *                of a KV head per pass over the cache, so num_q_heads / Hkv
 *                = 9..16 takes two passes, 17..24 three, and so on
 *   softmax_scale  0 means 1 / sqrt(128)
 *   out          bf16 [n_seqs, num_q_heads, 128], 16-byte aligned, in device
 *                memory or page-locked host memory
 *   workspace    device scratch of >= oscar_decode_workspace_bytes bytes,
 *                16-byte aligned; contents need not be initialised
 * For a quantised token t with norm n_t the score is
 *   s_t = n_t * (H_d q) . (code_t * s + z) * softmax_scale,
 * for a window token s_t = q . k_t * softmax_scale; out = softmax(s) . v_hat.
 * Attends to exactly the tokens in the cache (append the current token first).
 * Host buffers: q and out may be page-locked host memory (cudaHostAlloc,
 * cudaHostRegister, torch pin_memory); the kernels then read q and write out
 * in place through the device mapping (over NVLink-C2C on Grace systems), so
 * a decode step from host inputs to host outputs needs no staging copies.
 * Pageable host memory and device memory of another device fail with
 * OSCAR_ERR_INVALID_ARG before anything is enqueued.
 * Stream order: the main kernel is launched as a programmatic dependent of
 * the kernel before it in `stream`.  Before it waits for that kernel it only
 * copies cache blocks of groups closed before the previous decode call on
 * this cache, when that call used the same stream (the library tracks its
 * appends and decodes); q, the workspace and all other inputs are read after
 * the wait, so a preceding kernel may produce q.  The arena must be written
 * through this library only.
 */
oscar_status oscar_decode_attention(oscar_cache* cache, int32_t n_seqs, const int32_t* seq_ids,
                                    const void* q, int32_t num_q_heads, float softmax_scale,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    void* stream);

/*
 * oscar_decode_attention with float32 outputs: the merged attention output
 * before any bf16 rounding, for callers that keep attention outputs in
 * float32 (and for checking the decode at float32 precision).
 *   out  float32 [n_seqs, num_q_heads, 128], 16-byte aligned, device or
 *        page-locked host memory
 * Every other argument, the result before the output rounding, and the
 * errors are those of oscar_decode_attention.
 */
oscar_status oscar_decode_attention_f32(oscar_cache* cache, int32_t n_seqs, const int32_t* seq_ids,
                                        const void* q, int32_t num_q_heads, float softmax_scale,
                                        void* out, void* workspace, size_t workspace_bytes,
                                        void* stream);

/*
 * One decode step fused: append one token to each of `n_seqs` sequences,
 * then decode, with the same result as oscar_quantize_append (one row per
 * sequence) followed by oscar_decode_attention.  The ai-papers.net OScaR
 * summary, section "まとめと今後の展望", notes that the quantisation
 * overhead weighs relatively more at short context; this call removes one
 * launch from most decode steps.
 *   k_new, v_new  device bf16 [n_seqs, Hkv, 128], the new token of each
 *                 sequence (16-byte aligned)
 *   other arguments as for oscar_decode_attention (q and out may be host
 *   buffers in the same way).
 * When no sequence's new length is a multiple of 128 (127 steps in 128),
 * the step is one decode launch: the combine kernel attends the new token as
 * the last window row straight from k_new / v_new and stores it into the
 * window.  When a group closes, the quantiser runs first (two launches), so
 * the group is attended quantised.  All arguments are validated before
 * anything is enqueued; on error nothing changes.
 */
oscar_status oscar_append_decode(oscar_cache* cache, int32_t n_seqs, const int32_t* seq_ids,
                                 const void* k_new, const void* v_new, const void* q,
                                 int32_t num_q_heads, float softmax_scale, void* out,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Chunked-prefill attention over the cache: each of the n_q queries of a new
 * chunk of sequence `seq` attends to every token already in its cache
 * (quantised groups and window; no mask, the cache precedes the chunk), with
 * the decode path's scores and values (OScaR abstract; ai-papers.net
 * "OScaRの提案手法").  Call it before appending the chunk; the chunk's own
 * causal attention is merged in by the caller with lse.
 *   q            bf16 [n_q, num_q_heads, 128], 16-byte aligned
 *   out          bf16 [n_q, num_q_heads, 128], 16-byte aligned
 *   lse          fp32 [n_q, num_q_heads] or NULL: ln sum_t exp(s_t) per row
 *                (natural log, scores times softmax_scale)
 *   q, out and lse may be device or page-locked host memory (see
 *   oscar_decode_attention); other memory fails with OSCAR_ERR_INVALID_ARG.
 *   softmax_scale  0 means 1 / sqrt(128)
 *   workspace    NULL, or device memory (16-byte aligned) of workspace_bytes
 *                for partial results: the history's groups are then split
 *                into parts processed by separate CTAs and merged by a
 *                second kernel, so that the CTAs fill whole waves of SMs.
 *                As many parts are used as fit, up to the number that
 *                oscar_prefill_workspace_bytes sizes; NULL (or too small for
 *                two parts) runs unsplit.  Results agree within rounding.
 * Any GQA ratio.  The sequence must be non-empty.
 */
oscar_status oscar_prefill_attention(oscar_cache* cache, int32_t seq, int32_t n_q, const void* q,
                                     int32_t num_q_heads, float softmax_scale, void* out, float* lse,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * Workspace bytes that let oscar_prefill_attention split the history of
 * sequence `seq` (at its current length) for n_q queries of num_q_heads
 * heads: parts x Hkv x n_q x (num_q_heads / Hkv) x 528 bytes, 0 when no
 * split pays off (short histories, or rows that already fill the SMs).
 */
oscar_status oscar_prefill_workspace_bytes(const oscar_cache* cache, int32_t seq, int32_t n_q,
                                           int32_t num_q_heads, size_t* out_bytes);

/*
 * Decode that allocates nothing and takes no workspace.  The OScaR pages have
 * no counterpart to this call; it exists for callers that cannot allocate
 * device memory where they decode (code inside a memory pool or arena it does
 * not own, plugins whose host framework forbids allocation on the serving
 * path, callers that must keep a fixed device footprint).
 *   Same arguments and results as oscar_decode_attention, without workspace.
 *   The split-K partials go to a file-scope device array of 4 MiB that every
 *   GPU loading this library holds until the process exits.  Calls needing
 *   more than that (sequences x KV heads plus two rows per SM of partials)
 *   fail with OSCAR_ERR_CAPACITY and a message; use oscar_decode_attention.
 *   The first call on a device looks up the array's device address (with
 *   the cache's device current); make that first call before any CUDA stream
 *   capture.  No device memory is allocated or freed, and nothing in the
 *   array needs to start at zero (each call writes every partial it reads).
 *   Every call shares the one array: calls whose kernels overlap on the GPU
 *   (different streams, or different threads without ordering) race on it
 *   and give wrong results.
 */
oscar_status oscar_decode_attention_noalloc(oscar_cache* cache, int32_t n_seqs, const int32_t* seq_ids,
                                            const void* q, int32_t num_q_heads, float softmax_scale,
                                            void* out, void* stream);

/* Footprint: kind = OSCAR_BYTES_USED / _BF16_EQUIVALENT for slot `seq`
 * (or all slots if seq == -1), or OSCAR_BYTES_ARENA.  Host arithmetic:
 * a full group costs 13,824 B per KV head (108 B per token) versus 65,536 B
 * (512 B per token) in bf16; a window token costs 512 B. */
oscar_status oscar_cache_bytes(const oscar_cache* cache, int32_t seq, int32_t kind,
                               size_t* out_bytes);

/* Arena offsets of the block of (seq, kv_head, group) and of the window of
 * (seq, kv_head), for inspection and tests. */
oscar_status oscar_cache_block_offset(const oscar_cache* cache, int32_t seq, int32_t kv_head,
                                      int32_t group, size_t* out_offset);
oscar_status oscar_cache_window_offset(const oscar_cache* cache, int32_t seq, int32_t kv_head,
                                       size_t* out_offset);

/*
 * Test hook of the failure path: the next INT2 decode launch made on the
 * calling thread (oscar_decode_attention, _f32 or oscar_append_decode) has
 * one bulk copy of its first CTA left unissued, and its bounded waits give up
 * after 2^14 polls instead of 2^24.  The consumer waiting for that copy then
 * gives up, the kernel sets the arena's error flag, skips its remaining work
 * and returns (no fault, no hang; the results of that call are undefined),
 * and oscar_cache_check reports OSCAR_ERR_DEVICE_TIMEOUT.  Later calls are
 * unaffected.  Not for production use.
 */
oscar_status oscar_test_arm_wait_timeout(void);

/* Test hook: for each of the n_seqs slots in seq_ids, the number of leading
 * groups whose blocks the next decode on `stream` would copy before its grid
 * dependency wait (INT32_MAX: all of them), from the host's record of the
 * appends, resets and decodes enqueued on this cache.  out: host int32
 * [n_seqs].  Enqueues nothing. */
oscar_status oscar_test_settled_groups(const oscar_cache* cache, int32_t n_seqs,
                                       const int32_t* seq_ids, void* stream, int32_t* out);

/* Synchronise `stream`, then read the device error flags of the arena.
 * Returns OSCAR_ERR_DEVICE_TIMEOUT if a kernel's bounded wait gave up since
 * the last check (and clears the flags), OSCAR_OK otherwise. */
oscar_status oscar_cache_check(oscar_cache* cache, void* stream);

/*
 * BF16 reference decode (the speed-ratio baseline standing in for the
 * pages' BF16 FlashDecoding-v2 comparator, ai-papers.net "実験結果"): the same
 * split-K structure over a plain bf16 cache.
 *   k_cache, v_cache  device bf16 [n_seqs_cap, Hkv, max_seq_len, 128]
 *   seq_ids / seq_lens host int32 [n_seqs]: slot and length (>= 1) of each
 *   q, out            bf16 [n_seqs, num_q_heads, 128], device or page-locked
 *                     host memory (the caches and the workspace: device only)
 * Scores are q . k_t * softmax_scale in float32, softmax and P.V in float32.
 */
oscar_status oscar_bf16_decode_workspace_bytes(int32_t n_seqs, int32_t num_kv_heads,
                                               int32_t num_q_heads, size_t* out_bytes);
oscar_status oscar_bf16_decode_attention(int32_t n_seqs, const int32_t* seq_ids,
                                         const int32_t* seq_lens, const void* k_cache,
                                         const void* v_cache, int32_t num_kv_heads,
                                         int32_t max_seq_len, const void* q,
                                         int32_t num_q_heads, float softmax_scale, void* out,
                                         void* workspace, size_t workspace_bytes, void* stream);

/* Profiling hook: when both are non-NULL, the following decode calls on this
 * thread record `start_event` / `stop_event` (cudaEvent_t) around their main
 * split-K kernel.  Pass NULLs to turn it off. */
oscar_status oscar_set_timing_events(void* start_event, void* stop_event);

/* Thread-local message of the last failing call ("" if none). */
const char* oscar_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* OSCAR_H */
