/*
 * oscar_kv.h -- C ABI of the GB300 (sm_103a) INT2 rotated paged KV cache.
 *
 * The method is OSCAR-style INT2 KV caching as described on the axbrief.com page
 * "Together AI's OSCAR breaks the 2-bit KV cache accuracy barrier":
 *   - section "attention-statistics rotation + Triton kernels": keys are rotated by
 *     R_K = U_Q * H_Had * P_br (U_Q = eigenvectors of the query covariance
 *     C_Q = (1/N) sum_n q_n^T q_n, H_Had the normalised 128-point Hadamard, P_br the
 *     bit-reversal permutation); the write path clips each token with c_K = 0.96 /
 *     c_V = 0.92 and quantises it per token to asymmetric INT2 in groups of
 *     G_K = 64 channels; the read path unpacks, dequantises and inverse-rotates
 *     inside one fused attention pass with no extra memory traffic;
 *   - section "attention-statistics rotation + Triton kernels", last paragraph: the
 *     value rotation R_V is absorbed offline into the projection weights, so values
 *     are written unrotated;
 *   - opening paragraph and section "OSCAR release": sink tokens and the recent
 *     window stay in BF16 (0.24% of a 128K context);
 * and on the techllm.github.io page "KV cache compression: TurboQuant, OSCAR,
 * EpiCache", section "OSCAR": a mixed-precision paged cache (recent tokens BF16,
 * older history INT2).
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA global-memory addresses on the current device; host
 *     pointers are plain CPU memory.  Each argument says which it is.
 *   - The caller allocates and frees ALL device memory (buffer sizes come from the
 *     *_bytes() queries).  The library allocates only its host-side handle.
 *   - Calls that take a stream enqueue their GPU work on it and return without
 *     waiting, unless stated otherwise.  `stream` is a cudaStream_t passed as void*
 *     (NULL = the legacy default stream).
 *   - Return value: OSCAR_OK (0) or a negative OSCAR_E* code.  Argument, capacity and
 *     alignment errors are detected on the host before anything is enqueued, and
 *     leave the cache unchanged.  OSCAR_ECUDA reports a CUDA launch or copy error;
 *     oscar_last_cuda_error() gives the CUDA error code.
 *   - One cache is used from one host thread and one stream at a time.
 *   - Inputs are assumed finite; NaN or Inf in keys, values or queries gives
 *     undefined codes and outputs (never out-of-bounds memory access).
 *   - Head mapping (grouped-query attention): query head hq reads KV head hq / G,
 *     G = num_q_heads / num_kv_heads.
 */
#ifndef OSCAR_KV_H
#define OSCAR_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OSCAR_OK 0
#define OSCAR_EINVAL (-1)     /* bad argument or shape */
#define OSCAR_ENOPAGES (-2)   /* the page pool or a page-table row is full */
#define OSCAR_EWORKSPACE (-3) /* workspace missing or too small */
#define OSCAR_ECUDA (-4)      /* a CUDA call failed */
#define OSCAR_EALIGN (-5)     /* a device pointer is not 16-byte aligned */
#define OSCAR_ERANGE (-6)     /* a request index or position is out of range */
#define OSCAR_ETIMEOUT (-7)   /* a bounded wait inside a kernel gave up (see oscar_decode_status) */
#define OSCAR_ESCRATCH (-8)   /* the call needs more scratch than oscar_decode_attention_noalloc has */

#define OSCAR_DTYPE_F32 0
#define OSCAR_DTYPE_BF16 1

/* Fixed geometry of this implementation. */
#define OSCAR_HEAD_DIM 128
#define OSCAR_PAGE_TOKENS 64   /* INT2 tokens per page */
#define OSCAR_GROUP 64         /* default channels per quantisation group (64 or 128 per tensor) */
#define OSCAR_MAX_GQA 16       /* largest num_q_heads / num_kv_heads */
/* Bytes of one (page, KV head) block with 64-channel groups for keys and values: K codes 2048
 * (32 per token), K scale/min 64x8, V codes 2048, V scale/min 64x8.  A tensor quantised in
 * 128-channel groups keeps one scale/min pair per token (64x4 bytes): 4864 bytes with keys in
 * groups of 64 and values in groups of 128, 4608 with both in groups of 128
 * (oscar_page_head_bytes).  Inside the two code regions the 2-bit codes are stored in the order
 * the decode kernel's tensor-core fragments read them (not the logical order); oscar_read_int2
 * returns them in the logical order. */
#define OSCAR_PAGE_HEAD_BYTES 5120

typedef struct {
    int32_t batch;             /* requests (rows of the page table), >= 1 */
    int32_t num_kv_heads;      /* >= 1 */
    int32_t num_q_heads;       /* num_kv_heads * G, G in {1..8, 12, 16} */
    int32_t head_dim;          /* must be 128 */
    int32_t page_size;         /* must be 64 */
    int32_t group_size;        /* key quantisation group: 64 or 128 channels */
    int32_t sink;              /* BF16 sink tokens, must be 64 */
    int32_t window;            /* BF16 recent-window tokens, must be 256 */
    int32_t max_pages_total;   /* physical INT2 pages in the pool, >= 1 */
    int32_t max_pages_per_seq; /* INT2 pages one request may hold, >= 1 */
    float clip_k;              /* key clip factor, 0 < c <= 1 (default 0.96) */
    float clip_v;              /* value clip factor, 0 < c <= 1 (default 0.92) */
    int32_t group_size_v;      /* value quantisation group: 64 or 128 channels; 0 = group_size */
} oscar_cache_desc;

typedef struct oscar_cache oscar_cache; /* opaque host handle */

/* Fill *d with the defaults (head_dim 128, page 64, groups of 64 for keys and values, sink 64,
 * window 256, clip 0.96 / 0.92); the caller then sets batch, heads and the page counts.
 * The group sizes select the page format.  Groups of 64 are the OSCAR pages' G_K = 64 (axbrief.com
 * OSCAR page, section "attention-statistics rotation + Triton kernels"); keys in groups of 64 with
 * values in groups of 128 (2.375 bits per stored value) and both in groups of 128 (2.25 bits, 2.28
 * with the BF16 sink and window of a 128K context) are the configurations behind the 2.38 and 2.28
 * effective bits the same page reports (section "Naive INT2 0 vs OSCAR 71.86"). */
void oscar_default_desc(oscar_cache_desc *d);
/* Bytes of one (page, KV head) block of the pool for the descriptor's group sizes (5120, 4864 or
 * 4608), or 0 if *d is invalid. */
size_t oscar_page_head_bytes(const oscar_cache_desc *d);

/* Device buffer sizes (bytes) the caller must allocate for a cache described by *d;
 * 0 if *d is invalid.
 *   pool:       max_pages_total * num_kv_heads * oscar_page_head_bytes(d); physical page p,
 *               KV head h starts at byte (p * num_kv_heads + h) * oscar_page_head_bytes(d).
 *   bf16:       batch * num_kv_heads * 2 * (sink + window) * 128 bf16 values, laid out
 *               [b][h][K|V][slot][128]; slot = pos for pos < sink, else
 *               sink + (pos - sink) % window.
 *   page_table: batch * max_pages_per_seq int32 ([b][logical page] -> physical page).
 *   seq_lens:   per-request metadata: batch int32 (tokens held per request), then, from byte
 *               16 * ceil(batch / 4), uint32 [batch][num_kv_heads]: the fp16 bits of the largest
 *               value scale the write path has quantised for that (request, KV head), zeroed
 *               when the request is released.  The read path derives its fp16 range limit for
 *               p * s_V from it.  Size: the sum of both parts rounded up to 16 bytes. */
size_t oscar_pool_bytes(const oscar_cache_desc *d);
size_t oscar_bf16_bytes(const oscar_cache_desc *d);
size_t oscar_page_table_bytes(const oscar_cache_desc *d);
size_t oscar_seq_lens_bytes(const oscar_cache_desc *d);

/* Create a host handle over caller-owned device buffers (all 16-byte aligned, sizes as
 * above).  The handle keeps the pointers but never frees them.  All requests start
 * empty and the free list hands out physical pages 0, 1, 2, ... until
 * kv_page_table_init() sets another order.  Nothing is enqueued; the first sync
 * clears the device page table and lengths.  pool and bf16 need no initial contents:
 * whatever bits sit in slots and pages a request has not reached (NaN included) never
 * reach a result.
 * Errors: OSCAR_EINVAL (bad descriptor or NULL), OSCAR_EALIGN. */
int oscar_cache_create(const oscar_cache_desc *d, void *pool, void *bf16, int32_t *page_table,
                       int32_t *seq_lens, oscar_cache **out);
int oscar_cache_destroy(oscar_cache *c);
/* Tokens currently held by request b (host mirror), or a negative error. */
int64_t oscar_cache_length(const oscar_cache *c, int32_t b);

/* ---------------------------------------------------------------- kv_page_table
 * The page table maps each request's INT2 history (positions sink .. len - window - 1,
 * 64 per page) onto physical pages of the pool, so a request's pages need not be
 * contiguous (the pages say OSCAR plugs into paged attention without a custom layout:
 * axbrief.com OSCAR page, section "OSCAR release"; techllm.github.io page, section
 * "OSCAR").  The free list and a mirror of the table live on the host: init, reserve
 * and release touch host memory only and mark rows dirty; kv_page_table_sync (also
 * called by kv_quant_append and oscar_decode_attention) copies the dirty entries and
 * lengths to the device buffers with cudaMemcpyAsync on its stream. */

/* Reset every request to length 0 and set the order in which free physical pages are
 * handed out: page_order (host, max_pages_total distinct ids in [0, max_pages_total))
 * or NULL for 0, 1, 2, ...  The next sync clears the device table and lengths.
 * Errors: OSCAR_EINVAL (not a permutation; nothing changes). */
int kv_page_table_init(oscar_cache *c, const int32_t *page_order);
/* Make sure request b owns the pages its INT2 history needs once it holds `new_len`
 * tokens, taking them from the free list.  Errors: OSCAR_ENOPAGES (the pool or the
 * row is full; nothing is taken), OSCAR_ERANGE. */
int kv_page_table_reserve(oscar_cache *c, int32_t b, int64_t new_len);
/* Return request b's pages to the free list and set its length to 0. */
int kv_page_table_release(oscar_cache *c, int32_t b);
/* Copy dirty page-table entries and lengths to the device (async on `stream`). */
int kv_page_table_sync(oscar_cache *c, void *stream);
/* Host mirror of request b's row: writes up to max_out physical ids to `pages` (host)
 * and returns how many pages b holds (or a negative error). */
int kv_page_table_read(const oscar_cache *c, int32_t b, int32_t *pages, int32_t max_out);
/* Physical pages left on the free list. */
int32_t kv_page_table_free_pages(const oscar_cache *c);

/* ---------------------------------------------------------------- write path
 * kv_quant_append: append new_tokens[b] tokens (host array, batch entries, >= 0) to
 * every request b.  k and v (device, bf16, [sum_b new_tokens[b], num_kv_heads, 128],
 * requests in order b = 0, 1, ..., tokens in position order) are the new keys (NOT
 * rotated) and values.  rk (device, fp32, [num_kv_heads][128][128], row-major, row j =
 * input channel) is R_K of each KV head.
 * Position p of request b goes to the sink when p < sink, else to the window ring; a
 * position that falls out of the window (p < len - window) is rotated (keys only:
 * k~ = k . R_K, fp32, serial fused multiply-add over input channels 0..127), clipped
 * (lo = c * group min, hi = c * group max), quantised (s = fp16((hi - lo) / 3),
 * m = fp16(lo), code = clamp(rint((clamp(x, lo, hi) - m) / s), 0, 3), 0 when s = 0)
 * and stored in its INT2 page.  Tokens leaving the window are quantised from their
 * BF16 window copy, so appending L tokens at once or one by one stores the same bytes.
 * Pages are reserved as needed (OSCAR_ENOPAGES leaves the cache unchanged).
 * Range: the clipped group minimum and (hi - lo) / 3 must be representable in fp16
 * (|c * min|, |c * max| up to about 65504); larger values give undefined codes and scales.
 * A group whose scale rounds to 0 in fp16 (a constant group, or a range below 2^-25) stores
 * s = 0 and codes 0, so every element dequantises to m.
 * Source: axbrief.com OSCAR page, section "attention-statistics rotation + Triton
 * kernels" (rotation, c_K, c_V, G_K = 64, per-token asymmetric INT2, V unrotated). */
int kv_quant_append(oscar_cache *c, const void *k, const void *v, const int32_t *new_tokens,
                    const float *rk, void *stream);

/* kv_quant_append_layers: the same append for n_layers caches at once (the layers of one model,
 * which append the same tokens per request), in two kernel launches in all instead of two per
 * layer.  caches[l], k[l], v[l] and rk[l] (host arrays of n_layers entries) are layer l's cache,
 * new keys, new values and R_K, each exactly as for kv_quant_append; new_tokens is shared.  Every
 * cache must have the same batch, KV heads, group sizes and current lengths (OSCAR_EINVAL
 * otherwise); clip factors may differ.  workspace (device, 16-byte aligned, at least
 * kv_quant_append_layers_workspace_bytes(n_layers)) receives the layers' kernel parameters, so it
 * must not be reused until the call's kernels have run.  The bytes stored are those of n_layers
 * kv_quant_append calls.  Pages are reserved layer by layer: OSCAR_ENOPAGES for layer l leaves
 * layers 0 .. l - 1 with pages reserved for the new tokens but no token appended anywhere.
 * Errors: OSCAR_EINVAL, OSCAR_EALIGN, OSCAR_EWORKSPACE, OSCAR_ENOPAGES, OSCAR_ECUDA.
 * Source: the fused write path of the axbrief.com OSCAR page, section "attention-statistics
 * rotation + Triton kernels", applied to every layer's cache. */
size_t kv_quant_append_layers_workspace_bytes(int32_t n_layers);
int kv_quant_append_layers(oscar_cache *const *caches, int32_t n_layers, const void *const *k,
                           const void *const *v, const int32_t *new_tokens, const float *const *rk,
                           void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------- read path
 * oscar_decode_attention: one decode query per request and query head against every
 * token the request holds.  q (device, [batch, num_q_heads, 128], OSCAR_DTYPE_F32 or
 * OSCAR_DTYPE_BF16) is unrotated; rk as for kv_quant_append.  out (device,
 * [batch, num_q_heads, 128], out_dtype) receives softmax(q K^T / sqrt(128)) V over the
 * BF16 sink + window tokens (plain q) and the INT2 tokens (q . R_K against the
 * dequantised rotated keys, which equals inverse-rotating every key because R_K is
 * orthogonal).  The INT2 pages are unpacked and dequantised on chip; no dequantised
 * copy reaches global memory.  Requests with length 0 get zeros.
 * workspace (device, >= oscar_decode_workspace_bytes(c) bytes, 16-byte aligned) holds
 * the rotated queries and the split-K partial results; it needs no initialisation.
 * Numeric range: any finite query and any stored scale.  The tensor-core kernel scales each
 * (request, KV head)'s queries by a power of two before splitting them into fp16 high and low
 * parts, and keeps every P' = p * s_V below 2^15 by lowering its reference maximum as larger value
 * scales appear, so neither operand overflows fp16.  Its one precision limit: inside one
 * (request, KV head), tokens whose value scale is more than about 2^21 times smaller than the
 * largest value scale streamed before them by the same warp get fewer significant bits in P'
 * (fp16 subnormals); their share of the output is that much smaller too.
 * Source: axbrief.com OSCAR page, section "attention-statistics rotation + Triton
 * kernels" (fused read path). */
size_t oscar_decode_workspace_bytes(const oscar_cache *c);
int oscar_decode_attention(oscar_cache *c, const void *q, int32_t q_dtype, const float *rk,
                           void *out, int32_t out_dtype, void *workspace, size_t workspace_bytes,
                           void *stream);

/* oscar_decode_step: one decode step of every request, the write path and the read path in one
 * call.  It appends one token per request (k, v: device, bf16, [batch, num_kv_heads, 128], as for
 * kv_quant_append with new_tokens[b] = 1 for every b) and then runs oscar_decode_attention with q
 * (all arguments as there).  The result, the cache contents and the errors are the same as those
 * of the two calls in a row, bit for bit; on the warp-MMA path the append runs inside the first
 * attention kernel (the leaving key is rotated with the same R_K loads as the queries) instead of
 * in launches of its own.  On the SIMT path it makes the two calls.  Argument, capacity and
 * alignment errors are found before anything is enqueued and leave the cache unchanged.
 * Source: axbrief.com OSCAR page, section "attention-statistics rotation + Triton kernels" (the
 * rotated, quantised write path and the fused read path); joining them into one step is this
 * library's scheduling, not something the page describes. */
int oscar_decode_step(oscar_cache *c, const void *k, const void *v, const void *q, int32_t q_dtype,
                      const float *rk, void *out, int32_t out_dtype, void *workspace,
                      size_t workspace_bytes, void *stream);

/* oscar_decode_step_host: oscar_decode_step with the step's inputs and output in host memory.  It
 * enqueues on stream the copies of k_host and v_host (bf16 [batch, num_kv_heads, 128]) and q_host
 * (q_dtype [batch, num_q_heads, 128]) into the device buffer staging, oscar_decode_step on those
 * copies, and the copy of the output (out_dtype [batch, num_q_heads, 128]) to out_host.  Nothing
 * waits: out_host holds the result once the stream has passed the call (synchronise the stream, or
 * an event recorded after the call).  Host buffers in page-locked memory keep the copies
 * asynchronous; pageable memory works, but its copies wait for the host.  staging (device, 16-byte
 * aligned, >= oscar_decode_step_host_staging_bytes(c, q_dtype, out_dtype) bytes; 0 for invalid
 * arguments) must not be reused until the stream has passed the call.  Results, cache contents and
 * errors are those of oscar_decode_step on device copies of the inputs; argument errors
 * (OSCAR_EINVAL for a NULL host pointer, OSCAR_EWORKSPACE for a short staging buffer) are found before
 * anything is enqueued. */
size_t oscar_decode_step_host_staging_bytes(const oscar_cache *c, int32_t q_dtype, int32_t out_dtype);
int oscar_decode_step_host(oscar_cache *c, const void *k_host, const void *v_host, const void *q_host,
                           int32_t q_dtype, const float *rk, void *out_host, int32_t out_dtype, void *staging,
                           size_t staging_bytes, void *workspace, size_t workspace_bytes, void *stream);

/* oscar_prefill_attention: attention of the queries of a chunk of new tokens (chunked prefill).
 * Each request b must have just appended its last n_q[b] tokens (host array, 0 <= n_q[b] <= 256 and
 * <= its length) through kv_quant_append; q (device, [sum_b n_q[b]][num_q_heads][128], requests in
 * order, tokens in position order; OSCAR_DTYPE_F32 or OSCAR_DTYPE_BF16) holds their queries, and
 * out (device, same layout, out_dtype) receives, for the query at position p, softmax attention over
 * the request's cached positions 0 .. p, each in the precision the cache holds it in after the append
 * (BF16 sink and window, INT2 history): with at most 256 new tokens every INT2 token precedes every
 * query, so the causal limit only cuts the BF16 window.  The queries of a request are processed in
 * groups of up to 16 / G that share every unpacked page (as extra head rows of the decode kernels).
 * workspace (device, >= oscar_prefill_workspace_bytes(c), 16-byte aligned).  Requires the
 * warp-MMA decode path (OSCAR_EINVAL otherwise).  Errors: OSCAR_ERANGE (an n_q out of range),
 * OSCAR_EWORKSPACE, OSCAR_EALIGN, OSCAR_EINVAL.
 * Source: techllm.github.io page, section "OSCAR" (the mixed-precision paged cache serves long
 * prompts); the causal view of a cache that holds the chunk in mixed precision is this library's
 * reading (the pages do not describe prefill attention). */
size_t oscar_prefill_workspace_bytes(const oscar_cache *c);
int oscar_prefill_attention(oscar_cache *c, const void *q, int32_t q_dtype, const int32_t *n_q,
                            const float *rk, void *out, int32_t out_dtype, void *workspace,
                            size_t workspace_bytes, void *stream);

/* Which decode kernel oscar_decode_attention runs (process-wide; default OSCAR_PATH_WARP_MMA):
 * OSCAR_PATH_WARP_MMA: every warp streams its own contiguous run of INT2 pages through a
 *                      bulk-async-copy ring and runs scores and P.V on warp-level tensor-core
 *                      MMAs (mma.sync m16n8k16, fp16 in, fp32 accumulate) with the 2-bit
 *                      codes turned into MMA operands in registers;
 * OSCAR_PATH_SIMT:     one CTA per split, CUDA-core dot products (the baseline the tensor-core
 *                      path is measured against).
 * Both give the same result within the parity tolerance.  Any other value: OSCAR_EINVAL. */
#define OSCAR_PATH_SIMT 1
#define OSCAR_PATH_WARP_MMA 2
int oscar_set_decode_path(int32_t path);
/* Per-launch device time of the INT2 attention kernel of oscar_decode_attention (the warp-MMA
 * kernel, or the split kernel on the SIMT path), from two CUDA events recorded on the caller's
 * stream around that one launch.  oscar_kernel_timing(c, n) creates 2n events (host-side event
 * objects, no device memory) and records the next n decode calls on c; n = 0 stops and frees
 * them.  oscar_kernel_timing_read waits for the recorded events, writes up to max_n durations in
 * milliseconds (call order) to the host array ms, sets *n_out and starts a new record.  Calls
 * beyond the n recorded ones are not timed.  Not a counterpart of anything on the OSCAR pages: a
 * measurement aid. */
int oscar_kernel_timing(oscar_cache *c, int32_t capacity);
int oscar_kernel_timing_read(oscar_cache *c, float *ms, int32_t max_n, int32_t *n_out);
/* Synchronise `stream` and report whether the last decode or prefill call that used `workspace`
 * completed normally (OSCAR_OK) or one of its bounded in-kernel waits gave up
 * (OSCAR_ETIMEOUT; its output is then undefined).  The flag is the workspace's first word. */
int oscar_decode_status(const void *workspace, size_t workspace_bytes, const oscar_cache *c,
                        void *stream);
/* Limit of the bounded waits inside the decode kernels (process-wide): a wait for a page copy
 * gives up after one test and then `iters` tests that may each sleep up to 1 ms (default 2000,
 * about 2 s), sets the error word that oscar_decode_status / oscar_decode_status_noalloc read and
 * ends that warp's work.  Copies already in flight are always waited for (about 2 s at most)
 * before a warp exits.  iters = 0 makes a wait give up at its first failed test, which lets a
 * test exercise the timeout path without a fault; iters < 0 restores the default.  Not a
 * counterpart of anything on the OSCAR pages.  Errors: OSCAR_EINVAL (iters > 1000000). */
int oscar_set_wait_limit(int32_t iters);
/* Timeout-path check (process-wide, default off): with on != 0, the first kernel of every
 * warp-MMA decode call also makes one bounded wait on a shared-memory barrier that nothing
 * arrives at.  It runs out after the wait limit above, sets the same error word a page copy that
 * never lands would set (so oscar_decode_status / oscar_decode_status_noalloc report
 * OSCAR_ETIMEOUT), and the call otherwise completes normally.  It lets a test exercise the
 * timeout reporting without any fault; it is not for production use.  No counterpart on the
 * OSCAR pages.  Always returns OSCAR_OK. */
int oscar_set_wait_probe(int32_t on);

/* oscar_decode_attention_noalloc: oscar_decode_attention without a workspace argument, for
 * callers that cannot allocate device memory at the time they run attention: code executing
 * inside a host-side framework hook that forbids allocation (an inference-engine plugin's
 * enqueue, a real-time loop that must not touch the allocator), or a process whose device
 * memory is already fully reserved by another runtime.  No counterpart on the OSCAR pages: it
 * is a deployment convenience of this library.
 * Scratch comes from one fixed 16 MiB array in the library's device code, which every GPU that
 * loads the library holds until the process exits.  A call whose scratch (rotated queries,
 * split-K partials, an error word) would not fit returns OSCAR_ESCRATCH and enqueues nothing;
 * e.g. 32 requests x 64 query heads (8 KV heads) need about 10.5 MiB.  It always uses the
 * warp-level MMA decode kernel and gives the same result as oscar_decode_attention on that path.
 * It calls no cudaMalloc / cudaFree and no allocating library routine.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with that device current,
 * so make that first call before any stream capture.  All calls share the array and it keeps
 * the last call's contents: calls that may run at the same time on the GPU (other streams,
 * other threads, two caches) race on it and must be serialised by the caller.  Nothing in the
 * array has to start at zero: the one word that must (the flag a bounded in-kernel wait sets
 * when it gives up) is cleared by each call before its kernels read it.  That flag sits at a
 * fixed place in the array; oscar_decode_status_noalloc reads it.  Like the other decode calls,
 * this one first uploads any page-table entries and lengths that changed on the host since the
 * last upload (cudaMemcpyAsync from the handle's host memory); a caller that wants the call to
 * issue no host-to-device copy calls kv_page_table_sync beforehand.  q, rk, out and the dtypes
 * are as for oscar_decode_attention. */
int oscar_decode_attention_noalloc(oscar_cache *c, const void *q, int32_t q_dtype, const float *rk,
                                   void *out, int32_t out_dtype, void *stream);
/* Synchronise `stream` and report whether the last oscar_decode_attention_noalloc call on the
 * current device completed normally (OSCAR_OK) or one of its bounded in-kernel waits gave up
 * (OSCAR_ETIMEOUT; its output is then undefined).  Allocates nothing.  No counterpart on the OSCAR
 * pages. */
int oscar_decode_status_noalloc(void *stream);

/* ---------------------------------------------------------------- calibration
 * oscar_build_rk: R_K = U_Q * H_Had * P_br for num_kv_heads heads from n query samples
 * per head.  q (device, fp32, [num_kv_heads][n][128]) are unrotated query samples;
 * rk (device, fp32, [num_kv_heads][128][128]) receives R_K (row vectors: k~ = k . R_K).
 * C_Q = (1/n) sum q^T q is accumulated in fp64, U_Q (eigenvalues descending, each
 * eigenvector signed so its largest-magnitude entry is positive) comes from a parallel
 * cyclic Jacobi eigen-solver in fp64, H_Had[i][j] = (-1)^popcount(i & j) / sqrt(128),
 * P_br[i][j] = [j == bitrev7(i)].  workspace >= oscar_build_rk_workspace_bytes(heads).
 * Given rows of S V instead (the attention outputs of calibration queries: score-weighted
 * values, S the softmax scores), the same computation builds the value rotation
 * R_V = U_S * H_Had * P_br, because C_S = (1/N) V^T S^T S V is their covariance.  The library
 * stores values as given, so R_V is folded into the value and output projections offline.
 * Source: axbrief.com OSCAR page, section "attention-statistics rotation + Triton
 * kernels"; techllm.github.io page, section "OSCAR" (Hadamard + bit reversal). */
size_t oscar_build_rk_workspace_bytes(int32_t num_kv_heads);
int oscar_build_rk(const float *q, int64_t n, int32_t num_kv_heads, float *rk, void *workspace,
                   size_t workspace_bytes, void *stream);

/* Streaming calibration of R_K (the same C_Q, eigen-solver and assembly as oscar_build_rk, for
 * more query samples than one call holds, or samples that arrive over time).  The accumulator
 * (device, oscar_cq_accumulator_bytes(num_kv_heads) bytes, 16-byte aligned, caller-owned) holds
 * per KV head the fp64 sums of q^T q (128 x 128) and the sample count.  oscar_cq_reset zeroes it;
 * oscar_cq_accumulate adds n samples per head (q: device, fp32, [num_kv_heads][n][128]; n = 0 is a
 * no-op); oscar_cq_finalize divides by the count and writes R_K (rk: device, fp32,
 * [num_kv_heads][128][128]) using workspace >= oscar_build_rk_workspace_bytes(num_kv_heads).  The
 * accumulator is left unchanged, so more samples can be added and R_K refreshed.  At least one
 * sample per head must have been added before finalizing (otherwise R_K is undefined).
 * Source: axbrief.com OSCAR page, section "attention-statistics rotation + Triton kernels"
 * (C_Q = (1/N) sum_n q_n^T q_n); the splitting into calls is this library's. */
size_t oscar_cq_accumulator_bytes(int32_t num_kv_heads);
int oscar_cq_reset(void *acc, int32_t num_kv_heads, void *stream);
int oscar_cq_accumulate(const float *q, int64_t n, int32_t num_kv_heads, void *acc, void *stream);
int oscar_cq_finalize(const void *acc, int32_t num_kv_heads, float *rk, void *workspace,
                      size_t workspace_bytes, void *stream);

/* Calibration samples of the value rotation R_V: the rows of S V, y_i = sum_t s_it v_t with
 * s_i = softmax(q_i k^T / sqrt(128)), for n calibration queries against t_keys keys and values per
 * KV head (q: [num_kv_heads][n][128], k, v: [num_kv_heads][t_keys][128], y: [num_kv_heads][n][128];
 * all device fp32, 16-byte aligned).  Their covariance is the page's score-weighted value
 * covariance C_S = (1/N) V^T S^T S V, so oscar_build_rk (or the streaming calls above) given y
 * builds R_V = U_S H_Had P_br.  Logits in fp32, sums of p and p v in fp64.
 * Errors: OSCAR_ERANGE (n < 1, t_keys < 1 or t_keys > 8192), OSCAR_EINVAL, OSCAR_EALIGN.
 * Source: axbrief.com OSCAR page, section "attention-statistics rotation + Triton kernels"
 * (value rotation from the score-weighted value covariance, absorbed into W_V / W_O). */
int oscar_score_weighted_values(const float *q, int64_t n, const float *k, const float *v,
                                int32_t t_keys, int32_t num_kv_heads, float *y, void *stream);

/* ---------------------------------------------------------------- readback (synchronous)
 * Copy n INT2 tokens of request b, KV head h, starting at position pos0 (each position
 * must lie in the INT2 history) into host buffers, in the per-token logical format:
 * codes [n][32] bytes (channel 4i+j in bits 2j..2j+1 of byte i) and scale/min
 * [n][2 * 128 / group] fp16 bit patterns (s0, m0, s1, m1 for groups of 64; s, m for groups of
 * 128), for K and V.  Any host pointer may be NULL.  Synchronises `stream`. */
int oscar_read_int2(const oscar_cache *c, int32_t b, int32_t h, int64_t pos0, int64_t n,
                    uint8_t *k_codes, uint16_t *k_sm, uint8_t *v_codes, uint16_t *v_sm,
                    void *stream);
/* Copy n BF16 tokens (sink or window positions, each must be held in BF16) of request b,
 * KV head h from pos0 into host buffers k, v ([n][128] bf16 bit patterns; NULL allowed). */
int oscar_read_bf16(const oscar_cache *c, int32_t b, int32_t h, int64_t pos0, int64_t n,
                    uint16_t *k, uint16_t *v, void *stream);

/* ---------------------------------------------------------------- diagnostics */
const char *oscar_strerror(int code);
int oscar_last_cuda_error(void);
/* Kernel launches issued by this process so far (all entry points). */
int64_t oscar_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* OSCAR_KV_H */
