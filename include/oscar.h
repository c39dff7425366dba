/*
 * oscar.h - C ABI of the GB300 (sm_103a) OSCAR INT2 rotated paged KV cache.
 *
 * OSCAR ("Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
 * Quantization", arXiv 2605.17757) keeps a paged KV cache in which the first
 * ("sink") and the most recent tokens stay BF16 and the middle history is
 * stored as INT2 after a fixed per-layer rotation R = U . H_Had . P_br and
 * clipping (gist.science technical summary, section 2.2 B; arXiv abstract).
 * This library is the serving hot path: the write into pages, the append that
 * evicts the oldest recent token into INT2, and the fused decode attention
 * over the mixed cache.  Calibration (computing R and the clip thresholds,
 * section 2.2 A) is offline and not part of this library.
 *
 * Conventions
 *  - Every call returns oscar_status (0 = OK).  oscar_last_error() gives a
 *    thread-local message for the last failing call on this thread.
 *  - Tensor arguments are DEVICE pointers owned by the caller unless stated
 *    otherwise.  The library keeps no pointer beyond the call, except the two
 *    pools registered at oscar_create.
 *  - Work is enqueued asynchronously on the caller's stream (cudaStream_t
 *    passed as void*; NULL = legacy default stream).  Argument errors are
 *    reported synchronously.  Device-side errors (a page id out of range, a
 *    bounded wait that timed out) set a status word read by
 *    oscar_check_status().
 *  - Row-vector convention: a rotated vector is y = x R, R is d x d float32
 *    row-major (R[i*d + j]), 16-byte aligned (OSCAR_ERR_INVALID otherwise).
 *    Every R_K / R_V argument holds one such matrix per layer call, or, when
 *    the configuration's rotation_per_kv_head is 1, n_kv_heads of them back to
 *    back ([n_kv_heads][d][d], kv head h at R + h*d*d).
 *  - bf16 tensors are uint16 bit patterns of bfloat16.
 *
 * Memory layout (all little-endian)
 *  INT2 page pool: [num_layers][num_pages][n_kv_heads][block], where one
 *  (layer, page, kv head) block of P = page_size tokens is
 *      K codes  [P][d/4] bytes | K (scale, zero) [P][d/32][2] bf16 |
 *      V codes  [P][d/4] bytes | V (scale, zero) [P][d/32][2] bf16
 *  (d = 128, P = 64: 6144 bytes).  History token t of a request lives in page
 *  block_table[b][t / P], slot t % P (absolute-position paging).
 *  K code row (d/4 bytes = d/16 32-bit words): for lane tig in 0..3,
 *  w in [0, d/64), slot x in 0..7, let P8 = 8w + x, g = P8>>2, kt = (P8>>1)&1,
 *  h = P8&1, c = 32g + 16kt + 8h + 2*tig; word tig*(d/64)+w holds channel c
 *  at bits 2x and channel c+1 at bits 16+2x.
 *  V code row (d/8 16-bit half-words): half-word hw, slot s in 0..7 at bits
 *  2s holds channel 64*(hw % (d/64)) + 8s + hw / (d/64).
 *  Quantiser (per token, kv head, group of 32 rotated channels): y clipped to
 *  [-clip, clip]; zero = bf16(min); scale = bf16((max-min)/3);
 *  code = clamp(rne((y - zero)/scale), 0, 3) (all zero if scale == 0);
 *  dequantised value zero + code*scale.
 *
 *  BF16 window slab: [num_layers][max_requests][n_kv_heads][2 (K,V)][S+W][d]
 *  bf16, unrotated.  Sink token t (< S) is at slot t; recent token t is at slot
 *  S + (t - S) mod W.  Token t of a sequence of length n is sink if t < S,
 *  recent if t >= max(S, n - W), history (INT2) otherwise.
 *
 *  BF16 paged pool (comparison kernel only): [num_layers][num_pages]
 *  [n_kv_heads][2 (K,V)][P][d] bf16, token t at block_table[b][t/P], slot t%P.
 */
#ifndef OSCAR_H_
#define OSCAR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t oscar_status;
enum {
  OSCAR_OK = 0,
  OSCAR_ERR_INVALID = -1,     /* bad argument (null pointer, size, sink/recent mismatch) */
  OSCAR_ERR_OOM = -2,         /* page allocator exhausted */
  OSCAR_ERR_CUDA = -3,        /* a CUDA runtime call failed (message in oscar_last_error) */
  OSCAR_ERR_DEVICE = -4,      /* device status word set (bad page id, wait timeout) */
  OSCAR_ERR_UNSUPPORTED = -5  /* shape outside the supported set */
};

enum { OSCAR_DTYPE_F32 = 0, OSCAR_DTYPE_BF16 = 1 };

/* Device status bits reported by oscar_check_status (oscar_device_status). */
enum {
  OSCAR_DEV_BAD_PAGE = 1,     /* block table entry out of [0, num_pages) on a needed page */
  OSCAR_DEV_TIMEOUT = 2,      /* a bounded barrier wait gave up */
  OSCAR_DEV_BAD_LEN = 4,      /* seq_len / start_pos outside [0, max_pages*page_size] */
  OSCAR_DEV_BAD_SLOT = 8      /* req_slot outside [0, max_requests) */
};

typedef struct {
  int32_t num_layers;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t head_dim;          /* 64 or 128 */
  int32_t page_size;         /* 16, 32 or 64 */
  int32_t group_size;        /* 32 */
  int32_t sink;              /* S >= 0 */
  int32_t recent;            /* W >= 1 */
  int32_t max_requests;      /* window-slab slots */
  int32_t max_pages_per_req; /* block-table row capacity used for bounds checks */
  int32_t num_pages;         /* INT2 pages per layer */
  int32_t rotation_per_kv_head; /* 0: one R_K and one R_V per layer, shared by every kv head (the
                                   pages' fixed per-layer rotation): R_K, R_V are [d][d].  1: one
                                   rotation per (layer, kv head): R_K, R_V are [n_kv_heads][d][d],
                                   kv head h rotated by R[h] (a variant of ours; the clip thresholds
                                   stay per layer) */
} oscar_config;

typedef struct oscar_ctx oscar_ctx;

/* Thread-local message of the last failing call ("" if none). */
const char* oscar_last_error(void);

/* Library version string. */
const char* oscar_version(void);

/* Bytes of the INT2 page pool / BF16 window slab / one (page, kv head) block
 * for a configuration; 0 if the configuration is invalid. */
size_t oscar_int2_pool_bytes(const oscar_config* cfg);
size_t oscar_window_slab_bytes(const oscar_config* cfg);
size_t oscar_page_block_bytes(const oscar_config* cfg);

/* Validate cfg and create a context over caller-owned device buffers:
 * int2_pool (oscar_int2_pool_bytes) and window_slab (oscar_window_slab_bytes),
 * both 16-byte aligned (else OSCAR_ERR_INVALID).
 * The context keeps the raw pointers: both buffers must stay allocated until
 * oscar_destroy (and until any captured graph that uses them is destroyed).
 * Either pointer may be NULL for a host-only context (allocator calls work,
 * kernel calls return OSCAR_ERR_INVALID).  Creating a context with buffers
 * allocates a 4-byte device status word and max_requests x n_kv_heads int32
 * counters of the one-launch decode (zero between launches).  OSCAR_ERR_UNSUPPORTED for a shape
 * outside head_dim {64,128}, page_size {16,32,64}, group_size 32,
 * n_q_heads/n_kv_heads in {1,2,4,8}. */
oscar_status oscar_create(const oscar_config* cfg, void* int2_pool, void* window_slab, oscar_ctx** out);
oscar_status oscar_destroy(oscar_ctx* ctx);

/* ---------------------------------------------------------------- host page allocator
 * Source: the OSCAR serving path keeps the INT2 history in a paged cache that is
 * compatible with paged attention and prefix caching (gist.science technical
 * summary, section 2.2 B and section 3; arXiv abstract: fused kernels inside the
 * paged serving engines).  These calls are the page side of that cache: a page
 * is the unit a block table maps, and a refcount lets requests that share a
 * prefix share its pages.
 * Pages are shared by every layer (page id p addresses block p of each layer).
 * A freshly allocated page has refcount 1; a page returns to the free list
 * when its refcount drops to 0.  ids are host arrays.  Host-only: no device
 * work, no stream.  oscar_alloc_pages returns OSCAR_ERR_OOM (and allocates
 * nothing) when fewer than n pages are free; ref/unref of an id outside
 * [0, num_pages) or of a free page returns OSCAR_ERR_INVALID. */
oscar_status oscar_alloc_pages(oscar_ctx* ctx, int32_t n, int32_t* out_ids);
oscar_status oscar_ref_pages(oscar_ctx* ctx, const int32_t* ids, int32_t n);
oscar_status oscar_unref_pages(oscar_ctx* ctx, const int32_t* ids, int32_t n);
oscar_status oscar_page_refcount(oscar_ctx* ctx, int32_t id, int32_t* out_refcount);
oscar_status oscar_free_page_count(oscar_ctx* ctx, int32_t* out_n);

/* Copy the INT2 blocks of n pages of one layer to host memory (a test and
 * debugging aid; the cache itself is transient serving state).  host_dst
 * receives n x [n_kv_heads][block] bytes, page ids[i] at offset i x n_kv_heads
 * x block bytes (the layout above).  Synchronous: it waits for the copies (and
 * so for earlier work on the legacy default stream).  A page id outside
 * [0, num_pages) returns OSCAR_ERR_INVALID and copies nothing.  ids is a host
 * array. */
oscar_status oscar_read_pages(oscar_ctx* ctx, int32_t layer, const int32_t* ids, int32_t n, void* host_dst);

/* Pages a request of length n needs mapped: logical pages 0 .. (n_hist_end-1)/P
 * where n_hist_end = n - recent (0 if no history). */
int32_t oscar_pages_needed(const oscar_config* cfg, int32_t seq_len);

/* Fork request dst off request src at src's current length n (a branch point,
 * as for parallel sampling or a shared prompt).  Source: prefix caching over the
 * INT2 cache (gist.science technical summary, section 2.2 B: the serving kernel
 * stays compatible with prefix caching; section 3: prefix reuse is kept with the
 * compressed cache).  Host block-table rows: src_bt (read),
 * dst_bt (written, capacity max_pages_per_req; unused entries set to -1).
 * History pages that the prefix fills completely are shared (refcount + 1);
 * the page holding the end of the history, if partial, is copied into a newly
 * allocated page (copy-on-write) for every layer; the BF16 window slot of src
 * is copied to dst for every layer.  Copies are enqueued on stream. */
oscar_status oscar_fork_prefix(oscar_ctx* ctx, const int32_t* src_bt, int32_t* dst_bt, int32_t n,
                               int32_t src_slot, int32_t dst_slot, void* stream);

/* ---------------------------------------------------------------- write path
 * Varlen write (prefill or extend) of tokens [start_pos[b], start_pos[b]+len_b)
 * of each request b, len_b = cu_seqlens[b+1] - cu_seqlens[b]; total_tokens =
 * cu_seqlens[batch] (host value, sizes the grid).  K, V: [total_tokens]
 * [n_kv_heads][d] in dtype (OSCAR_DTYPE_BF16 or _F32).  Ring tokens that stop
 * being recent are first quantised from their stored BF16 values into INT2;
 * then each new token goes to the sink slot, the INT2 page (rotate by R_K / R_V
 * = y = x R, clip to [-clip, clip], quantise, pack), or the recent ring.
 * cu_seqlens [batch+1], start_pos [batch], req_slot [batch]: device int32.
 * block_table: device int32 [batch][bt_stride]; every page that receives a
 * history token must be mapped (else OSCAR_DEV_BAD_PAGE and the row is
 * skipped).  R_K, R_V: device float32 [d][d].  Source: rotation and clipping
 * of the history (summary section 2.2 A/B), fused write kernel (abstract). */
oscar_status oscar_write_kv(oscar_ctx* ctx, int32_t layer, const void* K, const void* V, int32_t dtype,
                            const int32_t* cu_seqlens, const int32_t* start_pos, int32_t batch,
                            int32_t total_tokens, const float* R_K, const float* R_V, float clip_K,
                            float clip_V, const int32_t* block_table, int32_t bt_stride,
                            const int32_t* req_slot, void* stream);

/* Same as oscar_write_kv for R = H_Had . P_br (U = I, the data-oblivious
 * Hadamard-only rotation): the rotation runs as a fast Walsh-Hadamard
 * transform instead of a dense product. */
oscar_status oscar_write_kv_hadamard(oscar_ctx* ctx, int32_t layer, const void* K, const void* V, int32_t dtype,
                                     const int32_t* cu_seqlens, const int32_t* start_pos, int32_t batch,
                                     int32_t total_tokens, float clip_K, float clip_V,
                                     const int32_t* block_table, int32_t bt_stride, const int32_t* req_slot,
                                     void* stream);

/* One decode-step append per request.  Source: the sink and most recent
 * tokens stay BF16 and the history is stored as INT2 after the rotation and
 * clipping (gist.science technical summary, section 2.2 B); so when a new token
 * arrives, the oldest recent token leaves the BF16 window and is written into
 * the INT2 history by the fused write path (arXiv abstract: fused write
 * kernel).  K_new, V_new [batch][n_kv_heads][d]
 * (dtype) is token seq_lens_before[b].  If seq_lens_before[b] - W >= S the
 * oldest recent token e = seq_lens_before[b] - W is first quantised from the
 * ring into page block_table[b][e / P] slot e % P; the new token then takes
 * its ring slot (or sink slot if seq_lens_before[b] < S).  The caller maps the
 * page of e beforehand (oscar_pages_needed(seq_lens_before + 1)). */
oscar_status oscar_append_step(oscar_ctx* ctx, int32_t layer, const void* K_new, const void* V_new, int32_t dtype,
                               const int32_t* seq_lens_before, int32_t batch, const float* R_K, const float* R_V,
                               float clip_K, float clip_V, const int32_t* block_table, int32_t bt_stride,
                               const int32_t* req_slot, void* stream);

/* Declare the clip thresholds a layer's INT2 history was written with, for a
 * cache filled outside this library (an uploaded image).  The write and append
 * calls declare theirs implicitly.  The decode kernels feed the history's BF16
 * scales and zeros to f16 tensor-core operands multiplied by 2^k, where k is the
 * largest exponent with clip * 2^k < 2^14 over every clip declared for the
 * layer (the smallest k is kept); INT2 decode of a layer with no declared clip
 * returns OSCAR_ERR_INVALID.  Clips must lie in [2^-86, 16384) (else
 * OSCAR_ERR_UNSUPPORTED, also from the write calls).  Host-only. */
oscar_status oscar_set_layer_clip(oscar_ctx* ctx, int32_t layer, float clip_K, float clip_V);

/* ---------------------------------------------------------------- decode
 * Bytes of decode workspace for batch requests of at most max_seq tokens. */
oscar_status oscar_decode_workspace_size(const oscar_config* cfg, int32_t batch, int32_t max_seq, size_t* bytes);

/* Fused decode attention over the mixed cache (summary section 2.2 B: unpack,
 * dequantise, inverse rotation and attention for the INT2 history; abstract:
 * fused decode kernel).  q: [batch][n_q_heads][d] (q_dtype); out:
 * [batch][n_q_heads][d] float32 (out_dtype F32) or bf16 (BF16).  seq_lens
 * [batch] (device) counts every cached token including the current one; query
 * head h reads kv head h / (n_q_heads / n_kv_heads); softmax scale 1/sqrt(d).
 * The query is rotated once (q' = q R_K) to score the INT2 history in the
 * rotated basis, history values accumulate in the rotated basis, and R_V^T is
 * applied once per output row; sink/recent tokens use q and accumulate
 * unrotated; both share one softmax.  sink/recent must equal the
 * configuration.  max_seq (host) bounds seq_lens and sizes the grid.
 * workspace: device scratch of oscar_decode_workspace_size bytes (256-byte
 * aligned); its contents need no initialisation.  The layer needs a declared
 * clip threshold (a write to it, or oscar_set_layer_clip).  R_K and R_V
 * (device float32 [d][d], the layer's fixed rotations) are read before the
 * kernels wait on the work queued ahead of them: they must not be written by
 * the kernel launched immediately before this call on the stream.
 *
 * Launches (oscar_set_decode_form).  Three kernels: q_rotate, split-K and
 * combine.  One kernel: its split CTAs form the rotated query themselves and
 * the last CTA of each (request, kv head) to finish (an atomic ticket on a
 * counter the context owns; no CTA waits on another) merges that pair's
 * partials and writes its output rows; before its dependency wait it only
 * prefetches into L2.  One-launch calls on one context share its counters: do
 * not run two of them concurrently on different streams (order them with
 * events).  After a failed launch, oscar_check_status also resets the
 * counters. */
oscar_status oscar_decode_attn(oscar_ctx* ctx, int32_t layer, const void* q, int32_t q_dtype, void* out,
                               int32_t out_dtype, const int32_t* block_table, int32_t bt_stride,
                               const int32_t* seq_lens, const int32_t* req_slot, int32_t batch, int32_t max_seq,
                               int32_t sink, int32_t recent, const float* R_K, const float* R_V,
                               void* workspace, size_t ws_bytes, void* stream);

/* One decode step of a layer, fused: append each request's new token and
 * attend over the cache that includes it.  Equivalent to oscar_append_step
 * with seq_lens_before[b] = seq_lens[b] - 1 followed by oscar_decode_attn with
 * seq_lens on the same stream (identical cache contents and outputs), with the
 * same arguments as those two calls (K_new, V_new: [batch][n_kv_heads][d] in
 * kv_dtype; seq_lens [batch] device int32 counts the new token).  The query
 * rotation and the append run as one grid ("step_prep": rotation CTAs first,
 * then append CTAs; no rotation CTAs when the decode is one launch), launched
 * as a programmatic dependent of the preceding kernel; the split-K kernel is
 * its dependent and reads only the page the append may be writing after the
 * dependency resolves.  The caller maps the
 * page of the evicted token beforehand, as for oscar_append_step. */
oscar_status oscar_decode_step(oscar_ctx* ctx, int32_t layer, const void* K_new, const void* V_new, int32_t kv_dtype,
                               const void* q, int32_t q_dtype, void* out, int32_t out_dtype,
                               const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                               const int32_t* req_slot, int32_t batch, int32_t max_seq, int32_t sink, int32_t recent,
                               const float* R_K, const float* R_V, float clip_K, float clip_V, void* workspace,
                               size_t ws_bytes, void* stream);

/* Allocation-free variant of oscar_decode_attn (no counterpart in the OSCAR
 * paper; it exists for callers that cannot allocate device memory).
 *
 * Some callers cannot hand over a workspace: an engine whose device memory is
 * all owned and budgeted by its own allocator, a plugin that must not call
 * cudaMalloc (which can synchronise the device and stall other work), or a
 * serving loop that is forbidden from allocating after start-up.  This call
 * takes the same arguments as oscar_decode_attn minus workspace/ws_bytes and
 * uses scratch in a file-scope device array of 8 MiB that the library keeps on
 * every GPU that loads it, until the process exits.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *  - Limit: the scratch oscar_decode_workspace_size would report for
 *    (batch, max_seq) must be at most 8 MiB (for example batch 1 up to 128K
 *    tokens at 32 q heads); larger calls return OSCAR_ERR_INVALID with a
 *    message and launch nothing.
 *  - The first call on a device looks up the array's device address (with that
 *    device current); make that first call before any stream capture.
 *  - All calls share the one array and it keeps the last call's contents
 *    (nothing in it needs to start at zero).  Calls whose kernels overlap on
 *    the GPU (different streams, or different host threads) race on it:
 *    serialise them. */
oscar_status oscar_decode_attn_noalloc(oscar_ctx* ctx, int32_t layer, const void* q, int32_t q_dtype, void* out,
                                       int32_t out_dtype, const int32_t* block_table, int32_t bt_stride,
                                       const int32_t* seq_lens, const int32_t* req_slot, int32_t batch,
                                       int32_t max_seq, int32_t sink, int32_t recent, const float* R_K,
                                       const float* R_V, void* stream);

/* ---------------------------------------------------------------- extend
 * Extend (chunked prefill) attention over the mixed cache (summary section 2.2 B:
 * the serving kernel handles paged attention and prefix caching over the INT2
 * history; section 3: prefix reuse kept with the INT2 cache).  Request b holds
 * prefix_lens[b] cached tokens and brings len_b = cu_seqlens[b+1] - cu_seqlens[b]
 * new tokens at positions prefix_lens[b] + i.  Query token i of request b
 * attends to every cached token in the form the cache stores it at length
 * prefix_lens[b] (INT2 history dequantised and rotated back, sink and recent
 * tokens BF16) and, causally, to the chunk's tokens 0..i, whose keys and
 * values are the K_new / V_new rows themselves.  Call it before writing the
 * chunk (oscar_write_kv with start_pos = prefix_lens): the cache must hold
 * exactly prefix_lens[b] tokens of request b.
 *  q: [total_tokens][n_q_heads][d] BF16; K_new, V_new: [total_tokens]
 *  [n_kv_heads][d] BF16 (another q_dtype or kv_dtype: OSCAR_ERR_UNSUPPORTED;
 *  the BF16 tiles take the query exactly as a BF16 tensor-core operand);
 *  out: [total_tokens][n_q_heads][d] float32 or bf16 (out_dtype).  q, K_new,
 *  V_new and out 16-byte aligned.  cu_seqlens [batch+1], prefix_lens [batch],
 *  req_slot [batch]: device int32; total_tokens = cu_seqlens[batch] and
 *  max_chunk >= every len_b (host values, they size the grids; a request whose
 *  chunk they do not cover sets OSCAR_DEV_BAD_LEN and gets no output).
 *  block_table [batch][bt_stride] maps the history pages of each prefix (a
 *  missing one sets OSCAR_DEV_BAD_PAGE); R_K, R_V: the layer's rotations
 *  (device float32 [d][d]); the layer needs a declared clip threshold.
 *  n_q_heads / n_kv_heads must divide 128 and batch must not exceed 65535
 *  (else OSCAR_ERR_UNSUPPORTED).
 *  workspace: device scratch of at least oscar_extend_workspace_size(cfg,
 *  total_tokens) bytes (256-byte aligned, no initialisation); it holds q R_K for
 *  every query row and R_V as f16 hi / lo planes (one per kv head with
 *  rotation_per_kv_head) for the epilogue's y R_V^T on the tensor cores.  With
 *  oscar_extend_workspace_size_unpacked(cfg, total_tokens, batch, max_prefix,
 *  max_chunk) bytes or more, the unpacked-prefix form runs: a pre-pass forms
 *  every 64-key tile that the query tiles of a request share (its INT2 history
 *  tiles, dequantised; its BF16 window tiles; its chunk's own tiles) once per
 *  call into the workspace, and the attention CTAs of all the request's query
 *  tiles copy those tiles instead of each forming them from the pages and rows.
 *  The workspace holds the window and chunk tiles for this max_chunk and T INT2
 *  tiles per (request, kv head), T as many as fit; a request with more history
 *  tiles forms its own.  Both forms give identical outputs.  Softmax scale 1/sqrt(d), query
 *  head h reads kv head h / (n_q_heads / n_kv_heads).  Kernels on the stream:
 *  the pre-pass (unpacked form), the query rotation, then the tensor-core
 *  attention (timing name "extend"). */
oscar_status oscar_extend_workspace_size(const oscar_config* cfg, int32_t total_tokens, size_t* bytes);
/* Workspace of the unpacked-prefix form for batch requests whose prefixes hold at
 * most max_prefix tokens and whose chunks at most max_chunk (the max_chunk given
 * to oscar_extend_attn): the base size plus, per (request, kv head), one operand
 * tile (42 KB at d = 128, 26 KB at d = 64) per 64 positions of the INT2 history
 * (672 B per history token and kv head at d = 128, against the cache's 96 B: a
 * working copy for one call), of the BF16 window and of the chunk.  Negative
 * arguments: OSCAR_ERR_INVALID. */
oscar_status oscar_extend_workspace_size_unpacked(const oscar_config* cfg, int32_t total_tokens, int32_t batch,
                                                  int32_t max_prefix, int32_t max_chunk, size_t* bytes);
oscar_status oscar_extend_attn(oscar_ctx* ctx, int32_t layer, const void* q, int32_t q_dtype, const void* K_new,
                               const void* V_new, int32_t kv_dtype, void* out, int32_t out_dtype,
                               const int32_t* cu_seqlens, const int32_t* prefix_lens, int32_t batch,
                               int32_t total_tokens, int32_t max_chunk, const int32_t* block_table, int32_t bt_stride,
                               const int32_t* req_slot, const float* R_K, const float* R_V, void* workspace,
                               size_t ws_bytes, void* stream);

/* One chunked-prefill step of a layer: oscar_extend_attn followed by
 * oscar_write_kv of the same chunk (start_pos = prefix_lens), with the
 * arguments of those two calls on one stream (identical outputs and cache
 * contents).  The write runs after the attention has read the window slots and
 * pages it overwrites.  clip_K and clip_V are declared for the layer first, so
 * the first chunk of a fresh layer may use this call.  The caller maps the pages
 * that the chunk's history tokens (and the ring tokens it evicts) land in,
 * as for oscar_write_kv. */
oscar_status oscar_extend_step(oscar_ctx* ctx, int32_t layer, const void* q, int32_t q_dtype, const void* K_new,
                               const void* V_new, int32_t kv_dtype, void* out, int32_t out_dtype,
                               const int32_t* cu_seqlens, const int32_t* prefix_lens, int32_t batch,
                               int32_t total_tokens, int32_t max_chunk, const int32_t* block_table, int32_t bt_stride,
                               const int32_t* req_slot, const float* R_K, const float* R_V, float clip_K,
                               float clip_V, void* workspace, size_t ws_bytes, void* stream);

/* In-house comparison: standard split-K paged decode over an all-BF16 cache
 * (layout above), same grid and staging as the INT2 kernel.  bf16_pool points
 * at the whole [num_layers][num_pages]... pool; workspace from
 * oscar_bf16_decode_workspace_size. */
oscar_status oscar_bf16_decode_workspace_size(const oscar_config* cfg, int32_t batch, int32_t max_seq,
                                              size_t* bytes);
oscar_status oscar_bf16_decode_attn(oscar_ctx* ctx, int32_t layer, const void* bf16_pool, const void* q,
                                    int32_t q_dtype, void* out, int32_t out_dtype, const int32_t* block_table,
                                    int32_t bt_stride, const int32_t* seq_lens, int32_t batch, int32_t max_seq,
                                    void* workspace, size_t ws_bytes, void* stream);

/* Self-test of the device-side failure path (no counterpart in the OSCAR
 * paper).  Every kernel bounds its mbarrier waits and, when one runs out, sets
 * OSCAR_DEV_TIMEOUT in the status word instead of trapping, so the context
 * stays usable.  This call launches one small kernel that waits on a barrier
 * nothing arrives on until limit_us microseconds (1 .. 1e6) have passed, then
 * sets OSCAR_DEV_TIMEOUT; oscar_check_status reports it and clears it. */
oscar_status oscar_selftest_wait_timeout(oscar_ctx* ctx, int32_t limit_us, void* stream);

/* ---------------------------------------------------------------- status, tracing
 * Synchronise stream, read and clear the device status word.  Returns
 * OSCAR_ERR_DEVICE (bits in *out_bits if non-NULL) if any kernel flagged an
 * error since the last check. */
oscar_status oscar_check_status(oscar_ctx* ctx, void* stream, int32_t* out_bits);

/* ---------------------------------------------------------------- decode launch form
 * How the INT2 decode calls (oscar_decode_attn, oscar_decode_step,
 * oscar_decode_attn_noalloc) launch: OSCAR_DECODE_AUTO (the library's choice
 * for the batch; the default), OSCAR_DECODE_THREE_KERNELS (query rotation,
 * split-K and combine kernels) or OSCAR_DECODE_ONE_LAUNCH (the one-kernel
 * form described at oscar_decode_attn whenever batch <= max_requests, three
 * kernels otherwise).  The forms agree within floating-point rounding (the
 * rotated query is summed in another order).  Host-only; OSCAR_ERR_INVALID
 * for any other value. */
#define OSCAR_DECODE_AUTO 0
#define OSCAR_DECODE_THREE_KERNELS 1
#define OSCAR_DECODE_ONE_LAUNCH 2
oscar_status oscar_set_decode_form(oscar_ctx* ctx, int32_t form);

/* Kernel timing for tracing: when enabled, the library brackets each launch
 * of the named kernel family with CUDA events on the launch stream.
 * oscar_kernel_time returns the summed milliseconds and launch count since the
 * last reset (synchronises the recorded events).  Names: "decode_splitk",
 * "decode_combine", "q_rotate", "step_prep", "append", "evict", "write", "bf16_prepare",
 * "bf16_decode", "bf16_combine", "extend", "selftest".  Launches
 * recorded into a CUDA graph get external event-record nodes: replay the graph
 * once, then read; the events return to the library when read, so a graph
 * captured with timing on is replayed at most once.  With timing on, the decode
 * kernels are launched without programmatic dependent launch. */
oscar_status oscar_set_timing(oscar_ctx* ctx, int32_t enable);
oscar_status oscar_kernel_time(oscar_ctx* ctx, const char* name, double* out_ms, int32_t* out_launches);
oscar_status oscar_reset_timing(oscar_ctx* ctx);

/* Number of kernel launches this context has issued (all families). */
int64_t oscar_launch_count(oscar_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* OSCAR_H_ */
