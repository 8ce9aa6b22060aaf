/*
 * pagedkv.h -- C ABI of the GB300 (sm_103a) paged KV decode library.
 *
 * One decode step of grouped-query attention (GQA) for a batch of sequences,
 * each with one new query token, over a KV cache stored in fixed-size pages
 * that sequences reach through their own page-table rows (rows may share
 * pages, e.g. a common prompt prefix), plus the append of the step's new K/V
 * rows into the page pool.  Around it: the rotary embedding (with an optional
 * per-head RMS norm) fused into the append, a shared-prefix decode that reads
 * a common prefix once per KV head, several causal query tokens per sequence,
 * and a host radix cache of prompt prefixes over the pool.
 *
 * Where the operations are defined (page title, section):
 *   - CacheIR, "Compiler Example": the decode graph lowers attention into
 *     fused_rmsnorm_qkv_rope followed by paged_attention_decode over the cached
 *     keys and values.
 *   - CacheIR, "Current Capabilities" (Runtime row) and "Boundaries":
 *     persistent shared page-backed KV pools, batched decode over shared page
 *     tables, multi-batch page-table decode attention with GQA mapping, a
 *     batched paged-attention ABI and a reduced paged-attention decode.
 *   - TorchInferno, "Runtime Scaffolds": runtime.paged (page-table KV allocation
 *     and materialization) and runtime.paged_attention (the paged attention
 *     reference); "Custom Kernels": paged_decode_attention and
 *     batched_paged_decode_attention; "OpenAI-Compatible Serving" knob list:
 *     KV-append, grouped and streaming (block-S) decode attention kernels.
 *   - Experimental LibTorch prefix cache, "Identity, ownership and output
 *     behavior": stream-ordered work, caller-owned lifetimes, host-side
 *     validation before launch and rejection of aliased output storage.
 *
 * Math (the plain reading; the pages print no formula): for sequence b with
 * context length L_b and query head hq,
 *     s_t = scale * <q[b][hq], k_t>,       t = 0 .. L_b - 1
 *     out[b][hq] = sum_t softmax(s)_t * v_t     (out = 0 when L_b = 0)
 * where k_t, v_t are row (t % P) of page page_table[b][t / P] for KV head
 * hq / (n_q_heads / n_kv_heads).  Arithmetic is fp32 with fp16/bf16 inputs;
 * the output is rounded to the input dtype (round to nearest even).
 *
 * Conventions for every call
 * --------------------------
 *   Pointers marked (device) are CUDA device pointers owned by the caller; the
 *   library never frees them and keeps no reference after the call returns
 *   (except pools created with borrowed memory, see kv_pool_create).  Pointers
 *   marked (host) are ordinary host memory.  All device work is enqueued on
 *   `stream` (a cudaStream_t; NULL = the legacy default stream) and nothing
 *   synchronises the host except pkv_read_device_status.
 *   Layouts (row-major, contiguous):
 *     q, out          [batch][n_q_heads][head_dim]
 *     k_pool, v_pool  [num_pages][n_kv_heads][page_size][head_dim]
 *     page_table      int32 [batch][table_stride]   (entries past the pages a
 *                                                    sequence uses are ignored)
 *     context_lens    int32 [batch]   tokens attended, including the new one
 *     k_new, v_new    [batch][n_kv_heads][head_dim]
 *     positions       int32 [batch]   slot written by the append; < 0 = skip
 *                                     (a padded batch slot never writes)
 *   Supported: dtype fp16 or bf16 (q, pools, out all the same); head_dim 64 or
 *   128; page_size a multiple of 16, at most 256; n_q_heads a multiple of
 *   n_kv_heads; every device pointer 16-byte aligned.
 *   Errors: argument errors are found on the host before anything is enqueued
 *   and returned as a pkv_status; nothing is launched then.  Errors that depend
 *   on device data (a page id outside [0, num_pages), a context length beyond
 *   table_stride * page_size) are found by the kernels, which skip the bad
 *   access and set bits in a device status word (PKV_DEV_*).  No kernel traps,
 *   asserts or waits without a bound.  No C++ exception crosses this ABI.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* null pointer, bad size or shape */
    PKV_ERR_UNSUPPORTED = 2,   /* valid but not built: head_dim, page_size, dtype */
    PKV_ERR_ALIAS = 3,         /* out overlaps an input */
    PKV_ERR_OUT_OF_PAGES = 4,  /* allocator has too few free pages */
    PKV_ERR_WORKSPACE = 5,     /* workspace missing, too small or misaligned */
    PKV_ERR_CUDA = 6,          /* a CUDA runtime call failed */
    PKV_ERR_DEVICE_CHECK = 7,  /* pkv_read_device_status found a set bit */
    PKV_ERR_REFCOUNT = 8       /* retain/release of a page that is not allocated */
} pkv_status;

typedef enum pkv_dtype { PKV_F16 = 0, PKV_BF16 = 1 } pkv_dtype;

/* Bits of the device status word. */
#define PKV_DEV_BAD_PAGE 0x1u   /* a page id outside [0, num_pages) was skipped */
#define PKV_DEV_BAD_LEN  0x2u   /* a length/position beyond the table row was clamped/skipped */
#define PKV_DEV_TIMEOUT  0x4u   /* a bounded wait on a copy gave up (copy never landed) */
#define PKV_DEV_BAD_PREFIX 0x8u /* a table row does not start with the shared prefix's pages */

typedef struct CUstream_st* pkv_stream; /* same type as cudaStream_t */
typedef struct pkv_pool pkv_pool;       /* opaque */

/* Human-readable name of a status code.  Never NULL. */
const char* pkv_status_string(pkv_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int pkv_version(void);

/* Check of the failure path every copy wait of the decode kernels takes
 * (Experimental LibTorch prefix cache, "Model and operation coverage": a
 * pending producer held by a watchdog rather than waited on forever).  One
 * warp polls, at most `tries` times, an mbarrier that nothing ever completes;
 * when the polls run out it ORs PKV_DEV_TIMEOUT into *status (device, 4 bytes)
 * and writes the wait's duration in ns to *elapsed_ns (device, may be NULL),
 * then returns: nothing traps and the context stays usable.  The decode
 * kernels give up the same way after 2^22 polls and report PKV_DEV_TIMEOUT
 * through pkv_read_device_status.  tries == 0 or status NULL: INVALID_ARG. */
pkv_status pkv_check_bounded_wait(uint32_t tries, uint32_t* status, unsigned long long* elapsed_ns,
                                  pkv_stream stream);

/* ------------------------------------------------------------------------
 * Page pool and host page allocator
 * (CacheIR, "Current Capabilities": persistent shared CUDA page-backed KV
 *  pools; "Boundaries": shared KV page allocator accounting across forked
 *  request sessions; TorchInferno, "Runtime Scaffolds": runtime.paged).
 * ------------------------------------------------------------------------ */

/* Create a pool of num_pages pages, each [n_kv_heads][page_size][head_dim].
 * k_pool / v_pool (device): both NULL -> the pool allocates (cudaMalloc) and
 * owns the memory; both non-NULL -> the pool borrows them (they must stay
 * alive until kv_pool_destroy).  *out receives the handle.  The host
 * allocator starts with every page free.  Errors: INVALID_ARG, UNSUPPORTED,
 * CUDA (allocation failed). */
pkv_status kv_pool_create(int num_pages, int page_size, int n_kv_heads, int head_dim,
                          pkv_dtype dtype, void* k_pool, void* v_pool, pkv_pool** out);

/* Free the handle (and the memory, if owned).  NULL is accepted.  The caller
 * must make sure no enqueued work still uses owned memory. */
pkv_status kv_pool_destroy(pkv_pool* pool);

/* Device base addresses of the K and V pools (NULL for a NULL handle). */
void* kv_pool_k(const pkv_pool* pool);
void* kv_pool_v(const pkv_pool* pool);

/* Take n free pages (all or nothing); ids_out (host) receives n page ids, each
 * with reference count 1.  Errors: INVALID_ARG, OUT_OF_PAGES (nothing taken).
 * Thread-safe. */
pkv_status kv_pool_alloc_pages(pkv_pool* pool, int n, int32_t* ids_out);

/* Add one reference to each listed page (sharing a prefix page with another
 * sequence).  ids (host).  All ids are checked first; on REFCOUNT or
 * INVALID_ARG nothing changes.  Thread-safe. */
pkv_status kv_pool_retain_pages(pkv_pool* pool, const int32_t* ids, int n);

/* Drop one reference from each listed page; a page whose count reaches zero
 * returns to the free list.  All ids are checked first (an id listed more
 * times than its count, or a free page, is REFCOUNT and nothing changes).
 * Thread-safe. */
pkv_status kv_pool_release_pages(pkv_pool* pool, const int32_t* ids, int n);

/* Number of free pages; -1 for a NULL handle. */
int kv_pool_free_count(const pkv_pool* pool);

/* Reference count of one page (0 = free); -1 for a bad handle or id. */
int kv_pool_refcount(const pkv_pool* pool, int32_t page_id);

/* Pool geometry (any output pointer may be NULL). */
pkv_status kv_pool_info(const pkv_pool* pool, int* num_pages, int* page_size,
                        int* n_kv_heads, int* head_dim, pkv_dtype* dtype);

/* ------------------------------------------------------------------------
 * Prefix cache: a host radix tree of cached prompt prefixes over the pool
 * (TorchInferno, "Runtime Scaffolds": runtime.prefix, a radix prefix tree with
 * prefix-aware lookup, and runtime.prefix_cache; CacheIR, "Current
 * Capabilities": shared KV page allocator accounting across forked request
 * sessions).  Page-granular: only whole pages of tokens are cached and
 * shared, so a sequence's partly filled last page is always its own.  The
 * cache holds one pool reference per cached page; a match hands the caller
 * one more reference per matched page (release them with
 * kv_pool_release_pages when the sequence ends).  Thread-safe; takes the
 * cache's lock, then the pool's.  Not on the GPU path.
 * ------------------------------------------------------------------------ */
typedef struct pkv_prefix_cache pkv_prefix_cache; /* opaque */

/* A cache over `pool` (which must outlive it).  *out receives the handle. */
pkv_status pkv_prefix_cache_create(pkv_pool* pool, pkv_prefix_cache** out);

/* Release every cached page reference and free the cache (NULL: no-op). */
pkv_status pkv_prefix_cache_destroy(pkv_prefix_cache* cache);

/* Record that the first n_tokens/page_size full pages of `tokens` (host int32
 * token ids) are stored in pages[0 ..] (host int32 page ids, the sequence's
 * table row, each held by the caller).  Pages of a prefix already cached are
 * left as they are (the first insertion wins); new ones gain the cache's
 * reference.  *n_new (nullable): pages newly cached.  Errors: INVALID_ARG
 * (page id outside the pool), REFCOUNT (a new page that is not allocated);
 * on an error nothing is cached. */
pkv_status pkv_prefix_cache_insert(pkv_prefix_cache* cache, const int32_t* tokens, int n_tokens,
                                   const int32_t* pages, int* n_new);

/* Longest cached prefix of `tokens` in whole pages, at most max_pages: writes
 * its page ids to pages_out (host) and their count to *n_pages, and retains
 * each for the caller.  A new sequence's table row can start with them. */
pkv_status pkv_prefix_cache_match(pkv_prefix_cache* cache, const int32_t* tokens, int n_tokens,
                                  int32_t* pages_out, int max_pages, int* n_pages);

/* Free up to n_pages cached pages: least recently used leaves whose page only
 * the cache still references (a leaf's parent becomes a leaf in turn; a page
 * that another thread releases during the call waits for the next call).
 * O(cached pages + n_pages log cached pages).  *n_freed (nullable): pages
 * returned to the pool. */
pkv_status pkv_prefix_cache_evict(pkv_prefix_cache* cache, int n_pages, int* n_freed);

/* Pages currently cached (-1 for NULL). */
int pkv_prefix_cache_pages(const pkv_prefix_cache* cache);

/* Counters of a cache since its creation or the last reset (CacheIR,
 * "Current Capabilities": prefix-cache reuse with hit/miss counters).  A
 * lookup is one successful pkv_prefix_cache_match; it asks for
 * min(max_pages, n_tokens / page_size) whole pages. */
typedef struct pkv_prefix_cache_stats {
    uint64_t lookups;         /* match calls */
    uint64_t hits;            /* lookups that matched at least one page */
    uint64_t misses;          /* lookups that matched none */
    uint64_t pages_hit;       /* pages handed out by matches */
    uint64_t pages_missed;    /* pages asked for and not found */
    uint64_t pages_inserted;  /* pages newly cached by inserts */
    uint64_t pages_evicted;   /* pages returned to the pool by evictions */
} pkv_prefix_cache_stats;

/* Copy the counters to *out (host); reset != 0 zeroes them afterwards, in
 * the same locked step.  INVALID_ARG for a NULL cache or out. */
pkv_status pkv_prefix_cache_get_stats(pkv_prefix_cache* cache, int reset,
                                      pkv_prefix_cache_stats* out);

/* ------------------------------------------------------------------------
 * Per-step KV append
 * (TorchInferno, "OpenAI-Compatible Serving" knob list: KV-append kernel;
 *  CacheIR, "Compiler Example": the new K/V are written before the paged
 *  decode; TorchInferno, "Quickstart": a padded slot must never alias a live
 *  KV row).
 * ------------------------------------------------------------------------ */

/* For every b with positions[b] >= 0 and every KV head h, copy k_new[b][h][:]
 * and v_new[b][h][:] bit for bit into row positions[b] % page_size of page
 * page_table[b][positions[b] / page_size].  k_new, v_new, page_table,
 * positions (device).  dev_status (device, nullable): a uint32 that receives
 * PKV_DEV_BAD_PAGE / PKV_DEV_BAD_LEN bits (ORed in) for skipped rows.
 * Distinct sequences must not append into the same (page, slot).  One kernel
 * launch; batch = 0 launches nothing. */
pkv_status kv_append(const pkv_pool* pool, const void* k_new, const void* v_new,
                     const int32_t* page_table, int table_stride, const int32_t* positions,
                     int batch, uint32_t* dev_status, pkv_stream stream);

/* Rotary embedding of the step's queries and new keys, then the KV append
 * (CacheIR, "Compiler Example": rope(q, k) produces the q and k that
 * attention consumes; TorchInferno, "OpenAI-Compatible Serving" knob list: a
 * fused decode rotary + KV-append kernel).  The pages give no formula; this
 * library uses the rotate-half form of Llama/Mistral/Qwen-style models: in
 * every head, element i (i < D/2) pairs with element i + D/2 and the pair
 * turns by the angle positions[b] * rope_theta^(-2i/D):
 *     y_i = x_i cos a - x_{i+D/2} sin a,   y_{i+D/2} = x_{i+D/2} cos a + x_i sin a.
 * The angle is formed in double (theta^(-2i/D) computed on the host) and
 * reduced modulo 2 pi exactly; cos/sin and the rotation run in fp32 and are
 * rounded once to the pool's dtype (to nearest, ties to even), so each result
 * is within one unit in the last place of the exactly rounded rotation.  q [batch][n_q_heads][D] is
 * rotated into q_out (q_out may be q itself, no other overlap); k_new is
 * rotated and v_new copied into the pool as kv_append does (positions[b] < 0:
 * q is still rotated, nothing is written to the pool).  rope_theta must be
 * finite and > 0 (INVALID_ARG).
 *
 * Optional per-head RMS norm before the rotation (Experimental LibTorch
 * prefix cache, "Current execution limits": Q/K-normalised decoders write
 * normalised keys straight into their attention arenas): with q_norm_weight
 * (k_norm_weight) non-NULL, every q (k_new) row of each head first becomes
 *     n_d = x_d * w_d / sqrt(mean_d(x_d^2) + norm_eps),
 * w [head_dim] in the pool's dtype (device, 2-byte aligned), shared by all
 * heads; the mean square (a compensated fp32 sum of exact squares), 1 / rms
 * and the product are formed in fp32 before the rotation, and the result is
 * still rounded once to the dtype.  Either weight may be NULL (no norm on
 * that side); norm_eps finite and >= 0 when one is set (INVALID_ARG); with
 * norm_eps = 0 an all-zero row has no norm and gives NaN, as the formula
 * does.  One kernel launch. */
pkv_status kv_append_rope(const pkv_pool* pool, const void* q, const void* k_new,
                          const void* v_new, const int32_t* page_table, int table_stride,
                          const int32_t* positions, int batch, int n_q_heads, double rope_theta,
                          const void* q_norm_weight, const void* k_norm_weight, float norm_eps,
                          void* q_out, uint32_t* dev_status, pkv_stream stream);

/* Materialize each sequence's cached rows as a dense block:
 * k_out[b][h][t][:] = k_pool[page_table[b][t / P]][h][t % P][:] (and v) for
 * t < min(context_lens[b], max_len); other rows of k_out/v_out are not
 * written.  k_out, v_out [batch][n_kv_heads][max_len][head_dim] (device).
 * Bit copy (TorchInferno, "Runtime Scaffolds": runtime.paged
 * materialization).  dev_status as for kv_append. */
pkv_status kv_gather(const pkv_pool* pool, const int32_t* page_table, int table_stride,
                     const int32_t* context_lens, int batch, int max_len, void* k_out,
                     void* v_out, uint32_t* dev_status, pkv_stream stream);

/* ------------------------------------------------------------------------
 * Decode attention
 * (CacheIR, "Boundaries": multi-batch page-table decode attention with GQA
 *  mapping, reduced paged-attention decode; TorchInferno, "Custom Kernels":
 *  paged_decode_attention / batched_paged_decode_attention, and the
 *  grouped and streaming block-S decode variants in the serving knob list.)
 *
 * Work split: every (sequence, KV head) is cut into chunks of 16 tokens; the
 * chunks of the whole batch are laid end to end and divided into contiguous
 * ranges, one per worker (a warp), equal to within one chunk.  A worker reads
 * each chunk's K and V once for the whole query group.  A (sequence, KV head)
 * that lies in one worker's range is finished there; one spread over several
 * ranges leaves fp32 partial states (m, l, o) that are merged either by the
 * worker that finishes its last piece (a per-unit counter of finished chunks,
 * in the decode kernel) or by paged_decode_combine (see paged_decode_run's
 * merge).  The ranges, the merge order and so the result bits depend only on
 * the context lengths and the worker count, never on physical page ids or
 * timing: permuting pages or rerunning gives bitwise equal results.
 *
 * num_workers: 0 = automatic (the GPU's SM count x resident warps of the
 * kernel, capped so each worker gets at least 4 chunks); n > 0 = at most n
 * workers (n = 1: one worker walks the whole batch, no partial states).
 *
 * variant: which decode kernel computes the chunks.  Every call of one decode
 * (workspace size, plan, run, combine) must pass the same num_workers and
 * variant: both fix the worker count and the query sub-group size.
 * ------------------------------------------------------------------------ */
typedef enum pkv_decode_variant {
    PKV_VARIANT_AUTO = 0,          /* the tensor-core kernel */
    PKV_VARIANT_CUDA_CORES = 1,    /* fp32 FMA on CUDA cores; K/V chunks by 1-D bulk copies;
                                      query sub-groups of at most 8 heads */
    PKV_VARIANT_TENSOR_CORES = 2,  /* q.k and p.v by warp MMA (m16n8k16, fp32 accumulate);
                                      K/V chunks by swizzled 2-D tensor copies; query
                                      sub-groups of at most 16 heads; P enters the p.v
                                      product in the input dtype (bf16: as a high part
                                      plus a bf16 residual, two MMAs) */
    PKV_VARIANT_TCGEN05 = 3        /* several query tokens per sequence only
                                      (paged_decode_attention_multi), head_dim 128: units
                                      of up to 64 query rows (tokens x heads) on the
                                      fifth-generation tensor cores, one CTA per SM, the
                                      products taken transposed (128 tokens of a block as
                                      the tile's rows), accumulators in tensor memory;
                                      other calls: PKV_ERR_UNSUPPORTED */
} pkv_decode_variant;

/* Bytes of device workspace paged_decode_attention needs for these shapes on
 * the current device with this num_workers and variant.  *bytes receives the
 * size.  Errors: INVALID_ARG, UNSUPPORTED, CUDA (device query failed). */
pkv_status paged_decode_workspace_size(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                       int num_workers, pkv_decode_variant variant,
                                       size_t* bytes);

/* Plan step: validates context_lens on the device (clamping to the table row,
 * flagging PKV_DEV_BAD_LEN), resets the status word and the merge counters,
 * and writes the chunk prefix sums, the worker count and the ranges into the
 * workspace.  One kernel (one CTA). */
pkv_status paged_decode_plan(const int32_t* context_lens, int batch, int n_q_heads,
                             int n_kv_heads, int head_dim, int page_size, int table_stride,
                             int num_workers, pkv_decode_variant variant, void* workspace,
                             size_t ws_bytes, pkv_stream stream);

/* Main step on a workspace prepared by paged_decode_plan with the same shapes,
 * num_workers and variant; every run needs a plan of its own (the plan resets
 * the status word and the merge counters).  The decode kernel (persistent
 * grid of workers; asynchronous copies of K/V chunks into shared memory, fp32
 * online softmax).  Writes out for every (sequence, KV head) finished by one
 * worker, zeros for sequences with no tokens, and partial states for the
 * rest.  merge = 1: the worker that finishes the last piece of a split
 * (sequence, KV head) merges it into out, so out is complete when the kernel
 * ends; merge = 0: split units are left to paged_decode_combine.  Both give
 * bitwise equal out.  merge other than 0 or 1 is INVALID_ARG.  Pools of more
 * than 2^31 - 1 rows (num_pages * n_kv_heads * page_size) are UNSUPPORTED by
 * the tensor-core variant. */
pkv_status paged_decode_run(const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* page_table, int table_stride, int batch,
                            int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                            int num_pages, pkv_dtype dtype, float scale, void* out,
                            void* workspace, size_t ws_bytes, int num_workers,
                            pkv_decode_variant variant, int merge, pkv_stream stream);

/* Combine step after paged_decode_run with merge = 0: for every (sequence,
 * KV head) split over several workers, out = sum_i w_i o_i / sum_i w_i l_i
 * with w_i = 2^(m_i - max m) (partials keep m in base-2 units).  One CTA per
 * (sequence, KV head); unsplit ones exit at once. */
pkv_status paged_decode_combine(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                pkv_dtype dtype, void* out, void* workspace, size_t ws_bytes,
                                int num_workers, pkv_decode_variant variant, pkv_stream stream);

/* The whole decode: plan + run (merge = 0) + combine (three kernels on
 * `stream`, chained with programmatic dependent launch).  q, k_pool, v_pool, page_table,
 * context_lens, out, workspace (device).  out must not overlap q, the pools,
 * the table, the lengths or the workspace (ALIAS).  ws_bytes >=
 * paged_decode_workspace_size(...) (else WORKSPACE).  scale multiplies q.k
 * before the softmax (usually 1/sqrt(head_dim)). */
pkv_status paged_decode_attention(const void* q, const void* k_pool, const void* v_pool,
                                  const int32_t* page_table, int table_stride,
                                  const int32_t* context_lens, int batch, int n_q_heads,
                                  int n_kv_heads, int head_dim, int page_size, int num_pages,
                                  pkv_dtype dtype, float scale, void* out, void* workspace,
                                  size_t ws_bytes, int num_workers, pkv_decode_variant variant,
                                  pkv_stream stream);

/* One whole decode step: the KV append of the step's new rows fused into the
 * plan launch, then the decode and combine kernels (three launches on
 * `stream`, chained with programmatic dependent launch).  Equivalent to
 * kv_append(...) followed by paged_decode_attention(...) on the same stream,
 * with k_pool / v_pool written in place.  k_new, v_new [batch][n_kv_heads]
 * [head_dim] and positions int32 [batch] (device) as for kv_append; every
 * other argument as for paged_decode_attention.  Append errors (bad page id
 * or position beyond the table row) are reported through the workspace status
 * read by pkv_read_device_status.  (CacheIR, "Compiler Example": the new K/V
 * are written into the cache, then paged_attention_decode runs.) */
pkv_status paged_decode_step(const void* k_new, const void* v_new, const int32_t* positions,
                             const void* q, void* k_pool, void* v_pool,
                             const int32_t* page_table, int table_stride,
                             const int32_t* context_lens, int batch, int n_q_heads,
                             int n_kv_heads, int head_dim, int page_size, int num_pages,
                             pkv_dtype dtype, float scale, void* out, void* workspace,
                             size_t ws_bytes, int num_workers, pkv_decode_variant variant,
                             pkv_stream stream);

/* paged_decode_step with the rotary embedding of kv_append_rope applied to q
 * and k_new before the append, in the same plan launch (TorchInferno,
 * "OpenAI-Compatible Serving" knob list: the fused decode rotary + append
 * kernel).  q holds the step's un-rotated queries; the rotated queries are
 * written into `out`, which the decode reads as its query and then overwrites
 * with the attention output (each (sequence, head) row is read before its own
 * result is written).  q_norm_weight, k_norm_weight, norm_eps: the optional
 * per-head RMS norm of kv_append_rope.  Arguments otherwise as for
 * paged_decode_step; rope_theta finite and > 0.  Three launches. */
pkv_status paged_decode_step_rope(const void* k_new, const void* v_new, const int32_t* positions,
                                  const void* q, void* k_pool, void* v_pool,
                                  const int32_t* page_table, int table_stride,
                                  const int32_t* context_lens, int batch, int n_q_heads,
                                  int n_kv_heads, int head_dim, int page_size, int num_pages,
                                  pkv_dtype dtype, float scale, double rope_theta,
                                  const void* q_norm_weight, const void* k_norm_weight,
                                  float norm_eps, void* out, void* workspace, size_t ws_bytes,
                                  int num_workers, pkv_decode_variant variant,
                                  pkv_stream stream);

/* paged_decode_step with the step's inputs and its output in page-locked host
 * memory (cudaHostAlloc / cudaMallocHost / cudaHostRegister, or a pinned torch
 * tensor): k_new, v_new, positions, q, page_table, context_lens and out are
 * HOST pointers; k_pool, v_pool and workspace are device memory as before.
 * No copy engine is used: the plan launch reads the lengths, the new rows,
 * the positions and the table straight from host memory (the append writes
 * the pools as in paged_decode_step) while extra CTAs of the same launch copy
 * q and the page table into the workspace; the decode and combine kernels
 * read those copies and store the result straight into `out`.  On a
 * Grace-Blackwell system these accesses cross NVLink-C2C.  The result is in
 * `out` once the stream's work is done (e.g. after cudaStreamSynchronize);
 * the inputs must stay unchanged until then.  Outputs are bitwise those of
 * paged_decode_step on device copies of the same inputs (same kernels, same
 * schedule).  Each host range is checked at its first and last byte
 * (page-locked, mapped for the current device, contiguous): else INVALID_ARG
 * and nothing is launched.  ws_bytes >= paged_decode_step_host_workspace_size
 * (...) (else WORKSPACE).  Other arguments and errors as for
 * paged_decode_step.  (CacheIR, "Compiler Example": the new K/V are written
 * into the cache, then paged_attention_decode runs; the host-buffer form is
 * this library's.)  Three launches. */
pkv_status paged_decode_step_host(const void* k_new, const void* v_new, const int32_t* positions,
                                  const void* q, void* k_pool, void* v_pool,
                                  const int32_t* page_table, int table_stride,
                                  const int32_t* context_lens, int batch, int n_q_heads,
                                  int n_kv_heads, int head_dim, int page_size, int num_pages,
                                  pkv_dtype dtype, float scale, void* out, void* workspace,
                                  size_t ws_bytes, int num_workers, pkv_decode_variant variant,
                                  pkv_stream stream);

/* Bytes of the workspace of paged_decode_step_host: the decode's own
 * (paged_decode_workspace_size) followed by room for q [batch][n_q_heads]
 * [head_dim] and the page table [batch][table_stride], each from a 256-byte
 * boundary.  Same shape errors as paged_decode_workspace_size;
 * table_stride <= 0 is INVALID_ARG. */
pkv_status paged_decode_step_host_workspace_size(int batch, int n_q_heads, int n_kv_heads,
                                                 int head_dim, int table_stride, int num_workers,
                                                 pkv_decode_variant variant, size_t* bytes);

/* ------------------------------------------------------------------------
 * Shared-prefix decode (CacheIR, "Current Capabilities": batched decode over
 * shared page tables; Experimental LibTorch prefix cache, "Short shared prefix
 * qualification": related requests should share immutable block storage).
 *
 * For a batch whose rows all begin with the same prefix_tokens tokens stored
 * in the same pages (columns 0 .. prefix_tokens/P - 1 of every table row equal
 * to row 0's), the prefix is attended once per KV head for all B*G query rows,
 * each sequence's own tokens are attended as usual, and the two partial states
 * of every (sequence, head) are merged: out equals paged_decode_attention's
 * within the decode tolerance.  The prefix pass runs on 128-row tiles of the
 * fifth-generation tensor cores (tcgen05, accumulators in tensor memory; each
 * prefix chunk is read once per tile) for the tensor-core variant (AUTO), and
 * as a decode of 8-row virtual units on CUDA cores for the CUDA-core variant.
 * prefix_tokens > 0, a multiple of page_size, at most table_stride *
 * page_size (INVALID_ARG); every context_lens[b] >= prefix_tokens (else
 * PKV_DEV_BAD_LEN); rows that do not start with row 0's prefix pages set
 * PKV_DEV_BAD_PREFIX (their results are then wrong).  Both read through
 * pkv_read_device_status(workspace).  Four launches: one holding the plans,
 * the query gather and the prefix check; the prefix pass; the suffix decode;
 * the merge.  The workspace size depends on the device's SM count (the
 * prefix pass is split into one wave of tiles): query it on the device that
 * decodes.
 * ------------------------------------------------------------------------ */
pkv_status paged_decode_prefix_workspace_size(int batch, int n_q_heads, int n_kv_heads,
                                              int head_dim, int num_workers,
                                              pkv_decode_variant variant, size_t* bytes);

pkv_status paged_decode_attention_prefix(const void* q, const void* k_pool, const void* v_pool,
                                         const int32_t* page_table, int table_stride,
                                         const int32_t* context_lens, int batch, int n_q_heads,
                                         int n_kv_heads, int head_dim, int page_size,
                                         int num_pages, pkv_dtype dtype, float scale,
                                         int prefix_tokens, void* out, void* workspace,
                                         size_t ws_bytes, int num_workers,
                                         pkv_decode_variant variant, pkv_stream stream);

/* ------------------------------------------------------------------------
 * Several query tokens per sequence (speculative or suffix decoding).
 * (Experimental LibTorch prefix cache, "Current execution limits": causal
 * suffix queries of a request, from one up to 64, attended in tiles of 16
 * queries per warp.)
 *
 * q and out [batch][n_queries][n_q_heads][head_dim]; the n_queries new tokens
 * of sequence b are its last ones (already in the cache), so query j stands at
 * position context_lens[b] - n_queries + j and attends causally to tokens
 * 0 .. context_lens[b] - n_queries + j; a query with no such token (when
 * context_lens[b] < n_queries - j) gives zeros.  A unit of work is the query
 * rows one warp serves, up to 32 (two m16 tiles sharing each K/V chunk): the
 * queries are cut into the fewest tiles of at most 32 tokens (equal sizes but
 * the last), and a tile of t tokens takes the most heads h of the GQA group
 * with t * h <= 32; every K/V chunk of a KV head is read once per (tile, head
 * block).  1 <= n_queries <= 64 (else UNSUPPORTED);
 * tensor-core variant only (CUDA_CORES: UNSUPPORTED).  n_queries = 1 is
 * paged_decode_attention.  Three launches.
 * ------------------------------------------------------------------------ */
pkv_status paged_decode_multi_workspace_size(int batch, int n_queries, int n_q_heads,
                                             int n_kv_heads, int head_dim, int num_workers,
                                             pkv_decode_variant variant, size_t* bytes);

pkv_status paged_decode_attention_multi(const void* q, const void* k_pool, const void* v_pool,
                                        const int32_t* page_table, int table_stride,
                                        const int32_t* context_lens, int batch, int n_queries,
                                        int n_q_heads, int n_kv_heads, int head_dim,
                                        int page_size, int num_pages, pkv_dtype dtype,
                                        float scale, void* out, void* workspace, size_t ws_bytes,
                                        int num_workers, pkv_decode_variant variant,
                                        pkv_stream stream);

/* ------------------------------------------------------------------------
 * Decode without a caller-provided workspace.
 * (No counterpart on the source pages: an addition of this library.)
 *
 * Some callers cannot allocate device memory at the point where they decode:
 * a serving loop that forbids allocation after warm-up (cudaMalloc / cudaFree
 * may synchronise the device and stall every stream), a plugin or custom op
 * inside a host framework that owns all device memory through its own arena
 * and offers no workspace hook, or an embedded runtime with a fixed memory
 * budget.  This entry point needs no workspace from them: it computes exactly
 * what paged_decode_attention computes (same arguments without workspace and
 * ws_bytes, same kernels), with its workspace taken from a fixed array of
 * PKV_NO_ALLOC_SCRATCH_BYTES bytes that the library defines in device memory.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 *   - Size limit: shapes whose workspace (paged_decode_workspace_size with the
 *     same num_workers and variant) exceeds PKV_NO_ALLOC_SCRATCH_BYTES are
 *     rejected with PKV_ERR_WORKSPACE before anything is launched.
 *   - Every GPU that loads the library holds the array until the process exits.
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current) and caches it; make that first call
 *     before any stream capture.  The cached address belongs to the device's
 *     context of that moment: resetting the device (cudaDeviceReset) after the
 *     first call is not supported.
 *   - Operands must be on the current device: the call runs on it and uses its
 *     array.
 *   - All calls share the one array and it keeps the last call's contents; the
 *     plan kernel of each call rewrites every field that must start fresh (the
 *     header, counters and the status word), so nothing needs clearing by the
 *     caller.  Calls that overlap on the GPU (on different streams, or from
 *     different threads without ordering) race on the array: order them.
 *   - Data errors (page ids outside the pool, lengths beyond the table row)
 *     are skipped and flagged in the array's status word, as in the workspace
 *     of paged_decode_attention; pkv_read_no_alloc_status reads it. */
#define PKV_NO_ALLOC_SCRATCH_BYTES (32u << 20)

pkv_status paged_decode_attention_no_alloc(const void* q, const void* k_pool, const void* v_pool,
                                           const int32_t* page_table, int table_stride,
                                           const int32_t* context_lens, int batch,
                                           int n_q_heads, int n_kv_heads, int head_dim,
                                           int page_size, int num_pages, pkv_dtype dtype,
                                           float scale, void* out, int num_workers,
                                           pkv_decode_variant variant, pkv_stream stream);

/* Copy the status of the last plan/decode/step call on this workspace to
 * *status_out (host): the OR of the PKV_DEV_* bits of its kernels.  This call
 * synchronises with the device.  Returns DEVICE_CHECK when any bit is set,
 * OK otherwise (CUDA on a failed copy). */
pkv_status pkv_read_device_status(const void* workspace, uint32_t* status_out);

/* The same for the last paged_decode_attention_no_alloc call on the current
 * device: the PKV_DEV_* bits in the status word of the library's fixed
 * scratch (which the caller never sees).  Synchronises with the device;
 * returns DEVICE_CHECK when any bit is set, OK otherwise (CUDA on a failed
 * copy or address lookup). */
pkv_status pkv_read_no_alloc_status(uint32_t* status_out);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
