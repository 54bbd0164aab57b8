/*
 * pagedattn: paged K/V attention for NVIDIA GB300 (sm_103a).
 *
 * A C ABI over hand-written CUDA kernels. Query heads attend over a per-layer
 * pool of fixed-size K/V pages through a per-request block table, without
 * gathering a dense K/V tensor first.
 *
 * Conventions shared by every call:
 *   - All tensors are raw DEVICE pointers to contiguous row-major buffers
 *     owned by the caller. bf16 values are passed as their 16-bit patterns.
 *   - Layouts (Week 3 Day 4: Direct Paged Attention, "The Paged Attention
 *     API" and "How This Maps to tiny-llm"; Tutorial 13: Paged Attention and
 *     Memory Management, section 6 "Paged Attention Metadata"):
 *       query        [B, H_q, L, D]            bf16
 *       out          [B, H_q, L, D]            bf16
 *       key_pages    [P, H_kv, page_size, D]   bf16 (one pool per layer)
 *       value_pages  [P, H_kv, page_size, D]   bf16
 *       block_table  [B, max_pages]            int32, physical page ids
 *       context_lens [B]                       int32, valid tokens per request
 *     Logical position j of request b is slot j % page_size of physical page
 *     block_table[b, j / page_size] (Week 3 Day 4, "Why block_table
 *     Matters"). Entries past ceil(context_lens[b] / page_size) are never
 *     read and may hold anything.
 *   - GQA: query head h_q reads KV head h_q / (H_q / H_kv).
 *   - Causal mask: query row i of request b sits at absolute position
 *     context_lens[b] - L + i (the rows are the newest L positions) and sees
 *     keys 0..that position. With causal = 0 every row sees all
 *     context_lens[b] keys. A row that sees no key returns zeros.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Every call is asynchronous on it; nothing synchronises except
 *     pa_get_device_error.
 *   - Errors: a call that returns anything but PA_OK launched nothing and
 *     touched no buffer. Per-request values that live on the device
 *     (block_table entries, context_lens, slot_mapping) cannot be checked on
 *     the host; the kernels check them, never access memory outside the
 *     buffers for a bad value, and record it in a device error word that
 *     pa_get_device_error reads.
 *   - The library allocates no device memory on any call.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,    /* null pointer, bad size, bad scale, misalignment */
    PA_ERR_UNSUPPORTED = 2,    /* D not 64/128, H_q % H_kv != 0, page_size not a
                                  power of two in 1..256, shapes beyond limits */
    PA_ERR_WORKSPACE = 3,      /* workspace missing or smaller than required    */
    PA_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed          */
    PA_ERR_DEVICE_BOUNDS = 5,  /* a kernel met an out-of-range page id, slot or
                                  context length (from pa_get_device_error)     */
    PA_ERR_DEVICE_TIMEOUT = 6, /* a kernel's bounded wait on its own copies ran
                                  out (from pa_get_device_error)                */
    PA_ERR_NO_PAGES = 7        /* pa_kv_cache: the page pool or a block-table row
                                  is full; nothing was changed                  */
} pa_status;

/* Bits of the device error word reported by pa_get_device_error. */
#define PA_DEVERR_PAGE_ID      0x1u  /* block_table entry outside [0, P)           */
#define PA_DEVERR_SLOT         0x2u  /* slot_mapping entry >= P * page_size         */
#define PA_DEVERR_CONTEXT_LEN  0x4u  /* context_lens entry < 0 or > max_pages*ps    */
#define PA_DEVERR_TIMEOUT      0x8u  /* pipeline wait gave up                       */

/* Problem sizes shared by every call. */
typedef struct pa_shape {
    int32_t batch;         /* B: requests                                       */
    int32_t num_q_heads;   /* H_q (unused by pa_append_kv)                      */
    int32_t num_kv_heads;  /* H_kv, must divide H_q                             */
    int32_t head_dim;      /* D: 64 or 128                                      */
    int32_t q_len;         /* L: query rows per request; for pa_append_kv the
                              number of new tokens per request (L_new)          */
    int32_t num_pages;     /* P: pages in the pool                              */
    int32_t max_pages;     /* row length (stride) of block_table                */
} pa_shape;

/*
 * Write path: scatter new K/V rows into the page pool by slot_mapping.
 * (Reading vLLM's PagedAttention Kernel, 3.2 "Writing into the cache":
 * the flat slot of a token is physical_block * page_size + offset.)
 *
 *   key, value      [B, H_kv, L_new, D] bf16, 16-byte aligned
 *   key_pages, value_pages  [P, H_kv, page_size, D] bf16, modified in place
 *   slot_mapping    [B, L_new] int32. slot < 0: no token (padding), skipped.
 *                   slot >= P * page_size: skipped, PA_DEVERR_SLOT recorded.
 *                   Two tokens with the same slot: undefined which one lands.
 *   shape.q_len = L_new; shape.num_q_heads and shape.max_pages are unused.
 * The copy is bit-exact.
 */
pa_status pa_append_kv(const void *key, const void *value, void *key_pages,
                       void *value_pages, const int32_t *slot_mapping,
                       int32_t page_size, pa_shape shape, void *stream);

/*
 * Bytes of scratch workspace pa_decode needs for `shape` on the CURRENT
 * device (it depends on the device's SM count). 0 on invalid shapes.
 * It holds one partial (max, sum, output) state per block for every segment
 * (request x KV head x tile of 16 query rows; at most 65536 segments) that
 * straddles blocks; its contents on entry do not matter.
 */
size_t pa_decode_workspace_bytes(pa_shape shape);

/*
 * Decode attention: split-KV over the cached context (Week 3 Day 4,
 * "Choose a Schedule for Each Query Shape" and "Task 2": partition the
 * context across parallel workers and merge their partial (max, sum,
 * output) states; Reading vLLM's PagedAttention Kernel, 3.3: partitions
 * computed in parallel and combined afterwards). Any L >= 1 is computed
 * correctly; the schedule is built for small L (one-token decode).
 *
 *   scale            > 0 and finite (the Python binding maps None to 1/sqrt(D))
 *   max_context_len  an upper bound of context_lens used only to size the
 *                    grid (0 = unknown); larger entries are still correct.
 *   workspace        device scratch of at least pa_decode_workspace_bytes
 *                    bytes, 16-byte aligned; any contents. Calls that share a
 *                    workspace must not overlap on the GPU.
 * The work is two kernels on `stream`: the split-KV pass and a small merge
 * pass, chained by programmatic dependent launch (each waits for the kernel
 * before it in the stream before touching any data).
 */
pa_status pa_decode(const void *query, const void *key_pages,
                    const void *value_pages, const int32_t *block_table,
                    const int32_t *context_lens, int32_t page_size, float scale,
                    int causal, void *out, pa_shape shape,
                    int32_t max_context_len, void *workspace,
                    size_t workspace_bytes, void *stream);

/*
 * pa_decode without a caller-provided workspace. (The pages have no
 * counterpart: this entry point exists for callers of this library that
 * cannot allocate device memory, e.g. a host program embedded in another
 * runtime that owns every device allocation and only hands out the input and
 * output pointers, or a serving loop where cudaMalloc/cudaFree are off limits
 * because they can synchronise the device mid-flight.)
 *
 * Same arguments, checks and result as pa_decode, minus the workspace: the
 * scratch is a 32 MiB array inside the library's device image, held by every
 * GPU that loads this part of the library until the process exits. The call
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Shapes whose scratch (pa_decode_workspace_bytes) exceeds 32 MiB are
 *     rejected with PA_ERR_WORKSPACE before anything is launched.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents (the decode needs nothing in it to start at zero).
 *     Calls that overlap on the GPU (other streams, other host threads) race
 *     on the array: order them.
 *   - The array's device address is cached per device for the life of the
 *     process. cudaDeviceReset (or any reset of the device's primary
 *     context) ends the context it was looked up in, and with it the cached
 *     address (and that of the library's device error word): do not call
 *     this library on a device after resetting it in the same process.
 */
pa_status pa_decode_noalloc(const void *query, const void *key_pages,
                            const void *value_pages, const int32_t *block_table,
                            const int32_t *context_lens, int32_t page_size,
                            float scale, int causal, void *out, pa_shape shape,
                            int32_t max_context_len, void *stream);

/*
 * Dense baseline, first step (Week 3 Day 4, "Measure the Direct Page Walk":
 * the dense path gathers each request's cached K/V into contiguous memory
 * before attending; the direct page walk does without this copy). Copies,
 * for every request b, KV head h and position t < context_lens[b], the row
 * pages[block_table[b][t / page_size]][h][t % page_size][:] of key_pages and
 * value_pages into key_dense[b][h][t][:] and value_dense[b][h][t][:].
 *   key_dense, value_dense  device, [B, H_kv, dense_len, D] bf16, 16-byte
 *                           aligned, owned by the caller; rows at or past a
 *                           request's context are not written.
 *   shape                   batch, num_kv_heads, head_dim, num_pages,
 *                           max_pages are used.
 * A block-table entry outside the pool skips its rows and records
 * PA_DEVERR_PAGE_ID; a context longer than dense_len or the block table
 * records PA_DEVERR_CONTEXT_LEN and is cut to fit. Bit copy, one kernel on
 * `stream` (programmatic dependent launch, like pa_append_kv).
 */
pa_status pa_gather_kv(const void *key_pages, const void *value_pages,
                       const int32_t *block_table, const int32_t *context_lens,
                       int32_t page_size, pa_shape shape, int32_t dense_len,
                       void *key_dense, void *value_dense, void *stream);

/*
 * Dense baseline, second step: decode attention over dense K/V buffers
 * [B, H_kv, dense_len, D] (as pa_gather_kv writes them), with the same
 * split-KV kernel, arithmetic and workspace as pa_decode; request b's keys
 * are rows 0 .. context_lens[b] - 1 of its block, no block table is read.
 * On the same K/V values the result is bit-identical to pa_decode's.
 *   dense_len  a multiple of 64, >= every context length (a longer context
 *              records PA_DEVERR_CONTEXT_LEN and is cut to dense_len).
 *   shape      num_pages and max_pages are ignored.
 *   workspace  as for pa_decode (pa_decode_workspace_bytes of the shape).
 */
pa_status pa_decode_dense(const void *query, const void *key_dense,
                          const void *value_dense, const int32_t *context_lens,
                          int32_t dense_len, float scale, int causal, void *out,
                          pa_shape shape, int32_t max_context_len, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * Prefill attention: query rows in tiles, every K/V tile resolved through
 * block_table (Week 3 Day 4, "Task 2", the long-query page-walking
 * schedule), causal by default with the bottom-right offset above. Needs no
 * workspace. Tensor-core kernels (tcgen05, TMEM) for head_dim 128 or 64 and
 * every page size. A KV group of one query head computes that head in both
 * halves of a two-head block. Pages of fewer than 8 tokens are copied into
 * shared memory row by row instead of one TMA box per page.
 */
pa_status pa_prefill(const void *query, const void *key_pages,
                     const void *value_pages, const int32_t *block_table,
                     const int32_t *context_lens, int32_t page_size, float scale,
                     int causal, void *out, pa_shape shape, void *stream);

/*
 * FP8 page pools (Reading vLLM's PagedAttention Kernel, section 3.2: the
 * write path takes the cache dtype and per-tensor k_scale / v_scale). A pool
 * holds e4m3 codes (1 byte per element: sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, largest finite 448), [num_pages, num_kv_heads, page_size,
 * head_dim] like the bf16 pools; a code c stands for value(c) * scale.
 * head_dim 128 only.
 */

/*
 * pa_append_kv for e4m3 pools: every element of the new rows (bf16) is
 * stored as the e4m3 code nearest to fp32(x) / scale (the quotient rounded to
 * fp32 first; ties to the even code; magnitudes past 448 saturate to 448; a
 * NaN gives a NaN code). k_scale and v_scale must be finite and > 0. Same
 * slots, checks and error reporting as pa_append_kv.
 */
pa_status pa_append_kv_fp8(const void *key, const void *value, void *key_pages,
                           void *value_pages, const int32_t *slot_mapping, int32_t page_size,
                           float k_scale, float v_scale, pa_shape shape, void *stream);

/*
 * pa_decode over e4m3 pools: the same split-KV schedule, arguments,
 * workspace (pa_decode_workspace_bytes) and result as pa_decode, with every
 * K element value(code) * k_scale and every V element value(code) * v_scale.
 * The kernel reads the codes straight from the pages (half the bytes of the
 * bf16 pools) and multiplies on the tensor cores in f16, into which e4m3
 * values convert exactly; the query is taken in f16 too, so its elements
 * must have magnitudes within f16's range (below 65504; below 2^-14 they keep
 * fewer bits). A NaN code in a visible slot gives NaN; slots past a
 * request's context are never read. Any query length;
 * for prefill chunks pa_prefill_fp8 is the faster call.
 */
pa_status pa_decode_fp8(const void *query, const void *key_pages, const void *value_pages,
                        const int32_t *block_table, const int32_t *context_lens, int32_t page_size,
                        float scale, float k_scale, float v_scale, int causal, void *out,
                        pa_shape shape, int32_t max_context_len, void *workspace,
                        size_t workspace_bytes, void *stream);

/*
 * Bytes of device workspace pa_prefill_fp8 needs for `shape` (head_dim 128)
 * with contexts of at most max_context_len tokens, on the CURRENT device; 0
 * on invalid shapes. It holds bf16 copies of K and V in pages of 128 tokens
 * (batch * ceil(max_context_len / 128) pages of num_kv_heads * 128 * 128
 * elements each, 64 KiB per page and KV head for K and V together), their
 * page table, and the split prefill's workspace when pa_prefill_fp8 takes
 * that kernel for the shape, or the pairs kernel's tail pieces' (the same
 * rules as pa_attention's prefill route).
 */
size_t pa_prefill_fp8_workspace_bytes(pa_shape shape, int32_t max_context_len);

/*
 * Prefill attention over e4m3 pools (the pools of pa_append_kv_fp8): the
 * result of pa_decode_fp8 (every K element value(code) * k_scale, every V
 * element value(code) * v_scale, bottom-right causal mask when `causal`) on
 * the tensor-core prefill kernels. Two kernels on `stream`:
 *   1. the K/V tokens each request can see are copied into bf16 pages of
 *      128 tokens in the workspace, each code converted to its exact value
 *      (e4m3 values are bf16 values; a NaN code stays NaN);
 *   2. the kernels of pa_attention's prefill route (pa_prefill's, with tail
 *      pieces at 1.5 to 2 items per SM, or pa_prefill_split's below 1.5)
 *      attend over the copies, with scale * k_scale as the softmax scale and
 *      the output multiplied by v_scale, so the scaled values are never
 *      rounded.
 * Arguments as pa_decode_fp8. max_context_len bounds context_lens and sizes
 * the copy; a longer entry records PA_DEVERR_CONTEXT_LEN and is cut to
 * ceil(max_context_len / 128) * 128 tokens. workspace: at least
 * pa_prefill_fp8_workspace_bytes(shape, max_context_len) bytes, 256-byte
 * aligned, any contents; calls sharing one must not overlap on the GPU.
 * head_dim 128 only (PA_ERR_UNSUPPORTED otherwise); k_scale and v_scale
 * finite and > 0 (PA_ERR_INVALID_ARG).
 */
pa_status pa_prefill_fp8(const void *query, const void *key_pages, const void *value_pages,
                         const int32_t *block_table, const int32_t *context_lens,
                         int32_t page_size, float scale, float k_scale, float v_scale, int causal,
                         void *out, pa_shape shape, int32_t max_context_len, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * The dispatch of pa_attention for e4m3 pools: pa_decode_fp8 for query rows
 * L <= 8 (the page's rule: the e4m3 decode reads K/V once per 16-row tile of
 * a KV group), pa_prefill_fp8 otherwise, with the same arguments. The workspace is the one that call takes, at
 * least pa_attention_fp8_workspace_bytes(shape, max_context_len) bytes,
 * 256-byte aligned (0 bytes: invalid shape or head_dim other than 128).
 */
size_t pa_attention_fp8_workspace_bytes(pa_shape shape, int32_t max_context_len);
pa_status pa_attention_fp8(const void *query, const void *key_pages, const void *value_pages,
                           const int32_t *block_table, const int32_t *context_lens,
                           int32_t page_size, float scale, float k_scale, float v_scale,
                           int causal, void *out, pa_shape shape, int32_t max_context_len,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * Bytes of device workspace pa_prefill_split needs for `shape` and
 * page_size on the CURRENT device, or 0 when the shape takes a prefill
 * kernel that needs none (head_dim 64, page_size < 8, one query head per
 * KV group). The size depends only on the device's SM count (about 130 KiB
 * per SM), not on the batch.
 */
size_t pa_prefill_workspace_bytes(pa_shape shape, int32_t page_size);

/*
 * Prefill attention with the same arguments, result and checks as
 * pa_prefill, on a kernel that balances the work over the GPU: the K/V
 * tiles of every (request, pair of query heads of one KV group, tile of 128
 * query rows; with an odd group size the last pair of each group holds its
 * last head twice and writes it once) form one stream, cut into equal
 * ranges for a persistent grid
 * of one block per SM (the split-KV idea of Week 3 Day 4, "Choose a
 * Schedule for Each Query Shape", applied to the long-query schedule). An
 * item cut by range boundaries is finished by the block holding its first
 * tiles, which merges the partial softmax states its later pieces (done
 * first by the following blocks) left in the workspace. The launch is
 * cooperative (all blocks resident); where the device cannot hold every
 * block at once, the call runs pa_prefill's kernels instead.
 *   workspace        device memory of at least pa_prefill_workspace_bytes,
 *                    256-byte aligned, any contents (nothing needs clearing;
 *                    each launch tags its counters with its own stamp).
 *                    Calls that share a workspace must not overlap on the GPU.
 * Shapes for which pa_prefill_workspace_bytes is 0 run pa_prefill (the
 * workspace is then not touched). PA_ERR_WORKSPACE when the workspace is
 * missing, too small or misaligned. The output is the same softmax as
 * pa_prefill's up to rounding (the pieces' states are combined in fp32).
 */
pa_status pa_prefill_split(const void *query, const void *key_pages,
                           const void *value_pages, const int32_t *block_table,
                           const int32_t *context_lens, int32_t page_size, float scale,
                           int causal, void *out, pa_shape shape, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * Route chosen by pa_attention for these sizes: 0 = decode, 1 = prefill.
 * The rule sits at this boundary (Week 3 Day 4, "Choose a Schedule for Each
 * Query Shape": short queries take the vector decode schedule, long ones the
 * page-walking prefill; no dense fallback). The thresholds are this
 * library's, set by timing both kernels on GB300 (the page's own rule,
 * L <= 8, was set on other hardware): decode for L <= 24, and for L <= 32
 * when max_context_len >= 3072; prefill otherwise. Returns -1 on invalid
 * shapes.
 */
int32_t pa_attention_route(pa_shape shape, int32_t max_context_len);

/*
 * Dispatching entry point: runs pa_decode or pa_prefill as
 * pa_attention_route says, with the same arguments. The workspace is
 * required only when the route is decode. On the prefill route, given a
 * workspace of at least pa_prefill_workspace_bytes (256-byte aligned), it
 * runs pa_prefill_split when the shape has fewer than 1.5 (request, head
 * pair, 128-row query tile) items per SM, where whole blocks would leave
 * SMs idle; otherwise pa_prefill's kernel, and with one to two items per SM
 * (head_dim 128) that kernel balances the blocks through the workspace: a
 * block holding two items hands the last K/V tiles of its second item to a
 * block holding one, which runs them first and leaves their softmax state
 * (O / l in bf16, the maximum and the sum in fp32); the first block merges it
 * at its end. No block waits for another: the side that arrives second merges
 * (normally the first block), and both sides merge with the same arithmetic,
 * so the bits do not depend on the order. The output is the same softmax up
 * to rounding. With NULL or a smaller workspace: pa_prefill as it is.
 */
pa_status pa_attention(const void *query, const void *key_pages,
                       const void *value_pages, const int32_t *block_table,
                       const int32_t *context_lens, int32_t page_size,
                       float scale, int causal, void *out, pa_shape shape,
                       int32_t max_context_len, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * Synchronises `stream`, then reads and clears the device error word of the
 * current device. *flags (may be NULL) receives the PA_DEVERR_* bits seen
 * since the last call. Returns PA_OK when no bit was set,
 * PA_ERR_DEVICE_TIMEOUT when the timeout bit was set, PA_ERR_DEVICE_BOUNDS
 * for any other bit, PA_ERR_CUDA if synchronising failed.
 */
pa_status pa_get_device_error(void *stream, uint32_t *flags);

/*
 * Host-side page allocator and per-step metadata (host code, no GPU work).
 * One pa_kv_cache is one layer's page pool of num_pages pages of page_size
 * tokens, and the pages each request (seq_id) holds in it (Week 3 Day 4,
 * "Decode Metadata"; Tutorial 13, section 4 "The Request Cache"). Not
 * thread-safe: one host thread per cache at a time.
 *   - pages are handed out freed-first (the last freed page first), else the
 *     lowest page id never handed out;
 *   - pa_kv_cache_plan places new tokens by the tail-fill rule: the next token
 *     goes into the request's tail page while it has room, otherwise into a
 *     new page;
 *   - pa_kv_cache_release returns every page of a request exactly once; a
 *     second release (or an unknown seq_id) is PA_ERR_INVALID_ARG.
 */
typedef struct pa_kv_cache pa_kv_cache;

pa_status pa_kv_cache_create(int32_t num_pages, int32_t page_size, pa_kv_cache **cache);
void pa_kv_cache_destroy(pa_kv_cache *cache);

/* A new request with no tokens; PA_ERR_INVALID_ARG if seq_id exists. */
pa_status pa_kv_cache_add(pa_kv_cache *cache, int64_t seq_id);
pa_status pa_kv_cache_release(pa_kv_cache *cache, int64_t seq_id);

/* Pages not held by any request; -1 on a null cache. */
int32_t pa_kv_cache_free_pages(const pa_kv_cache *cache);
/* Tokens cached for seq_id; -1 if unknown. */
int32_t pa_kv_cache_context_len(const pa_kv_cache *cache, int64_t seq_id);

/*
 * One scheduler step for n requests: request i (seq_ids[i], all distinct and
 * added) gets new_tokens[i] (0 .. l_new) new tokens. Writes, into host
 * arrays:
 *   block_table   [n, max_pages]  the request's page ids in logical order,
 *                                 -1 after the last;
 *   context_lens  [n]             tokens cached after this step;
 *   slot_mapping  [n, l_new]      the flat slot (page * page_size + offset)
 *                                 of each new token in order, -1 after the
 *                                 last (may be NULL when l_new == 0).
 * All or nothing: if the pool runs out of pages or a request would need more
 * than max_pages pages, nothing is changed and PA_ERR_NO_PAGES is returned;
 * bad arguments give PA_ERR_INVALID_ARG, also with nothing changed.
 */
pa_status pa_kv_cache_plan(pa_kv_cache *cache, int32_t n, const int64_t *seq_ids,
                           const int32_t *new_tokens, int32_t max_pages, int32_t l_new,
                           int32_t *block_table, int32_t *context_lens, int32_t *slot_mapping);

/*
 * Snapshot and restore (Tutorial 13, section 7 "Transactional Safety"): a
 * snapshot is a copy of the cache's bookkeeping (free list, fresh-page
 * counter, every request's pages and length). Restoring it puts the cache
 * back as it was when the snapshot was taken, so a step whose K/V write or
 * attention launch failed after pa_kv_cache_plan succeeded can be undone.
 * Pool contents are not part of a snapshot and need no restoring: the rows a
 * failed step wrote lie in free pages or past a request's context length,
 * which no kernel reads. The caller owns the snapshot and frees it with
 * pa_kv_cache_snapshot_destroy; restoring a snapshot of another cache is
 * PA_ERR_INVALID_ARG. A snapshot stays valid after restore (restore it again
 * to roll back again).
 */
typedef struct pa_kv_cache_snapshot pa_kv_cache_snapshot;

pa_status pa_kv_cache_snapshot_take(const pa_kv_cache *cache, pa_kv_cache_snapshot **snapshot);
pa_status pa_kv_cache_restore(pa_kv_cache *cache, const pa_kv_cache_snapshot *snapshot);
void pa_kv_cache_snapshot_destroy(pa_kv_cache_snapshot *snapshot);

/*
 * One scheduler step run from the host in a single call (Week 3 Day 4,
 * "Decode Metadata": the batch's page metadata prepared once per step):
 * pa_kv_cache_plan writes the three tables, packed as block_table [n,
 * max_pages], then context_lens [n], then slot_mapping [n, l_new] (int32),
 * into `host_tables`; one asynchronous copy moves them to `device_tables`;
 * then pa_append_kv writes the new K/V rows and pa_attention (causal, with
 * max_context_len = the largest planned context length) runs over the step,
 * all on `stream`.
 *   host_tables    pinned host memory of at least
 *                  pa_kv_cache_step_table_bytes(n, max_pages, l_new) bytes.
 *                  The copy is asynchronous: the caller must not rewrite this
 *                  region (for example by the next step) before the copy has
 *                  run (use one region per step in flight, or synchronise).
 *   device_tables  device memory of the same size, 4-byte aligned; the
 *                  kernels of this step read it.
 *   key_new, value_new  [n, num_kv_heads, l_new, head_dim] bf16 (device);
 *                  rows past a request's new_tokens[i] are not written.
 *   query, out     [n, num_q_heads, l_new, head_dim] bf16 (device); a request
 *                  with fewer than l_new new tokens has its new tokens in its
 *                  last new_tokens[i] rows (bottom-right causal alignment);
 *                  its earlier rows attend as tokens already cached.
 *   key_pages, value_pages  the layer's pool [num_pages, num_kv_heads,
 *                  page_size, head_dim] bf16, num_pages and page_size as
 *                  given to pa_kv_cache_create.
 *   workspace      as pa_attention (required when the step takes the decode
 *                  route, L <= pa_attention_route's threshold).
 * Returns the plan's status (nothing changed on failure), PA_ERR_CUDA if the
 * copy could not be issued, or the status of pa_append_kv / pa_attention; in
 * the last two cases the plan stays applied and a snapshot taken before the
 * call undoes it.
 */
size_t pa_kv_cache_step_table_bytes(int32_t n, int32_t max_pages, int32_t l_new);
pa_status pa_kv_cache_step(pa_kv_cache *cache, int32_t n, const int64_t *seq_ids,
                           const int32_t *new_tokens, int32_t l_new, int32_t max_pages,
                           void *host_tables, void *device_tables, size_t table_bytes,
                           const void *key_new, const void *value_new, const void *query,
                           void *key_pages, void *value_pages, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, float scale, void *out,
                           void *workspace, size_t workspace_bytes, void *stream);

/* Static, human-readable name of a status code. */
const char *pa_status_string(pa_status status);

/* Library version, e.g. "0.1.0". */
const char *pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
