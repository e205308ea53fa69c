/*
 * zp.h -- C ABI of the GB300 (sm_103a) Compressed PagedAttention hot path.
 *
 * The method: "Zipage: Maintain High Request Concurrency for LLM Reasoning
 * through Compressed PagedAttention" as summarised on gist.science (Dutch
 * "Technische samenvatting / Methodologie", Korean "기술 요약 / 2. 방법론"),
 * over the paged KV cache of "Paged KV cache and continuous batching for LLMs"
 * ("How it works").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer documented as "device" is CUDA device memory OWNED BY THE
 *    CALLER.  The library never frees caller memory.  The library owns only
 *    the opaque zp_cache handle and the device workspace it allocates in
 *    zp_cache_create (status word, tensor maps, per-call scratch).
 *  - bf16 tensors are passed as void* and hold IEEE bfloat16 values.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call only enqueues work on `stream`: nothing
 *    synchronises except zp_cache_status, and nothing allocates after
 *    zp_cache_create, so every call that takes a zp_cache handle, except
 *    zp_cache_status, can be captured into a CUDA graph and replayed.
 *  - Argument errors that the host can see are returned synchronously,
 *    before anything is enqueued.  Errors that only the device can see (a
 *    length or block id read from device memory, an empty free stack) are
 *    recorded in the handle's sticky status word, and every later kernel of
 *    the same call skips its writes; read the word with zp_cache_status.
 *  - A handle serves at most one call of each entry point in flight at a
 *    time.  zp_compress may run concurrently with zp_paged_decode_attn and
 *    zp_append_kv on another stream when they touch disjoint requests.
 *    zp_compress, zp_compress_prefill, zp_append_slots, zp_alloc_rows,
 *    zp_release_rows and zp_fork_rows change the free stack or refcounts:
 *    order them (one stream, or events).  More concurrency needs
 *    more handles.
 *
 * KV pool layout (one K pool and one V pool per layer, caller-owned):
 *     pool[num_blocks][num_kv_heads][block_size][head_dim]   bf16, contiguous
 * so one (block, kv head) slab is block_size*head_dim*2 bytes (4 KiB at
 * b = 16, d = 128) and one token row is head_dim*2 bytes.  All layers and kv
 * heads of a request share its block table row.  Pool base addresses must be
 * 16-byte aligned.
 */
#ifndef ZP_H
#define ZP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t zp_status;

#define ZP_OK 0
#define ZP_ERR_INVALID_ARG (-1)   /* bad argument (host- or device-detected) */
#define ZP_ERR_UNSUPPORTED (-2)   /* shape or size outside the supported set */
#define ZP_ERR_OUT_OF_BLOCKS (-3) /* free stack too short for the target blocks */
#define ZP_ERR_DEVICE_CHECK (-4)  /* inconsistent cache state found on the device */
#define ZP_ERR_CUDA (-5)          /* a CUDA runtime call failed */
#define ZP_ERR_TIMEOUT (-6)       /* a bounded device-side wait gave up */

typedef struct zp_cache zp_cache;

/* Shape of the cache and the caller's per-layer pools.
 * Supported: head_dim 64 or 128, block_size 16, num_q_heads a multiple of
 * num_kv_heads.  max_requests bounds the rows of any block table passed to
 * the handle and the batch of any call; max_blocks_per_req bounds the row
 * stride of those tables (it sizes the workspace). */
typedef struct {
    int32_t num_layers;         /* L >= 1 */
    int32_t num_kv_heads;       /* Hkv >= 1 */
    int32_t num_q_heads;        /* Hq, multiple of Hkv */
    int32_t head_dim;           /* d: 64 or 128 */
    int32_t block_size;         /* b: 16 */
    int32_t num_blocks;         /* physical blocks in each pool */
    int32_t max_requests;       /* >= 1 */
    int32_t max_blocks_per_req; /* >= 2 */
    void *const *k_pools;       /* host array of L device pointers (bf16 pools) */
    void *const *v_pools;       /* host array of L device pointers (bf16 pools) */
} zp_cache_desc;

/* Free-block stack and refcounts of the pool (device, caller-owned).
 * free_ids[0 .. *free_count) are the free block ids; the top of the stack is
 * free_ids[*free_count - 1].  refcount[blk] counts the block-table entries
 * (over all live requests) that point at blk; a free block has refcount 0. */
typedef struct {
    int32_t *free_ids;   /* device [capacity] */
    int32_t *free_count; /* device [1] */
    int32_t *refcount;   /* device [num_blocks] */
    int32_t capacity;    /* length of free_ids, >= 1 */
} zp_block_pool;

/* Creates a handle over caller-owned pools and allocates its workspace.
 * Returns ZP_ERR_INVALID_ARG / ZP_ERR_UNSUPPORTED for a bad descriptor
 * (checked before any CUDA call), ZP_ERR_CUDA if an allocation fails.
 * *out is set only on success; the current CUDA device is recorded. */
zp_status zp_cache_create(const zp_cache_desc *desc, zp_cache **out);

/* Frees the handle and its workspace (not the pools).  NULL is a no-op.
 * The caller must make sure no work that uses the handle is in flight. */
void zp_cache_destroy(zp_cache *cache);

/* Compressed PagedAttention compression of R requests, every layer and kv head
 * ("Methodologie" §1, §3, §5 of the Dutch summary; "방법론" A, C, E of the
 * Korean summary).  A request qualifies when it holds n_max full blocks
 * (lengths == n_max * block_size).  For each (request, layer, kv head):
 *   importance  softmax(q . k / sqrt(d)) of the w window queries (the last w
 *               tokens, always in the last block; query i sees keys up to its
 *               own position), averaged over the w queries and the
 *               num_q_heads/num_kv_heads query heads of the group;
 *   redundancy  Lightning Redundancy Score: mean cosine similarity of a key to
 *               the other block_size-1 keys of its own block (0 for a zero key);
 *   score       importance - lambda * redundancy over the C = T - w
 *               candidates (T = n_max * block_size);
 *   select      keep the (n_max-1)*b - w highest scores (at equal score the
 *               lower index), i.e. evict exactly b candidates; the window is
 *               always kept;
 *   compact     the kept tokens, in original order, fill blocks 0..n_max-2 of
 *               the request; block n_max-1 stays reserved for decoding.
 * Blocks are decided on the refcounts at call start: a block with refcount 1
 * is rewritten in place; a block with refcount > 1 (a shared prefix) is never
 * written -- its destination is a fresh target block popped from the top of
 * the free stack (in request, block order), and it loses one reference per
 * compressing holder; a shared reserved block is replaced by a fresh block.
 * A block whose refcount reaches 0 is pushed on the free stack (after the
 * pops), in the order a sequential pass over (request, block) zeroes it.
 * Afterwards table rows hold the destination blocks and lengths are
 * (n_max-1)*b.
 *
 *  block_tables  device int32 [num_rows][bt_stride], in/out
 *  lengths       device int32 [num_rows], in/out (== n_max*b on input)
 *  req_idx       device int32 [R] row of each compressing request, distinct,
 *                or NULL for rows 0..R-1
 *  window_q      device bf16 [L][R][Hq][w][d]: window queries of request r
 *                (row g*w + i of kv head h's group is query head h*G+g at
 *                window slot i, the query of token T - w + i)
 *  n_max         blocks per request at compression; T = n_max*b must split
 *                into at most 16 equal chunks of at most 2048 tokens, each a
 *                multiple of 128 (every multiple of 128 up to 2048; 4096, 8192,
 *                ... up to 32768 when divisible accordingly)
 *  window        w, 1 <= w <= b, w * (Hq/Hkv) <= 64
 *  lambda        redundancy weight
 *  pool          free stack + refcounts, updated in place
 *  scores_out    NULL or device fp32 [L][R][Hkv][T]: candidate scores
 *                (+inf at window positions)
 *  kept_out      NULL or device int32 [L][R][Hkv][(n_max-1)*b]: kept source
 *                positions, ascending
 * All-or-nothing: on a device-detected error (bad length, bad or duplicate
 * row, bad block id, refcount inconsistent, free stack too short) nothing is
 * written and the sticky status records the error. */
zp_status zp_compress(zp_cache *cache, int32_t *block_tables, int32_t bt_stride,
                      int32_t num_rows, int32_t *lengths, const int32_t *req_idx, int32_t R,
                      const void *window_q, int32_t n_max, int32_t window, float lambda,
                      const zp_block_pool *pool, void *stream, float *scores_out,
                      int32_t *kept_out);

/* Bytes of caller workspace zp_compress_prefill needs for R requests and a
 * table stride of bt_stride blocks (the upper bound of every request's
 * length).  Host only; no CUDA call. */
zp_status zp_compress_prefill_workspace_size(const zp_cache *cache, int32_t R, int32_t bt_stride,
                                             size_t *bytes);

/* Compression at admission of requests longer than the budget (Dutch summary
 * "Methodologie" §1: the kept entries move into the first n_max-1 blocks, the
 * n_max-th block is reserved for decoding, and the excess blocks are
 * released; §3: shared blocks compress into fresh target blocks).  Request i
 * (row = req_idx[i], or i) holds T_i = lengths[row] tokens, n_max*16 <= T_i
 * <= bt_stride*16, in blocks 0 .. ceil(T_i/16)-1 of its table row (the last
 * possibly partial).  Per (request, layer, kv head), with C_i = T_i - window:
 *   scores as in zp_compress over the T_i keys (the window is the last
 *   `window` tokens; the redundancy of a key in a partial last block is its
 *   mean cosine to the other filled slots of that block, 0 if alone);
 *   keep the (n_max-1)*16 - window best candidates (ties to the lower index)
 *   and the window, in original order, in blocks 0 .. n_max-2;
 *   blocks 0 .. n_max-1: destinations by the rule of zp_compress (refcount 1
 *   at call start: rewritten in place / kept as the reserved block; > 1: a
 *   fresh target popped from the free stack, one reference dropped);
 *   blocks n_max .. ceil(T_i/16)-1: one reference dropped each, pushed on the
 *   free stack (after the pops, in request-then-block order) when that
 *   empties it, table entry set to -1.
 * Afterwards lengths are (n_max-1)*16.
 *
 *  block_tables, lengths, req_idx, pool  as in zp_compress (lengths as above)
 *  window_q      device bf16 [L][R][Hq][window][d] (the last `window` tokens)
 *  bt_stride     at most max_blocks_per_req of the handle, and bt_stride * 16
 *                <= 32768 (ZP_ERR_UNSUPPORTED beyond)
 *  workspace     device, 256-byte aligned, at least the bytes
 *                zp_compress_prefill_workspace_size reports; caller-owned,
 *                only used during the call's kernels
 *  scores_out    NULL or device fp32 [L][R][Hkv][bt_stride*16]: candidate
 *                scores, +inf at window positions, entries at T_i and beyond
 *                not written
 *  kept_out      NULL or device int32 [L][R][Hkv][(n_max-1)*16], ascending
 * All-or-nothing like zp_compress.  Orders with zp_compress and
 * zp_append_slots (all three change the free stack and refcounts). */
zp_status zp_compress_prefill(zp_cache *cache, int32_t *block_tables, int32_t bt_stride,
                              int32_t num_rows, int32_t *lengths, const int32_t *req_idx,
                              int32_t R, const void *window_q, int32_t n_max, int32_t window,
                              float lambda, const zp_block_pool *pool, void *workspace,
                              size_t workspace_bytes, void *stream, float *scores_out,
                              int32_t *kept_out);

/* Paged decode attention over the block tables of one layer ("Paged KV cache
 * and continuous batching for LLMs", "How it works"): for request i and query
 * head hq (kv head hq / (Hq/Hkv)),
 *     out = sum_t softmax_t(scale * q . k_t) v_t,   t < lengths[row],
 * token t living in block block_tables[row][t / b], slot t % b, where
 * row = req_idx[i] (or i when req_idx is NULL).  fp32 accumulation, one
 * round-to-nearest-even to bf16.  A zero length gives a zero output.
 *
 *  layer         0 <= layer < L
 *  q             device bf16 [R][Hq][d]
 *  block_tables  device int32 [num_rows][bt_stride] (read only)
 *  lengths       device int32 [num_rows], 0 <= lengths[row] <= bt_stride * b
 *  req_idx       device int32 [R] or NULL
 *  out           device bf16 [R][Hq][d]
 * A length or block id out of range is recorded as ZP_ERR_DEVICE_CHECK in the
 * sticky status; the affected outputs are then undefined. */
zp_status zp_paged_decode_attn(zp_cache *cache, int32_t layer, const void *q,
                               const int32_t *block_tables, int32_t bt_stride, int32_t num_rows,
                               const int32_t *lengths, const int32_t *req_idx, int32_t R,
                               float scale, void *out, void *stream);

/* Paged decode attention for callers that cannot allocate device memory.
 * The paper has no counterpart: this is a deployment variant of
 * zp_paged_decode_attn.  Some callers cannot call cudaMalloc where they run
 * decode attention: an allocator or memory-pool callback (allocating there
 * would re-enter the allocator), a plug-in in a process whose host owns all
 * device memory, a real-time path that must not wait on the allocator.  This
 * call needs no zp_cache handle and allocates nothing: it runs the same
 * kernels as zp_paged_decode_attn, with the two pools' tensor maps encoded on
 * the host and passed in the launch parameters, and with the same splits its
 * results are those of zp_paged_decode_attn bit for bit.  Its split-K
 * partial results live in one fixed device array compiled into the library
 * (about 16.3 MiB), created when the library's device code is loaded into a
 * CUDA context -- usually at the first call in that context -- and held until
 * the process exits.
 *
 *  k_pool, v_pool  device bf16 pools of one layer, [num_blocks][num_kv_heads][16][head_dim],
 *                  16-byte aligned (ZP_ERR_INVALID_ARG otherwise)
 *  q, out          device bf16 [R][num_q_heads][head_dim], q 16-byte and out
 *                  2-byte aligned (ZP_ERR_INVALID_ARG otherwise); other
 *                  arguments as in zp_paged_decode_attn
 *  status          nullable device int32: device-detected errors (a length or
 *                  block id out of range) are recorded there with atomicCAS from 0
 *                  (with NULL they go to the array's last word and are not read)
 * Limits: head_dim 64 or 128, block size 16, num_q_heads / num_kv_heads <= 16,
 * R * num_q_heads <= 32768 (ZP_ERR_UNSUPPORTED beyond); fewer splits than
 * zp_paged_decode_attn's where the array cannot hold their partials.
 * The array's device address belongs to the current CUDA context (another
 * context on the same device, or the primary context re-created after
 * cudaDeviceReset, has its own copy).  A call made while `stream` is not
 * being captured looks the address up in the current context (a host-side
 * lookup) and records it; a call made while `stream` is being captured uses
 * only an address recorded earlier in the same context and returns
 * ZP_ERR_UNSUPPORTED, before any other CUDA call, when there is none.  So in
 * each context make the first call before any stream capture (and again
 * after cudaDeviceReset).
 * Every call shares the array and each call overwrites the slots it reads,
 * so nothing needs clearing between calls; calls that overlap on the GPU (two
 * streams, or two threads) race on it and must be serialised by the caller. */
zp_status zp_paged_decode_attn_noalloc(const void *k_pool, const void *v_pool, int32_t num_blocks,
                                       int32_t num_kv_heads, int32_t num_q_heads,
                                       int32_t head_dim, const void *q,
                                       const int32_t *block_tables, int32_t bt_stride,
                                       int32_t num_rows, const int32_t *lengths,
                                       const int32_t *req_idx, int32_t R, float scale, void *out,
                                       int32_t *status, void *stream);

/* Reserves the slot of each listed request's next decode token, request
 * after request in list order ("Paged KV cache and continuous batching for
 * LLMs", "How it works": a block is taken only when the previous ones are
 * full; a write into a shared block first copies it, block-level
 * copy-on-write), and lists the requests that become due for compression
 * (Dutch summary "Methodologie" §1: N_max blocks held and the last one full).
 * For request i (row = req_idx[i], or i) with p = lengths[row], the new
 * token goes to block entry e = p / 16, slot p % 16:
 *   - block_tables[row][e] < 0 (allowed only at slot 0): a fresh block is
 *     popped and becomes the entry;
 *   - else, if that block's refcount, as updated by the requests before this
 *     one, is > 1: a fresh block is popped, slots 0 .. p%16 - 1 of every
 *     layer and kv head (K and V) are copied into it, it becomes the entry,
 *     and the original loses one reference;
 *   - else the block is written in place (nothing to do here).
 * Popped blocks come from the top of the free stack, in list order, and get
 * refcount 1.  Then lengths[row] = p + 1, and when n_max > 0 and p + 1 ==
 * n_max * 16 the row is listed in trigger_rows (list order).  A table entry
 * beyond a row's filled blocks must be < 0 unless it holds a block already
 * reserved for the row (the empty last block zp_compress leaves).
 *
 *  block_tables  device int32 [num_rows][bt_stride], in/out
 *  lengths       device int32 [num_rows], in/out: 0 <= p < bt_stride * 16,
 *                and p < n_max * 16 when n_max > 0 (a full request is
 *                compressed first)
 *  req_idx       device int32 [R] distinct rows, or NULL for rows 0..R-1
 *  n_max         blocks per request at compression, or 0 for no limit
 *  pool          free stack + refcounts, updated in place
 *  trigger_rows  NULL or device int32 [R]: rows that reached n_max * 16
 *  trigger_count NULL or device int32 [1]: how many (0 after an error)
 * All-or-nothing: a row out of range or repeated, a length out of range, a
 * tail entry out of range (or < 0 at slot > 0), a tail block with fewer
 * references than rows of this call writing it -> ZP_ERR_INVALID_ARG; too few
 * free blocks -> ZP_ERR_OUT_OF_BLOCKS; a popped id out of range or with a
 * nonzero refcount -> ZP_ERR_DEVICE_CHECK; all recorded in the sticky status,
 * with nothing written.  R == 0 only zeroes *trigger_count. */
zp_status zp_append_slots(zp_cache *cache, int32_t *block_tables, int32_t bt_stride,
                          int32_t num_rows, int32_t *lengths, const int32_t *req_idx, int32_t R,
                          int32_t n_max, const zp_block_pool *pool, void *stream,
                          int32_t *trigger_rows, int32_t *trigger_count);

/* Blocks for the first tokens of requests entering the batch ("Paged KV
 * cache and continuous batching for LLMs", "How it works": blocks are taken
 * from the pool only as the tokens need them).  Request i (row = req_idx[i],
 * or i) must be empty (lengths[row] == 0, entries < 0); it gets counts[i]
 * tokens: entries 0 .. ceil(counts[i]/16)-1 become blocks popped from the top
 * of the free stack in (request, block) order, refcount 1, and lengths[row] =
 * counts[i].  The tokens' keys and values are the caller's to write.
 *
 *  counts        device int32 [R], 0 <= counts[i] <= bt_stride * 16
 * All-or-nothing: a bad or repeated row, a row that is not empty, a count out
 * of range -> ZP_ERR_INVALID_ARG; too few free blocks -> ZP_ERR_OUT_OF_BLOCKS;
 * a popped id out of range or with a nonzero refcount -> ZP_ERR_DEVICE_CHECK
 * (all in the sticky status).  Orders with every other call that changes the
 * pool. */
zp_status zp_alloc_rows(zp_cache *cache, int32_t *block_tables, int32_t bt_stride,
                        int32_t num_rows, int32_t *lengths, const int32_t *req_idx, int32_t R,
                        const int32_t *counts, const zp_block_pool *pool, void *stream);

/* Every block of finished or preempted requests back to the pool ("How
 * it works": a block's reference counter counts the tables that point at
 * it).  Request after request, entry after entry, each entry >= 0 of the row
 * (including a reserved, still empty block) drops one reference of its block,
 * which is pushed on the free stack when that empties it; the entry becomes
 * -1 and lengths[row] becomes 0.  Shared blocks survive while other rows hold
 * them.  All-or-nothing: a bad or repeated row, an entry >= num_blocks, a
 * block held by more released entries than its refcount ->
 * ZP_ERR_INVALID_ARG; no room on the free stack -> ZP_ERR_DEVICE_CHECK.
 * Orders with every other call that changes the pool. */
zp_status zp_release_rows(zp_cache *cache, int32_t *block_tables, int32_t bt_stride,
                          int32_t num_rows, int32_t *lengths, const int32_t *req_idx, int32_t R,
                          const zp_block_pool *pool, void *stream);

/* Forks requests ("How it works": parallel samples of one prompt share its
 * blocks, whose reference counters count the tables pointing at them): row
 * dst_rows[i], which must be empty (length 0, every entry < 0), becomes a copy
 * of row src_rows[i] -- the same entries (a reserved empty block included) and
 * the same length -- and every block entry gains one reference.  The next
 * write of either row into a shared partial block copies it first
 * (zp_append_slots).
 *
 *  src_rows, dst_rows  device int32 [n]; destinations distinct, none of them
 *                      a source in the same call
 *  refcount            device int32 [num_blocks], updated
 * All-or-nothing: a bad or repeated row, a destination that is not empty, a
 * source entry out of range or unreferenced -> ZP_ERR_INVALID_ARG in the
 * sticky status.  Orders with every other call that changes the pool. */
zp_status zp_fork_rows(zp_cache *cache, int32_t *block_tables, int32_t bt_stride,
                       int32_t num_rows, int32_t *lengths, const int32_t *src_rows,
                       const int32_t *dst_rows, int32_t n, int32_t *refcount, void *stream);

/* Writes one layer's new-token keys and values into the slots zp_append_slots
 * reserved ("Paged KV cache and continuous batching for LLMs", "How it
 * works"): for request i (row = req_idx[i], or i), token p = lengths[row] - 1
 * in block block_tables[row][p / 16], slot p % 16, gets k_new[i][h] and
 * v_new[i][h] for every kv head h.  Call it for each layer after
 * zp_append_slots, before that layer's zp_paged_decode_attn.
 *
 *  layer         0 <= layer < L
 *  k_new, v_new  device bf16 [R][num_kv_heads][head_dim], 16-byte aligned
 *  block_tables, lengths, req_idx as after zp_append_slots (read only)
 * A row, length or block id out of range is recorded as ZP_ERR_DEVICE_CHECK
 * in the sticky status and that row is skipped. */
zp_status zp_append_kv(zp_cache *cache, int32_t layer, const void *k_new, const void *v_new,
                       const int32_t *block_tables, int32_t bt_stride, int32_t num_rows,
                       const int32_t *lengths, const int32_t *req_idx, int32_t R, void *stream);

/* Redundancy of every key against ALL keys of its (request, layer, kv
 * head): the O(N^2 b^2) score that the Lightning Redundancy Score replaces
 * (Dutch summary "Methodologie" §5, Korean "방법론" E), computed for
 * comparison; the compression calls never use it.  With this library's
 * definition, red[t] = mean over the other keys k of the unit of
 * cos(K_t, K_k) (a zero key has cosine 0 with every key), over the
 * T_i = lengths[row] cached tokens of request i (row = req_idx[i], or i).
 * Computed as (K_t/|K_t| . S - 1) / (T_i - 1) with S the sum of the unit's
 * normalised nonzero keys: two passes over the keys, O(T d).
 *
 *  block_tables, lengths, req_idx  as in zp_paged_decode_attn (read only)
 *  red_out       device fp32 [L][R][Hkv][bt_stride*16]; entries at T_i and
 *                beyond are not written
 * A row, length or block id out of range is recorded as ZP_ERR_DEVICE_CHECK
 * (ZP_ERR_INVALID_ARG for a row) in the sticky status. */
zp_status zp_global_redundancy(zp_cache *cache, const int32_t *block_tables, int32_t bt_stride,
                               int32_t num_rows, const int32_t *lengths, const int32_t *req_idx,
                               int32_t R, float *red_out, void *stream);

/* The same score as zp_global_redundancy, computed the way the original
 * O(N^2 b^2) method pays for it: the dense T_i x T_i Gram matrix of every
 * unit on the tensor cores (tcgen05, bf16 products, fp32 accumulation in
 * tensor memory), red[t] = (sum_k cos(K_t, K_k) - 1) / (T_i - 1) from its
 * rows.  For comparison only; O(T^2 d) work per unit.  Arguments, output
 * layout and error reporting as zp_global_redundancy; a wait that runs out
 * records ZP_ERR_TIMEOUT. */
zp_status zp_global_redundancy_gram(zp_cache *cache, const int32_t *block_tables,
                                    int32_t bt_stride, int32_t num_rows, const int32_t *lengths,
                                    const int32_t *req_idx, int32_t R, float *red_out,
                                    void *stream);

/* Synchronises `stream`, returns the handle's sticky device status in
 * *out_status (ZP_OK or the first device-detected error since the last
 * read) and clears it.  Returns ZP_ERR_CUDA if the stream reports an error. */
zp_status zp_cache_status(zp_cache *cache, void *stream, int32_t *out_status);

/* Static description of a status code ("ok", "invalid argument", ...). */
const char *zp_status_string(zp_status status);

#ifdef __cplusplus
}
#endif

#endif /* ZP_H */
