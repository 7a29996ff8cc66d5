/*
 * pagedkv.h -- C ABI of the paged KV cache hot path for NVIDIA GB300 (sm_103a).
 *
 * Operations on a pool of fixed-size KV blocks:
 *
 *   copy_blocks             batched copy-on-write block copies (src -> dst);
 *   kv_swap_blocks          batched block moves to and from host memory;
 *   kv_append               slot-mapped write of each new token's K and V row
 *                           (the pages' reshape-and-cache step);
 *   paged_attention_decode  single-query attention per sequence, reading K and
 *                           V through the sequence's block table inside the
 *                           kernel (split over the GPU, merged by log-sum-exp).
 *
 * Sources, by page title and section:
 *   "Lecture 3: memory and prefix reuse in serving engines -- vLLM
 *   PagedAttention and SGLang RadixAttention" (semidirectx.com, CS349D notes),
 *   sec. 3.1 (blocks, block tables), sec. 3.2 (attention over scattered blocks;
 *   fused write-by-block-table kernel; copy-on-write copies batched into one
 *   launch), sec. 4.1 (copy-on-write);
 *   "Lecture 24: PagedAttention and vLLM" (semidirectx.com, CMU 11-868
 *   notes), sec. 3.2 (block-wise scores merged with an online softmax, the
 *   Flash-Decoding trick);
 *   "Part 3: single node" (random-liu.github.io), ch. 9 sec. 1 (grouped-query
 *   heads), ch. 11 sec. 3 (block table [max_num_reqs, max_num_blocks_per_req]),
 *   ch. 13 sec. 1 (slot_mapping: kv_cache[slot_mapping[i]] = new_kv);
 *   "S06 memory and KV cache: PagedAttention" (llminference.xinbetween.com),
 *   "Implementation" (pool layout [num_blocks, block_size, n_kv_heads,
 *   head_dim]; the block-table indirection happens inside the kernel).
 *
 * Conventions shared by every call
 *   - Memory: every device pointer is owned by the caller and must stay valid
 *     until the work queued on the stream has finished.  Pointers to element
 *     data and to the workspace must be 16-byte aligned; tensors are dense,
 *     row-major, with the layouts stated below.
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *     default stream).  Calls only enqueue work; none synchronises the host,
 *     except kv_pool_get_error.
 *   - Errors: argument checks run on the host before anything is enqueued and
 *     return a kv_status; nothing is enqueued on failure.  Data-dependent
 *     faults (an out-of-range slot, block id or copy pair; a too-short block
 *     table) are found by the kernels: the offending item is skipped, a bit is
 *     set in the pool's device error word, and kv_pool_get_error reports it.
 *   - Element types: q, out, new K/V rows and the pools all use the pool's
 *     kv_dtype.  Arithmetic in attention is fp32; one rounding to the output
 *     type at the end (round to nearest even).  An 8-bit pool
 *     (kv_pool_create_quantized) stores K and V as FP8 or INT8 codes while q,
 *     out and the new K/V rows keep a 16-bit type.
 *   - Devices: a pool belongs to the device that was current when it was
 *     created; every call on it must be made with that device current.
 *   - Tracing: each call that enqueues work (kv_append, copy_blocks,
 *     kv_swap_blocks, the three decode calls, paged_attention_prefill) is one
 *     NVTX range named after the call in the NVTX domain "pagedkv", opened on
 *     entry and closed on every return; with no profiling tool attached a
 *     range costs one pointer test.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KV_OK = 0,
    KV_EINVAL = 1,        /* a null pointer, bad size, misalignment, mismatch   */
    KV_EUNSUPPORTED = 2,  /* valid but not built: head_dim, group size, dtype  */
    KV_ECUDA = 3,         /* a CUDA runtime or driver call failed              */
    KV_ERANGE = 4,        /* kv_pool_get_error: the device error word is set   */
    KV_ENOWORKSPACE = 5   /* workspace too small (see the size query)          */
} kv_status;

typedef enum {
    KV_F32 = 0,
    KV_F16 = 1,
    KV_BF16 = 2,
    KV_FP8_E4M3 = 3,  /* 8-bit pools only (kv_pool_create_quantized)            */
    KV_INT8 = 4       /* 8-bit pools only (kv_pool_create_quantized)            */
} kv_dtype;

/* Bits of the device error word (kv_pool_get_error). */
#define KV_DEVERR_SLOT_RANGE   0x1  /* kv_append: slot >= num_blocks*block_size     */
#define KV_DEVERR_BLOCK_RANGE  0x2  /* decode: table entry outside [0, num_blocks)  */
#define KV_DEVERR_PAIR_RANGE   0x4  /* copy_blocks: src or dst outside the pool     */
#define KV_DEVERR_SEQ_RANGE    0x8  /* decode: seq_len > max_blocks_per_seq*bs      */
#define KV_DEVERR_TIMEOUT      0x10 /* a pipeline wait gave up (work was skipped)    */
#define KV_DEVERR_GROUP_RANGE  0x20 /* cascade: a group outside the batch, overlapping
                                       or out of order (its sharing is ignored)       */
#define KV_DEVERR_QUERY_RANGE  0x40 /* prefill: cu_seqlens decreasing or past
                                       num_tokens (the request is skipped), or a
                                       request with more than max_query_len queries
                                       (the queries past it are not computed)         */

typedef struct kv_pool* kv_pool_t;

/*
 * kv_pool_create -- describe a KV block pool held in caller memory.
 *
 * k_pool, v_pool: device pointers, each [num_blocks, block_size, num_kv_heads,
 *   head_dim] of `dtype` (the layout of the S06 page's k_cache), 16-byte aligned.
 * Limits: 1 <= block_size <= 256; head_dim in {64, 128}; num_kv_heads >= 1;
 *   num_blocks >= 1 and num_blocks * block_size < 2^31.
 * On success *out receives a handle.  The handle owns no pool memory: it holds
 *   the geometry, the TMA descriptors built from k_pool / v_pool (plain, and
 *   128-byte-swizzled for 16-bit head_dim-128 pools), and a 4-byte device
 *   error word that this call allocates (freed by kv_pool_destroy).
 * Errors: KV_EINVAL (null or misaligned pointer, size out of range),
 *   KV_EUNSUPPORTED (head_dim, dtype), KV_ECUDA.
 */
kv_status kv_pool_create(int num_blocks, int block_size, int num_kv_heads, int head_dim,
                         kv_dtype dtype, void* k_pool, void* v_pool, kv_pool_t* out);

/*
 * kv_pool_create_quantized -- describe an 8-bit KV block pool ("Part 3: single
 * node", random-liu.github.io, ch. 10: K and V are scaled and rounded to 8
 * bits when a token is written and turned back into wider numbers when the
 * attention reads them; INT8 with a fine-grained per-token scale, FP8 as a
 * shorter float).
 *
 * cache_dtype: KV_FP8_E4M3 or KV_INT8.  dtype: KV_F16 or KV_BF16, the type of
 *   q, out and of the new K/V rows given to kv_append.
 * k_pool, v_pool: device uint8 [num_blocks, block_size, num_kv_heads,
 *   head_dim] (one code per element), 16-byte aligned.
 * KV_FP8_E4M3: code = E4M3(x / scale) with the division in fp32, rounded to
 *   nearest (ties to even) and saturated to +-448 (infinities included; NaN
 *   stays NaN); value = E4M3 value of the code * scale.  k_scale / v_scale are
 *   the pool's K and V scales (finite, > 0); k_scales, v_scales must be NULL.
 * KV_INT8: one scale per (block, KV head, token row), decided when the row is
 *   written: amax = max |x| over its head_dim elements, inv = 127 / amax and
 *   scale = amax / 127 in fp32, code = x * inv rounded to nearest even and
 *   clipped to [-127, 127]; value = code * scale.  An all-zero row has scale 0;
 *   a row holding NaN or an infinity gets scale NaN and codes 0.  k_scales,
 *   v_scales: device fp32 [num_blocks, num_kv_heads, block_size], 16-byte
 *   aligned, owned by the caller; k_scale and v_scale are ignored.
 * Limits: head_dim 128; block_size a multiple of 16, at most 256; the rest as
 *   kv_pool_create.  copy_blocks moves codes and INT8 scales together; decode
 *   computes with the dequantised values (fp32 scores and softmax, as for
 *   16-bit pools).  paged_attention_decode_cascade has a prefix pass for 8-bit
 *   pools of block size 16 and 32.
 * Errors: KV_EINVAL, KV_EUNSUPPORTED, KV_ECUDA.
 */
kv_status kv_pool_create_quantized(int num_blocks, int block_size, int num_kv_heads,
                                   int head_dim, kv_dtype cache_dtype, kv_dtype dtype,
                                   void* k_pool, void* v_pool, float* k_scales, float* v_scales,
                                   float k_scale, float v_scale, kv_pool_t* out);

/* kv_pool_destroy -- free the handle and its error word (not the pools).
 * Work already queued with the handle must have finished.  NULL is a no-op. */
kv_status kv_pool_destroy(kv_pool_t pool);

/*
 * kv_append -- write each new token's K and V row into its slot
 * ("Part 3: single node", ch. 13 sec. 1: kv_cache[slot_mapping[i]] = new_kv).
 *
 * k_new, v_new: device [num_tokens, num_kv_heads, head_dim] of the pool dtype
 *   (of the pool's 16-bit type for an 8-bit pool, whose rows are quantised as
 *   kv_pool_create_quantized describes).
 * slot_mapping: device int64 [num_tokens]; slot = block * block_size + offset.
 *   A negative slot is padding and is skipped.  A slot >= num_blocks *
 *   block_size is skipped and sets KV_DEVERR_SLOT_RANGE.
 * Two tokens with the same slot: one of the rows wins (unspecified which).
 * num_tokens = 0 enqueues nothing.
 */
kv_status kv_append(kv_pool_t pool, const void* k_new, const void* v_new,
                    const int64_t* slot_mapping, int num_tokens, void* stream);

/*
 * copy_blocks -- copy-on-write block copies in one launch ("Lecture 3", sec. 3.2
 * and sec. 4.1): for every pair, K[dst] <- K[src] and V[dst] <- V[src], whole
 * blocks (block_size * num_kv_heads * head_dim elements each).
 *
 * pairs: device int32 [num_pairs, 2] holding (src, dst).  Precondition: the dst
 *   ids are distinct and no dst is also a src in the same call (the copies run
 *   concurrently).  A pair with an id outside [0, num_blocks) is skipped and
 *   sets KV_DEVERR_PAIR_RANGE.  num_pairs = 0 enqueues nothing.
 */
kv_status copy_blocks(kv_pool_t pool, const int32_t* pairs, int num_pairs, void* stream);

/*
 * kv_swap_blocks -- move whole blocks between the pool and a host-memory pool
 * of the same layout, all pairs in one launch ("Lecture 3", semidirectx.com
 * CS349D notes, sec. 5.2 and "Part 3: single node", ch. 14 sec. 3: a
 * preempted request's KV blocks are copied to CPU memory, handed out by a CPU
 * block allocator, and copied back to GPU blocks when it resumes).
 *
 * host_k, host_v: [num_host_blocks, block_size, num_kv_heads, head_dim] of the
 *   pool's element type (codes for an 8-bit pool), 16-byte aligned, in pinned
 *   host memory the device can address (cudaHostAlloc / cudaHostRegister, or
 *   managed memory); the kernel reads or writes it directly.
 * host_k_scales, host_v_scales: INT8 pools only, fp32 [num_host_blocks,
 *   num_kv_heads, block_size] in the same kind of memory; NULL otherwise.
 * pairs: int32 [num_pairs, 2] = (pool block, host block), device-accessible.
 *   KV_SWAP_OUT: host[h] <- pool[g]; KV_SWAP_IN: pool[g] <- host[h], codes and
 *   scales alike.  Precondition: destination blocks are distinct and no
 *   destination is a source of the same call.  A pair outside either pool is
 *   skipped and sets KV_DEVERR_PAIR_RANGE.  num_pairs = 0 enqueues nothing.
 * The host pool is read or written by the GPU when the stream reaches the
 *   call: the host must not touch those blocks until the stream has passed it.
 * Errors: KV_EINVAL (bad direction, pointer not device-accessible, misaligned,
 *   scales given or missing), KV_ECUDA.
 */
#define KV_SWAP_OUT 0   /* device pool -> host pool */
#define KV_SWAP_IN 1    /* host pool -> device pool */
kv_status kv_swap_blocks(kv_pool_t pool, void* host_k, void* host_v, float* host_k_scales,
                         float* host_v_scales, int num_host_blocks, const int32_t* pairs,
                         int num_pairs, int direction, void* stream);

/*
 * paged_attention_workspace_size -- bytes of device workspace that
 * paged_attention_decode needs for this pool, batch and head count on the
 * current device.  The value depends only on these arguments and the device.
 */
kv_status paged_attention_workspace_size(kv_pool_t pool, int batch, int num_q_heads,
                                         size_t* bytes);

/*
 * paged_attention_decode_launches -- how many kernels one
 * paged_attention_decode call with these arguments enqueues: 1 (the split
 * kernel, which also merges the pieces it cut), or 2 (split, then a merge
 * kernel: long contexts, where few (sequence, KV head) pairs are each cut
 * across many warps' ranges).  Like the workspace size, it depends only on
 * the arguments and the device.  A cascade call adds its prefix pass.
 * Errors: KV_EINVAL (null launches, bad shape), KV_EUNSUPPORTED, KV_ECUDA.
 */
kv_status paged_attention_decode_launches(kv_pool_t pool, int batch, int num_q_heads,
                                          int* launches);

/*
 * paged_attention_decode -- one query token per sequence attends over its
 * whole cached context ("Lecture 3", sec. 3.2; S06 "Implementation").
 *
 * For sequence b and query head h, with g = h / (num_q_heads / num_kv_heads)
 * (consecutive query heads share a KV head, "Part 3", ch. 9 sec. 1) and
 * L = seq_lens[b]:
 *     s_t = scale * dot(q[b,h,:], K[block_tables[b, t / bs], t % bs, g, :])
 *     out[b,h,:] = sum_t softmax(s)_t * V[block_tables[b, t / bs], t % bs, g, :]
 * over t = 0 .. L-1.  L = 0 gives zeros.  Only table entries
 * 0 .. ceil(L / bs) - 1 are read; the last block is loaded whole, but only its
 * rows below L contribute (the rest may hold anything, NaN included).
 *
 * q, out: device [batch, num_q_heads, head_dim] of the pool dtype.
 * block_tables: device int32 [batch, max_blocks_per_seq] (row-major).
 * seq_lens: device int32 [batch], the context length including the token the
 *   step appended.  L > max_blocks_per_seq * bs is clamped to the table and
 *   sets KV_DEVERR_SEQ_RANGE; an entry outside [0, num_blocks) is skipped
 *   (its tokens do not take part) and sets KV_DEVERR_BLOCK_RANGE.
 * num_kv_heads must equal the pool's; num_q_heads / num_kv_heads in {1,2,4,8};
 *   1 <= batch <= 4096.
 * workspace: device scratch of at least paged_attention_workspace_size bytes,
 *   16-byte aligned, owned by the caller.  Its contents need no initialisation
 *   and carry nothing the caller must manage between calls: it holds per-call
 *   partial results and piece counters; every call tags its counters with a
 *   fresh random 64-bit value and counts a counter of another tag as zero,
 *   so whatever the memory held before (an earlier call's counters, other
 *   data) is taken for a live count only if it matches that tag, with
 *   probability 2^-64.  Calls that use the same workspace must not overlap
 *   in time.
 * Errors: KV_EINVAL, KV_EUNSUPPORTED, KV_ENOWORKSPACE, KV_ECUDA.
 */
kv_status paged_attention_decode(kv_pool_t pool, const void* q, void* out,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* seq_lens, int batch, int num_q_heads,
                                 float scale, int num_kv_heads, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * paged_attention_cascade_workspace_size -- bytes of workspace that
 * paged_attention_decode_cascade needs (>= paged_attention_workspace_size).
 */
kv_status paged_attention_cascade_workspace_size(kv_pool_t pool, int batch, int num_q_heads,
                                                 int num_groups, size_t* bytes);

/*
 * paged_attention_decode_cascade -- paged_attention_decode for batches whose
 * sequences share prefix blocks ("Lecture 3", sec. 4.1: parallel samples and
 * beams point their tables at the same physical blocks; S06 "In production":
 * the cascade path batches the shared prefix apart from the diverging
 * suffixes).  The result is that of paged_attention_decode on the same
 * arguments (up to fp32 rounding); the grouping only lets each shared block be
 * read once per group instead of once per sequence.
 *
 * group_first, group_size, group_shared_blocks: device int32 [num_groups].
 *   Group k is sequences group_first[k] .. group_first[k] + group_size[k] - 1;
 *   its members' tables hold the same physical block ids in their first
 *   group_shared_blocks[k] entries.  Groups are disjoint and sorted by their
 *   first member; sequences outside every group are decoded plainly.
 *   Preconditions the kernel cannot check: the shared entries are identical
 *   across members (otherwise the first member's blocks are used for all of
 *   the prefix pass's blocks).  A group outside the batch, overlapping its
 *   predecessor or out of order is ignored (its members are decoded plainly)
 *   and sets KV_DEVERR_GROUP_RANGE.  The prefix pass attends the shared
 *   blocks that are full for every member (the count is clamped to each
 *   member's length / block size), in whole work units of the per-sequence
 *   pass: one block, or two for 8-bit pools of block size 16; shared blocks
 *   past those are read through each member's own table.
 * num_groups <= 1024.  head_dim 128, block size 16 or 32, 16-bit pools and
 *   8-bit pools with 16-bit queries have a prefix pass for every query/KV head
 *   ratio (1, 2, 4, 8), whose tiles hold 16 / ratio members' query rows and
 *   128 shared tokens; other shapes and num_groups = 0 are decoded by
 *   paged_attention_decode (same result).
 * workspace: at least paged_attention_cascade_workspace_size bytes.
 * Two kernels are enqueued (the shared-prefix pass, then the per-sequence
 * pass); the other arguments, errors and device error bits are those of
 * paged_attention_decode.
 */
kv_status paged_attention_decode_cascade(kv_pool_t pool, const void* q, void* out,
                                         const int32_t* block_tables, int max_blocks_per_seq,
                                         const int32_t* seq_lens, int batch, int num_q_heads,
                                         float scale, int num_kv_heads, const int32_t* group_first,
                                         const int32_t* group_size,
                                         const int32_t* group_shared_blocks, int num_groups,
                                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * paged_attention_prefill -- paged (chunked) prefill attention: several query
 * tokens per request, each attending causally to the request's cached tokens
 * and to the chunk's earlier tokens, K and V read through the block table
 * inside the kernel ("Part 3: single node", random-liu.github.io, ch. 13
 * sec. 1-2: the new tokens of a batch are flattened into one stream with
 * request boundaries cu_seqlens; a long prompt is processed one chunk per
 * iteration and a chunk attends to the cached earlier chunks through the
 * block table, as decode does).
 *
 * q, out: device [num_tokens, num_q_heads, head_dim] of the pool dtype (the
 *   query type of an 8-bit pool); the queries of request b are rows
 *   cu_seqlens[b] .. cu_seqlens[b+1]-1.
 * cu_seqlens: device int32 [batch + 1], non-decreasing, cu_seqlens[batch] <=
 *   num_tokens.  C_b = cu_seqlens[b+1] - cu_seqlens[b] queries for request b.
 * seq_lens: device int32 [batch]: L_b, the request's context length counted
 *   after this chunk's own K/V rows were appended (kv_append first).  The
 *   C_b queries are positions L_b - C_b .. L_b - 1, and query i sees
 *   positions 0 .. L_b - C_b + i.  C_b = 1 is one decode query.  A query
 *   whose position is negative (C_b > L_b) sees nothing and its output is 0.
 * block_tables: device int32 [batch, max_blocks_per_seq], as for decode.
 * max_query_len: an upper bound on every C_b (1 <= max_query_len <=
 *   num_tokens); it sizes the grid.
 * scale: > 0 and finite.  Arithmetic: fp32 scores and softmax on the tensor
 *   cores (products of 16-bit inputs, fp32 accumulation; the probabilities
 *   enter the second product as two 16-bit halves, so they keep fp32-level
 *   accuracy); one rounding of each output to the pool dtype.  8-bit pools:
 *   the codes are turned exactly into the query type in shared memory; FP8
 *   scales the scores by k_scale and the output by v_scale, INT8 each token's
 *   scores by its K scale and its probability by its V scale (all in fp32),
 *   so the result is attention over the dequantised values.
 * Limits: 16-bit and 8-bit pools, head_dim 128, block_size a power of two in
 *   [8, 128] (8-bit pools: [16, 128]), num_q_heads / num_kv_heads in
 *   {1, 2, 4, 8}, batch <= 65535.  num_tokens = 0 is a no-op.
 * Needs no workspace.  Output rows of queries that no request covers are not
 *   written.
 * Errors: KV_EINVAL (null, misaligned, num_kv_heads differing from the pool,
 *   scale not > 0, max_query_len out of range), KV_EUNSUPPORTED, KV_ECUDA.
 *   Device error bits: KV_DEVERR_QUERY_RANGE (malformed cu_seqlens, or
 *   C_b > max_query_len), KV_DEVERR_BLOCK_RANGE, KV_DEVERR_SEQ_RANGE (L_b
 *   larger than the table holds: clamped), KV_DEVERR_TIMEOUT.
 */
kv_status paged_attention_prefill(kv_pool_t pool, const void* q, void* out,
                                  const int32_t* cu_seqlens, int num_tokens, int max_query_len,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* seq_lens, int batch, int num_q_heads,
                                  float scale, int num_kv_heads, void* stream);

/*
 * paged_attention_decode_noalloc -- paged_attention_decode without a
 * caller-supplied workspace.  (The source pages have no counterpart: this is
 * an interface convenience of this library.)
 *
 * For callers that cannot allocate device memory -- for example a serving
 * engine that reserves the whole device for its KV pool up front and forbids
 * allocation inside the decode loop, or a plug-in whose host framework owns
 * the allocator and passes it only input and output buffers.  The scratch
 * comes from a 32 MiB array compiled into the library, held on every device
 * that loads the library until the process exits.  Arguments, layouts and
 * results are those of paged_attention_decode.
 *
 * The calling thread's current device must be the pool's device (KV_EINVAL
 * otherwise).  The first call on a device looks up that device's address of
 * the array (once, with the device current); make that first call before any
 * stream capture.  The call allocates nothing.  All calls share the one
 * array: calls whose work overlaps on the GPU (other streams, other host
 * threads) race on it and must be serialised by the caller.  Nothing
 * persists in it between calls (each call's counters carry its own random
 * tag, so an earlier call's contents count as empty).
 * Errors: those of paged_attention_decode, and KV_ENOWORKSPACE when the call
 *   would need more than the 32 MiB array holds (paged_attention_workspace_size
 *   tells the need; the piece counters take 16 bytes per sequence x KV head,
 *   so e.g. 4,096 sequences x 1,024 KV heads need 64 MiB of them).
 */
kv_status paged_attention_decode_noalloc(kv_pool_t pool, const void* q, void* out,
                                         const int32_t* block_tables, int max_blocks_per_seq,
                                         const int32_t* seq_lens, int batch, int num_q_heads,
                                         float scale, int num_kv_heads, void* stream);

/*
 * kv_pool_set_wait_limit -- how long one pipeline wait of the attention
 * kernels (paged_attention_decode, _cascade, _noalloc, paged_attention_prefill)
 * may last before the kernel gives up: it sets KV_DEVERR_TIMEOUT, stops
 * loading and attending, lets the copies and tensor-core products already in
 * flight finish (those waits always take the default limit) and returns; the
 * outputs of that call are then unspecified.  The default
 * and largest value is 2 s (2e9 ns); larger values are clamped to it.  A
 * limit of 0 makes every wait that does not find its tile already there give
 * up, which exercises the failure path with valid inputs.  Host-side only,
 * takes effect for the calls enqueued after it.  (The source pages have no
 * counterpart: the kernels' waits are bounded so that a fault cannot hang
 * the GPU, and this is the knob that tests that bound.)
 * Errors: KV_EINVAL (null pool).
 */
kv_status kv_pool_set_wait_limit(kv_pool_t pool, unsigned long long limit_ns);

/*
 * kv_pool_get_error -- read the pool's device error word (KV_DEVERR_* bits,
 * OR-ed over every call since the last clear).  Synchronises the device.
 * Returns KV_ERANGE when any bit is set, KV_OK when none is.
 */
kv_status kv_pool_get_error(kv_pool_t pool, int* device_error_bits);

/* kv_pool_clear_error -- zero the device error word (synchronous). */
kv_status kv_pool_clear_error(kv_pool_t pool);

/* kv_strerror -- static text for a status code. */
const char* kv_strerror(kv_status status);

/* kv_last_cuda_error -- the text of the last CUDA error this library met on
 * the calling thread ("" if none). */
const char* kv_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
