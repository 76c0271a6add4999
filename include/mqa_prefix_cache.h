/*
 * mqa_prefix_cache.h -- C ABI of the host-memory prefix cache of libmqa_kv.
 *
 * What it follows: Character.AI keeps the attention KV of every conversation
 * prefix in HOST memory between turns, in an LRU-managed tree of cached KV
 * tensors indexed by a rolling hash of the prefix tokens, so that a new request
 * finds the longest cached prefix (also when only part of it matches) and
 * skips recomputing it ("Character.AI inference optimisation" article, secret
 * 2; "Character.AI best practices" blog, "stateful caching" and "LRU cache
 * structure"; LLM-inference workshop transcript, 01:14:28-01:16:24: a radix
 * tree of prefixes instead of whole-prompt hashes, so that a prompt that
 * differs late still reuses its common prefix).
 *
 * Reading of the pages, in this library:
 *   - The unit of caching is one full page (page_size tokens) of every paged
 *     KV cache of the model (the caches of a layer stack share one block
 *     table): a prefix is cached page by page, a partial last page is not.
 *   - The tree has one node per cached page; a node's key is the rolling hash
 *     of all tokens from the start of the sequence to the end of its page
 *     (h <- h * 0x100000001b3 + token + 1, mod 2^64, over int32 tokens), and a
 *     hit is confirmed by comparing the page's tokens and its parent node, so a
 *     hash collision can cost a hit but never return wrong data.
 *   - The longest match of a token sequence is the largest k such that its
 *     first k pages are cached along one path from the root.
 *   - LRU: every match and insert stamps the pages of its path with a new
 *     time; when the host pool is full, the cached page without cached
 *     successors (a leaf) with the oldest stamp is evicted, one page at a time,
 *     never a page of the path being inserted.
 *   - The host pool is pinned host memory that the GPU reads and writes
 *     directly (on GB300 over the NVLink-C2C link): upload and offload are
 *     kernels that gather or scatter whole pages between the pool and device
 *     blocks, no per-page copy calls.
 *
 * Host pool layout: slot s holds, for each cache c in order, K codes
 * [page_size][head_dim] int8, V codes [page_size][head_dim] int8, K scales
 * [page_size] fp32, V scales [page_size] fp32: num_caches * page_size *
 * (2 * head_dim + 8) bytes per slot.
 *
 * Threading: one cache object is not thread-safe; calls on it must be
 * serialised by the caller.  Upload and offload enqueue work on `stream`;
 * the caller keeps match / insert / upload / offload of one cache in stream
 * order (a slot evicted by an insert may be overwritten by the next offload).
 */
#ifndef MQA_PREFIX_CACHE_H
#define MQA_PREFIX_CACHE_H

#include <stdint.h>

#include "mqa_kv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mqa_prefix_cache mqa_prefix_cache;  /* opaque */

/* Create a cache of up to host_pages pages of num_caches caches of shape
 * (page_size, head_dim).  pinned != 0 allocates the pool as pinned, device-
 * mapped host memory (needed by upload and offload); pinned == 0 allocates
 * ordinary host memory (tree bookkeeping only: upload and offload return
 * MQA_ERR_UNSUPPORTED).  *out receives the handle.  Returns MQA_OK,
 * MQA_ERR_INVALID_ARG (sizes < 1, num_caches > MQA_PC_MAX_CACHES, out NULL),
 * MQA_ERR_UNSUPPORTED (head_dim / page_size outside the supported set) or
 * MQA_ERR_CUDA (the pinned allocation failed). */
#define MQA_PC_MAX_CACHES 32
int mqa_pc_create(int32_t page_size, int32_t head_dim, int32_t num_caches, int64_t host_pages, int32_t pinned,
                  mqa_prefix_cache **out);

/* Free the pool and the tree (NULL is a no-op).  The caller first synchronises
 * any stream with upload / offload work of this cache in flight. */
void mqa_pc_destroy(mqa_prefix_cache *pc);

/* Longest cached prefix of tokens[0, n_tokens) (host): the number k of
 * whole pages matched, with their slots written to slots[0, min(k, max_pages))
 * (host).  The k pages are stamped most recently used.  Returns k >= 0 or
 * MQA_ERR_INVALID_ARG. */
int64_t mqa_pc_match(mqa_prefix_cache *pc, const int32_t *tokens, int64_t n_tokens, int64_t *slots,
                     int64_t max_pages);

/* Insert the whole pages of tokens[0, n_tokens) (host): pages already cached
 * are stamped, missing ones get a slot (evicting LRU leaves when the pool is
 * full).  For every NEW page, page_index[i] (its index in the sequence) and
 * slots[i] are written (host, up to max_new entries); the caller then copies
 * those pages into the pool with mqa_pc_offload before the next match can
 * upload them.  Insertion stops early when the pool holds nothing evictable
 * (every page lies on this path).  Returns the number of new pages (>= 0) or
 * MQA_ERR_INVALID_ARG. */
int64_t mqa_pc_insert(mqa_prefix_cache *pc, const int32_t *tokens, int64_t n_tokens, int64_t *page_index,
                      int64_t *slots, int64_t max_new);

/* Device -> pool: page i of every cache, from device block src_blocks[i] into
 * slot slots[i] (both host arrays of n entries), enqueued on stream.  The
 * caches must match the pool's shape and count (page_size, head_dim,
 * num_caches).  Returns MQA_OK, MQA_ERR_INVALID_ARG (a block or slot out of
 * range, a shape mismatch), MQA_ERR_UNSUPPORTED (pool not pinned) or
 * MQA_ERR_CUDA. */
int mqa_pc_offload(mqa_prefix_cache *pc, const mqa_kv_cache *caches, int32_t num_caches, const int32_t *src_blocks,
                   const int64_t *slots, int64_t n, void *stream);

/* Pool -> device: slot slots[i] into device block dst_blocks[i] of every
 * cache (host arrays of n entries), enqueued on stream; errors as offload.
 * This is the step before prefill: the uploaded pages are the cached prefix of
 * a sequence, and prefill then computes only the tokens after it. */
int mqa_pc_upload(mqa_prefix_cache *pc, const mqa_kv_cache *caches, int32_t num_caches, const int64_t *slots,
                  const int32_t *dst_blocks, int64_t n, void *stream);

/* Counters (host out[8]): cached pages, free slots, slot capacity, match
 * calls, pages matched, pages inserted, pages evicted, bytes per slot. */
int mqa_pc_stats(const mqa_prefix_cache *pc, int64_t *out);

#ifdef __cplusplus
}
#endif

#endif /* MQA_PREFIX_CACHE_H */
