/*
 * mqa_kv.h -- C ABI of libmqa_kv: int8 paged multi-query attention for
 * serving (NVIDIA GB300, sm_103a).
 *
 * The method (Character.AI's serving stack as described in "Character.AI
 * inference optimisation" article, secret 1, and the "Character.AI best
 * practices" blog, sections on multi-query attention, hybrid attention span,
 * cross-layer KV sharing and int8 quantisation):
 *   - multi-query attention: all query heads share ONE K/V head;
 *   - the KV cache is int8 with one fp32 scale per token for K and one for V;
 *   - local layers attend over a sliding window (1024 in the article; any
 *     window here), one layer in six is global;
 *   - adjacent layers read one shared cache through a layer -> cache map;
 *   - the cache is paged (block table per sequence) and prefix blocks may be
 *     shared read-only between sequences (LLM-inference workshop transcript,
 *     01:01:35-01:05:04: PagedAttention and prefix caching).
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers owned by the caller unless marked "host".
 *     The library allocates nothing, keeps no pointer after returning, and
 *     holds no per-call global state; calls are thread-safe.
 *   - All device work is enqueued on `stream` (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  The return value reports only
 *     synchronous argument validation and launch errors; faults inside a
 *     kernel surface at the caller's next synchronisation.
 *   - `dev_status` (nullable, device int32) collects MQA_DEV_* bits with an
 *     atomic OR when a kernel meets a bad device-side input (a block id outside
 *     the pool, a sequence length outside [1, max_seq_len], a bad cu_* entry) or
 *     a bounded wait that ran out.  The kernel never reads or writes outside the
 *     buffers described here: the offending tokens are skipped instead.
 *   - Supported shapes: head_dim in {64, 128}; num_q_heads in {8, 16, 32, 64};
 *     page_size in {16, 64}.  Other values return MQA_ERR_UNSUPPORTED.
 *   - bf16 tensors are IEEE bfloat16 bit patterns.
 */
#ifndef MQA_KV_H
#define MQA_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Synchronous return codes. */
#define MQA_OK 0
#define MQA_ERR_INVALID_ARG (-1)  /* null pointer, bad size, misaligned buffer, out-of-range index */
#define MQA_ERR_UNSUPPORTED (-2)  /* a shape outside the supported set */
#define MQA_ERR_WORKSPACE (-3)    /* workspace missing or smaller than required */
#define MQA_ERR_CUDA (-4)         /* a CUDA runtime call or launch failed */

/* Device-side status bits (OR-ed into *dev_status). */
#define MQA_DEV_BAD_BLOCK 1    /* block_table entry outside [0, num_blocks) */
#define MQA_DEV_BAD_SEQLEN 2   /* seq_lens entry outside [1, max_seq_len] or beyond the table */
#define MQA_DEV_BAD_CU 4       /* cu_new / cu_q entry inconsistent with seq_lens */
#define MQA_DEV_TIMEOUT 8      /* a bounded wait for a TMA copy ran out (2 s) */

/* Upper bound on the split-KV factor of one decode call. */
#define MQA_MAX_SPLITS 1024

/* One physical KV cache: a single shared K/V head.
 *   k_codes, v_codes: int8  [num_blocks][page_size][head_dim], 16-byte aligned
 *   k_scale, v_scale: fp32  [num_blocks][page_size],           16-byte aligned
 * Slot (blk, row) holds one token: x ~= code * scale. */
typedef struct mqa_kv_cache {
    int8_t *k_codes;
    int8_t *v_codes;
    float *k_scale;
    float *v_scale;
    int32_t num_blocks;
    int32_t page_size;
    int32_t head_dim;
} mqa_kv_cache;

/* A ragged batch over paged caches (shared by all caches that use the same
 * block table).
 *   block_table: int32 [batch][max_blocks]; entry i of sequence b is the
 *                physical block of its tokens [i*page, (i+1)*page).
 *   seq_lens:    int32 [batch]; tokens in the cache INCLUDING the ones the
 *                current step appends (>= 1).
 *   seq_lens_host: optional host copy of seq_lens (NULL allowed).  When given it
 *                is validated on the host and used to plan split-KV work.
 *   max_seq_len: host; an upper bound of every seq_lens entry, at most
 *                max_blocks * page_size unless ring_blocks > 0.
 *   ring_blocks: host; 0 = the table maps every page of a sequence.  R > 0 = a
 *                window-bounded cache for local layers: each sequence keeps only
 *                its R most recent pages, page i living in table entry i % R
 *                (a newer page overwrites the entry of the page R before it),
 *                R <= max_blocks.  Local layers of the "Character.AI inference
 *                article" (secret 1) attend over a 1024-token window, so their
 *                caches need ceil(1024 / page) + 1 pages per sequence, not the
 *                whole history.  Calls that read such a cache must stay inside
 *                the resident pages: mqa_decode_attn needs window > 0 and
 *                R >= (window - 1) / page + 2; mqa_prefill_attn needs window > 0
 *                and R >= (window + max_q_len - 2) / page + 2 (its chunk's keys
 *                and the windows of all its queries); otherwise
 *                MQA_ERR_INVALID_ARG.  kv_quant_append flags MQA_DEV_BAD_CU and
 *                skips a sequence appending more than R * page tokens in one
 *                call (they would overwrite one another). */
typedef struct mqa_batch {
    const int32_t *block_table;
    const int32_t *seq_lens;
    const int32_t *seq_lens_host;
    int32_t batch;
    int32_t max_blocks;
    int32_t max_seq_len;
    int32_t ring_blocks;
} mqa_batch;

/* Quantise and append new K/V tokens (one int8 code per element plus one fp32
 * scale per token and tensor: scale = max|x|/127, code = clamp(round half to
 * even(x/scale), -127, 127), both in IEEE fp32; an all-zero vector stores scale
 * 0 and codes 0).  Source: the int8 KV cache of the "Character.AI best
 * practices" blog, section "quantisation for training and serving"; the
 * per-token symmetric scheme is this library's reading of it.
 *
 *   cu_new:  int32 [batch+1] prefix sums; sequence b appends
 *            n_b = cu_new[b+1]-cu_new[b] tokens, which occupy its LAST n_b
 *            positions seq_lens[b]-n_b .. seq_lens[b]-1 (seq_lens already
 *            counts them).
 *   num_new_tokens: host; cu_new[batch].  0 is a no-op.
 *   k_new, v_new: bf16 [num_new_tokens][head_dim], 16-byte aligned.
 * Writes codes and scales in place.  Blocks holding shared prefixes must not
 * be targets.  Returns MQA_OK or a negative MQA_ERR_*. */
int kv_quant_append(const mqa_kv_cache *cache, const mqa_batch *batch, const int32_t *cu_new,
                    int32_t num_new_tokens, const void *k_new, const void *v_new, int32_t *dev_status,
                    void *stream);

/* Decode attention for one layer: the query of sequence b (one token, at
 * position seq_lens[b]-1) attends, for each of num_q_heads heads, to the keys
 * of cache caches[layer_to_kv[layer]] at positions
 *     max(0, L-window) .. L-1   (local layer, window > 0)
 *     0 .. L-1                  (global layer, window == 0).
 * out = softmax(sm_scale * q K^T) V over the dequantised cache.  Sources: MQA
 * and the local/global layer pattern of the Character.AI article, secret 1;
 * the tiled online softmax of the workshop transcript, 00:47:59-00:49:13.
 *
 *   caches[num_caches], layer_to_kv[num_layers]: HOST arrays.
 *   q:   bf16 [batch][num_q_heads][head_dim], 16-byte aligned.  sm_scale > 0.
 *   out: bf16 [batch][num_q_heads][head_dim], 16-byte aligned.
 *   num_splits: 0 = choose automatically (see mqa_decode_auto_splits), 1 = one
 *        CTA per (sequence, head group), S > 1 = the (sequence, head group, key
 *        block) list cut into equal shares over up to batch * groups * S / 2
 *        CTAs; a pair cut between CTAs is merged from its pieces' partials
 *        (flash-decoding).
 *   workspace: device scratch of at least
 *        mqa_decode_workspace_size(batch, num_q_heads, head_dim, S) bytes
 *        (16-byte aligned) when the effective split count S exceeds 1; may be
 *        NULL otherwise.  Its contents on entry do not matter.
 * Returns MQA_OK, or MQA_ERR_WORKSPACE if the workspace is too small. */
int mqa_decode_attn(const mqa_kv_cache *caches, int32_t num_caches, const int32_t *layer_to_kv,
                    int32_t num_layers, int32_t layer, int32_t window, const mqa_batch *batch,
                    const void *q, void *out, int32_t num_q_heads, float sm_scale, int32_t num_splits,
                    void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/* The split count mqa_decode_attn chooses when num_splits == 0 for this batch,
 * window and shape on the current device (>= 1), or a negative MQA_ERR_*. */
int mqa_decode_auto_splits(const mqa_batch *batch, int32_t window, int32_t num_q_heads, int32_t head_dim,
                           int32_t page_size);

/* Bytes of decode workspace for `num_splits` splits: room for fp32 partial
 * outputs [batch][num_splits][num_q_heads][head_dim], then fp32 log-sum-exps
 * [batch][num_splits][num_q_heads], then 64 KiB of merge descriptors, each
 * region 256-byte aligned.  0 when num_splits <= 1.  With S splits the decode
 * runs balanced shares over at most batch * groups * S / 2 CTAs (a group is 32
 * query heads at head_dim 128, 16 at head_dim 64), each keeping the partials of
 * the two (sequence, head group) pairs it may share with its neighbours there;
 * a second kernel merges them. */
size_t mqa_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t head_dim, int32_t num_splits);

/* Merge split-KV partial results (flash-decoding combine; the same log-sum-exp
 * identity the online softmax of the workshop transcript, 00:49:05-00:49:13,
 * relies on):
 *     M = max_s lse_s,  w_s = exp(lse_s - M),
 *     out = sum_s w_s o_s / sum_s w_s          (written as bf16).
 *   o_partial: fp32 [batch][num_splits][num_q_heads][head_dim]
 *   lse:       fp32 [batch][num_splits][num_q_heads], natural log; -inf marks an
 *              empty split, which contributes nothing.  A (sequence, head) whose
 *              splits are all empty gets out = 0.
 *   out:       bf16 [batch][num_q_heads][head_dim], 16-byte aligned. */
int split_kv_combine(const float *o_partial, const float *lse, int32_t batch, int32_t num_splits,
                     int32_t num_q_heads, int32_t head_dim, void *out, void *stream);

/* Chunked prefill attention for one layer over a cached (possibly
 * prefix-shared) context: sequence b has q_len_b = cu_q[b+1]-cu_q[b] new query
 * tokens at positions L-q_len_b .. L-1 (L = seq_lens[b]; their K/V must already
 * be appended with kv_quant_append).  Query t of sequence b attends causally to
 * keys max(0, i-window+1) .. i with i = L-q_len_b+t (window == 0: 0 .. i), read
 * from the int8 cache caches[layer_to_kv[layer]].  Sources: prefill is the
 * compute-bound phase (workshop transcript, 00:20:58-00:22:12); prefix caching
 * (01:04:36-01:05:04); the state cache that makes prefixes resident (Character.AI
 * article, secret 2).
 *
 *   cu_q:      int32 [batch+1] prefix sums of query tokens per sequence.
 *   total_q:   host; cu_q[batch].   max_q_len: host; max_b q_len_b (a sequence
 *              with more query tokens is skipped and flagged MQA_DEV_BAD_CU).
 *   q, out:    bf16 [total_q][num_q_heads][head_dim], 16-byte aligned.
 *   workspace: device scratch of mqa_prefill_workspace_size(...) bytes
 *              (16-byte aligned).  The call first converts, once per sequence,
 *              every key tile its queries can see to fp16 there; its contents on
 *              entry do not matter.
 * Returns MQA_OK, or MQA_ERR_WORKSPACE if the workspace is missing or too small. */
int mqa_prefill_attn(const mqa_kv_cache *caches, int32_t num_caches, const int32_t *layer_to_kv,
                     int32_t num_layers, int32_t layer, int32_t window, const mqa_batch *batch,
                     const int32_t *cu_q, int32_t total_q, int32_t max_q_len, const void *q, void *out,
                     int32_t num_q_heads, float sm_scale, void *workspace, size_t workspace_bytes,
                     int32_t *dev_status, void *stream);

/* Bytes of prefill workspace for a batch of `batch` sequences of at most
 * max_seq_len keys and max_q_len query tokens, at this window and head_dim:
 * per sequence, T = min(ceil(max_seq_len / 64), (window + max_q_len - 2) / 64
 * + 2 when window > 0) + 1 tiles of 64 keys, each a 256 * head_dim byte fp16
 * image (K and V as the tensor core reads them) and a 528-byte record (K and V
 * scales, the largest V scale, an all-valid flag), the records after the
 * images (256-byte aligned).  0 for an unsupported head_dim. */
size_t mqa_prefill_workspace_size(int32_t batch, int32_t max_seq_len, int32_t window, int32_t max_q_len,
                                  int32_t head_dim);

/* Decode attention without a workspace argument, for callers that cannot
 * allocate device memory (for example code running while a framework captures
 * a CUDA graph and forbids new allocations, serving loops whose memory budget
 * is reserved up front, or plugins with no access to the process's allocator).
 * The pages this library follows describe no counterpart to this call; it
 * exists for those callers.
 *
 * Same arguments and results as mqa_decode_attn, minus workspace.  Split-KV
 * partials go to one library-owned device array of 32 MiB that every GPU which
 * loads the library holds until the process exits.  num_splits == 0 picks the
 * automatic plan, narrowed until its workspace fits 32 MiB; an explicit
 * num_splits whose workspace exceeds 32 MiB returns MQA_ERR_WORKSPACE.  The
 * call allocates nothing (no cudaMalloc, no library allocation).  Every call
 * shares the one array: calls whose GPU work overlaps (other streams, other
 * threads) race and must be serialised by the caller.  The first call on a
 * device looks up the array's device address; make that first call before any
 * stream capture.  The address is kept for the life of the process: do not use
 * this entry point on a device after cudaDeviceReset (or after its primary
 * context was destroyed), because later calls would reuse the old address. */
int mqa_decode_attn_noalloc(const mqa_kv_cache *caches, int32_t num_caches, const int32_t *layer_to_kv,
                            int32_t num_layers, int32_t layer, int32_t window, const mqa_batch *batch,
                            const void *q, void *out, int32_t num_q_heads, float sm_scale, int32_t num_splits,
                            int32_t *dev_status, void *stream);

/* A static, human-readable name for a return code. */
const char *mqa_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* MQA_KV_H */
