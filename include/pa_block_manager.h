/*
 * pa_block_manager.h -- host-side manager of the paged KV block pool (part of libpagedattn.so).
 *
 * It decides which physical block holds which logical block of every sequence, and hands the
 * attention step its slots and block tables.  Pure host C++; no device memory, no CUDA calls.
 *
 *   "Serving LLMs with vLLM: Continuous Batching and PagedAttention Explained":
 *     "Blocks and Block Tables"  fixed-size blocks, a per-sequence table, a block is taken from
 *                                the free list only when the current one fills up;
 *     "Growing During Decode"    each step appends into the last block; a finished sequence
 *                                returns all its blocks at once;
 *     "Shared Prefixes", "The Savings in Numbers"  several tables point at one copy, with a
 *                                reference count;
 *     "Copy-on-Write"            writing into a block whose count is above one first copies it
 *                                to a fresh block for this sequence only.
 *   "Why a Second Kind of Engine: Batching, Paged Attention and Throughput", "Prefix caching":
 *     every full block is hashed by its tokens and the tokens before it; a map from hashes to
 *     blocks lets a new request reuse a cached prefix; cached blocks that no sequence uses are
 *     evicted least-recently-used first when space is needed.
 *
 * Determinism: free blocks are handed out lowest id first among never-used ones, then in the
 * order they were released; evictable cached blocks go in least-recently-released order.
 * Every call either completes or (returning PA_BM_NO_SPACE) changes nothing.
 * Not thread-safe: one manager per scheduler thread.
 */
#ifndef PAGED_KV_PA_BLOCK_MANAGER_H_
#define PAGED_KV_PA_BLOCK_MANAGER_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_block_manager pa_block_manager;

#define PA_BM_NO_SPACE (-1)   /* not enough free (or evictable) blocks; nothing changed */
#define PA_BM_BAD_ARG (-2)    /* unknown sequence, existing sequence where a new one is needed,
                                 negative count, too small output buffer */

/* A pool of num_blocks blocks of block_size token slots.  NULL on bad arguments. */
pa_block_manager* pa_bm_create(int32_t num_blocks, int32_t block_size);
void pa_bm_destroy(pa_block_manager* bm);

/* Blocks that can be handed out right now: never-used or released blocks plus cached blocks
 * that no sequence references (those are evicted on demand). */
int32_t pa_bm_num_free(const pa_block_manager* bm);

/* Append n tokens to sequence seq (created when unknown).  slots_out[i] receives the slot
 * (block * block_size + offset) of the i-th new token.  If the sequence's partly filled last
 * block is shared, it is first replaced by a fresh copy (copy-on-write): the pair (old, new) is
 * written to copy_pairs_out (at most one pair per call, so capacity 1 suffices) and the caller
 * must copy the block on the device (pa_copy_blocks) before writing the new tokens.
 * Returns the number of copy pairs written (0 or 1), PA_BM_NO_SPACE or PA_BM_BAD_ARG.
 * Blocks filled through this call carry no hash (they are never offered as a cached prefix). */
int32_t pa_bm_append(pa_block_manager* bm, int64_t seq, int32_t n, int64_t* slots_out,
                     int32_t* copy_pairs_out, int32_t copy_cap);

/* Like pa_bm_append, but with the token ids, which makes the sequence's full blocks cacheable.
 * For a sequence that has no tokens yet, the longest run of leading full blocks whose chained
 * hash (and token ids) match cached blocks is reused instead of allocated; *cached_tokens_out
 * receives the number of leading tokens whose K/V are already in the pool (the caller need not
 * compute or append them).  Every block this sequence fills is registered in the cache. */
int32_t pa_bm_append_tokens(pa_block_manager* bm, int64_t seq, const int32_t* tokens, int32_t n,
                            int64_t* slots_out, int32_t* copy_pairs_out, int32_t copy_cap,
                            int32_t* cached_tokens_out);

/* Leading tokens of `tokens` (a whole number of blocks) whose full blocks are in the prefix
 * cache right now, i.e. what pa_bm_append_tokens would reuse for a new sequence if nothing is
 * evicted first.  Changes nothing. */
int32_t pa_bm_cached_prefix(const pa_block_manager* bm, const int32_t* tokens, int32_t n);

/* New sequence child sharing every block of parent (reference counts + 1), e.g. for several
 * completions sampled from one prompt.  Returns 0 or PA_BM_BAD_ARG. */
int32_t pa_bm_fork(pa_block_manager* bm, int64_t parent, int64_t child);

/* Release all blocks of seq (reference counts - 1; a block whose count reaches 0 returns to the
 * free list, or to the evictable cache if it carries a hash).  Returns 0 or PA_BM_BAD_ARG. */
int32_t pa_bm_free(pa_block_manager* bm, int64_t seq);

/* Block table of seq into table_out[0..cap); returns the number of blocks (may exceed cap, in
 * which case only cap entries are written) or PA_BM_BAD_ARG. */
int32_t pa_bm_block_table(const pa_block_manager* bm, int64_t seq, int32_t* table_out,
                          int32_t cap);

/* Tokens held by seq, or PA_BM_BAD_ARG. */
int64_t pa_bm_num_tokens(const pa_block_manager* bm, int64_t seq);

/* Reference count of a block (0 for a free or only-cached block), or PA_BM_BAD_ARG. */
int32_t pa_bm_refcount(const pa_block_manager* bm, int32_t block);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_PA_BLOCK_MANAGER_H_ */
